"""SM-constrained GEMM running beside other work on the same GPU (the intra-device
parallelism that motivates capping the grid at num_sms: flashinfer PR #982
"SM-constraint-GEMM by triton persistent kernel", overview).  A memory-bound copy runs on a
second stream while the GEMM runs on num_sms SMs; the GEMM's result must equal its result
when run alone (same schedule, same summation order), and a Stream-K GEMM must finish without
timing out while the other kernel holds SMs."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
import sm_constrained_persistent_gb300 as sk
from sm_constrained_persistent_gb300 import inputs

pytestmark = pytest.mark.gpu


def _corun(fn_gemm, copy_iters=40, size=256 << 20):
    """Launch `copy_iters` large copies on one stream and the GEMM on another, concurrently."""
    src = torch.empty(size // 4, dtype=torch.float32, device="cuda").fill_(1.0)
    dst = torch.empty_like(src)
    s_copy, s_gemm = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s_copy):
        for _ in range(copy_iters):
            dst.copy_(src)
    with torch.cuda.stream(s_gemm):
        out = fn_gemm(s_gemm)
    torch.cuda.synchronize()
    return out, s_gemm


@pytest.mark.parametrize("mode", ["persistent", "streamk", "hybrid"])
@pytest.mark.parametrize("tile", ["auto", "128x128"])
@pytest.mark.parametrize("num_sms", [64, 76])
def test_gemm_beside_a_copy_matches_the_gemm_alone(cuda_device, mode, tile, num_sms):
    p = inputs.bf16_problem(2048, 2048, 4096, seed=3, operand_scale="sqrt_k", bias="bf16_uniform")
    a, b, bias = gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"]), gu.dev_bias(p["bias"])
    opts = None if tile == "auto" else {"tile_m": 128, "tile_n": 128}
    alone = sk.gemm_bf16(a, b, bias, mode=mode, num_sms=num_sms, options=opts)
    sk.stream_status()

    def gemm(stream):
        return sk.gemm_bf16(a, b, bias, mode=mode, num_sms=num_sms, options=opts, stream=stream)

    together, s = _corun(gemm)
    assert sk.sk_stream_status(s.cuda_stream) == sk.SK_OK
    assert np.array_equal(gu.host_bits(together), gu.host_bits(alone))
    ms, ns = gu.sample_positions(2048, 2048, n_random=512, n_rows=2, n_cols=2)
    ref = gu.reference(oracle.addmm_bf16_at(p["A"], p["B"], p["bias"], ms, ns), "bf16")
    got = together.float()[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()]
    gu.assert_close(got.cpu().numpy().astype(np.float64), ref, "bf16", f"{mode}/{tile}")


def test_mxfp4_streamk_beside_a_copy(cuda_device):
    p = inputs.mxfp4_problem(2048, 2048, 4096, seed=5, exp_range=1)
    args = (gu.dev_u8(p["A"]), gu.dev_u8(p["A_scale"]), gu.dev_u8(p["B"]), gu.dev_u8(p["B_scale"]))
    alone = sk.gemm_mxfp4(*args, None, out_dtype=torch.float32, mode="streamk", num_sms=76)
    sk.stream_status()
    together, s = _corun(lambda st: sk.gemm_mxfp4(*args, None, out_dtype=torch.float32,
                                                  mode="streamk", num_sms=76, stream=st))
    assert sk.sk_stream_status(s.cuda_stream) == sk.SK_OK
    assert np.array_equal(gu.host_bits(together), gu.host_bits(alone))
    ms, ns = gu.sample_positions(2048, 2048, n_random=512, n_rows=2, n_cols=2)
    ref = gu.reference(oracle.addmm_mxfp4_at(p["A"], p["A_scale"], p["B"], p["B_scale"], None, ms, ns),
                       "f32")
    got = together[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()]
    gu.assert_close(got.cpu().numpy().astype(np.float64), ref, "f32", "MXFP4 Stream-K co-run")
