"""The entry point that allocates nothing (sk_gemm_bf16_static), for callers that may not
allocate device memory when they run the GEMM (under an allocator they do not own, or on a
path where an allocation could synchronise the device): its output must match the regular
entry point's, and the oracle, on two calls in a row (the second call reuses the fixed
scratch array the first one left behind), and a call must allocate no device memory.  This
file is collected last so that a failure here stops a -x run only after every other test has
run."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
import sm_constrained_persistent_gb300 as sk
from sm_constrained_persistent_gb300 import inputs

pytestmark = pytest.mark.gpu

M, N, K = 1000, 1032, 2056   # ragged against the 128 x 128 tiles in every dimension
TORCH_OUT = {"bf16": torch.bfloat16, "f32": torch.float32}
SK_OUT = {"bf16": sk.SK_BF16, "f32": sk.SK_F32}
_problems = {}


def _problem(out):
    if out not in _problems:
        p = inputs.bf16_problem(M, N, K, seed=2024, operand_scale="sqrt_k",
                                bias="bf16_uniform" if out == "bf16" else "f32_normal")
        ref = gu.reference(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), out)
        _problems[out] = (p, ref)
    return _problems[out]


@pytest.mark.parametrize("out", ["bf16", "f32"])
@pytest.mark.parametrize("mode", ["streamk", "hybrid", "persistent", "dp", "auto"])
def test_static_scratch_entry_matches_allocating_entry_twice(cuda_device, mode, out):
    p, ref = _problem(out)
    a, b, bias = gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"]), gu.dev_bias(p["bias"])
    stream = torch.cuda.current_stream().cuda_stream
    want = torch.empty((M, N), dtype=TORCH_OUT[out], device="cuda")
    st = sk.sk_gemm_bf16(a.data_ptr(), b.data_ptr(), bias.data_ptr(), want.data_ptr(), SK_OUT[out],
                         M, N, K, 0, sk.MODES[mode], stream)
    assert st == sk.SK_OK
    assert sk.sk_stream_status(stream) == sk.SK_OK
    regular = gu.host_values(want)
    gu.assert_close(regular, ref, out, f"regular {mode}")
    for call in range(2):
        got = torch.full((M, N), float("nan"), dtype=TORCH_OUT[out], device="cuda")
        st = sk.sk_gemm_bf16_static(a.data_ptr(), b.data_ptr(), bias.data_ptr(), got.data_ptr(),
                                    SK_OUT[out], M, N, K, 0, sk.MODES[mode], stream)
        assert st == sk.SK_OK, sk.STATUS.get(st, st)
        assert sk.sk_gemm_bf16_static_status(stream) == sk.SK_OK
        values = gu.host_values(got)
        gu.assert_close(values, regular, out, f"{mode} call {call} against sk_gemm_bf16")
        gu.assert_close(values, ref, out, f"{mode} call {call} against the oracle")


@pytest.mark.parametrize("mode", ["streamk", "hybrid", "persistent", "dp"])
def test_static_scratch_entry_with_tall_stages_is_bit_exact(cuda_device, mode):
    # at most 64 rows of A: the static entry runs the tall-stage (128 K) kernel too
    m, n, k = 48, 2056, 4104
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = sk.sk_plan(0, m, n, k, 0, mode, sms, {"tile_m": 128, "tile_n": 128})
    assert (plan.tile_k, plan.iters) == (128, 33)
    p = inputs.bf16_problem(m, n, k, seed=77, integer=True, bias="f32_int")
    want = oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), oracle.F32)
    a, b, bias = gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"]), gu.dev_bias(p["bias"])
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        got = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
        st = sk.sk_gemm_bf16_static(a.data_ptr(), b.data_ptr(), bias.data_ptr(), got.data_ptr(),
                                    sk.SK_F32, m, n, k, 0, sk.MODES[mode], stream)
        assert st == sk.SK_OK, sk.STATUS.get(st, st)
        assert sk.sk_gemm_bf16_static_status(stream) == sk.SK_OK
        assert np.array_equal(gu.host_bits(got), want.view(np.uint32)), (mode, call)


def test_static_scratch_entry_allocates_no_device_memory(cuda_device):
    p, ref = _problem("bf16")
    a, b, bias = gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"]), gu.dev_bias(p["bias"])
    got = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fresh = torch.cuda.Stream()   # a stream the regular entry points have never used
    args = (a.data_ptr(), b.data_ptr(), bias.data_ptr(), got.data_ptr(), sk.SK_BF16, M, N, K, 0)
    assert sk.sk_gemm_bf16_static(*args, sk.MODES["streamk"], None) == sk.SK_OK   # set-up done
    torch.cuda.synchronize()
    free0, reserved0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved()
    for mode in ("streamk", "hybrid", "persistent"):
        assert sk.sk_gemm_bf16_static(*args, sk.MODES[mode], fresh.cuda_stream) == sk.SK_OK
        assert sk.sk_gemm_bf16_static_status(fresh.cuda_stream) == sk.SK_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_reserved() == reserved0
    gu.assert_close(gu.host_values(got), ref, "bf16", "static call on a fresh stream")


def test_static_scratch_entry_checks_arguments_like_the_regular_one(cuda_device):
    assert sk.sk_gemm_bf16_static(None, 16, None, 16, 1, 64, 64, 64, 0, 2, None) == sk.SK_ERR_INVALID_ARG
    assert sk.sk_gemm_bf16_static(16, 16, None, 16, 1, 64, 60, 64, 0, 2, None) == sk.SK_ERR_INVALID_ARG
    assert sk.sk_gemm_bf16_static(16, 16, None, 16, 1, 64, 64, 64, 0, 5, None) == sk.SK_ERR_INVALID_ARG
