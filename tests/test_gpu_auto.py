"""GPU parity of the automatic schedule and tile choice (SK_MODE_AUTO) against the CPU oracle:
whatever plan the cost model picks, the result is the addmm."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
import sm_constrained_persistent_gb300 as sk
from sm_constrained_persistent_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _device(cuda_device):
    yield


@pytest.mark.parametrize("shape", [(64, 1024, 2048), (300, 520, 4096), (1024, 1024, 8192),
                                   (2304, 768, 1024), (1536, 1536, 512)])
@pytest.mark.parametrize("num_sms", [0, 7, 64])
def test_bf16_auto_integer_inputs_are_bit_exact(shape, num_sms):
    M, N, K = shape
    p = inputs.bf16_problem(M, N, K, seed=M + N + K + num_sms, integer=True, bias="f32_int")
    c = gu.run_bf16(p, out="f32", mode="auto", num_sms=num_sms)
    want = oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), oracle.F32)
    assert np.array_equal(gu.host_bits(c), want.view(np.uint32))


def test_fp8_and_mxfp4_auto_match_oracle():
    p = inputs.fp8_problem(1024, 768, 2048, seed=3, operand_scale="sqrt_k", bias="bf16_uniform")
    c = sk.gemm_fp8(gu.dev_u8(p["A"]), gu.dev_u8(p["B"]), gu.dev_bias(p["bias"]), mode="auto")
    sk.stream_status()
    gu.assert_close(gu.host_values(c), gu.reference(oracle.addmm_fp8(p["A"], p["B"], p["bias"]),
                                                    "bf16"), "bf16", "fp8 auto")
    q = inputs.mxfp4_problem(768, 1024, 2048, seed=4, exp_range=2, bias="bf16_uniform")
    c = gu.run_mxfp4(q, out="bf16", mode="auto")
    ref = oracle.addmm_mxfp4(q["A"], q["A_scale"], q["B"], q["B_scale"], q["bias"])
    gu.assert_close(gu.host_values(c), gu.reference(ref, "bf16"), "bf16", "mxfp4 auto")


def test_backward_and_host_calls_accept_auto():
    p = inputs.bf16_problem(512, 256, 384, seed=5, integer=True, bias="bf16_int")
    a, b = gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"])
    dc = gu.dev_bf16(inputs.bf16_problem(512, 8, 256, seed=6, integer=True)["A"])   # 512 x 256
    da, db, dbias = sk.addmm_backward(dc, a, b, grad_dtype=torch.float32, mode="auto")
    ref = sk.addmm_backward(dc, a, b, grad_dtype=torch.float32, mode="dp")
    for x, y in zip((da, db, dbias), ref):
        assert torch.equal(x, y)      # integer inputs: exact under every schedule
    host = sk.gemm_host("bf16", torch.from_numpy(p["A"].view(np.int16)).view(torch.bfloat16),
                        torch.from_numpy(p["B"].view(np.int16)).view(torch.bfloat16),
                        mode="auto", out_dtype=torch.float32)
    want = oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], None), oracle.F32)
    assert np.array_equal(host.numpy().view(np.uint32), want.view(np.uint32))


def test_autotune_picks_a_measured_plan_that_auto_mode_then_uses():
    p = inputs.bf16_problem(1536, 1024, 2048, seed=21, operand_scale="sqrt_k", bias="f32_normal")
    a, b, bias = gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"]), gu.dev_bias(p["bias"])
    plan, ms = sk.autotune("bf16", a, b, bias, out_dtype=torch.float32, reps=3)
    assert plan.mode in (1, 2, 3) and ms > 0
    ref = gu.reference(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), "f32")
    auto = sk.gemm_bf16(a, b, bias, out_dtype=torch.float32, mode="auto")
    sk.stream_status()
    gu.assert_close(gu.host_values(auto), ref, "f32")
    # the same plan run explicitly gives the same bits: auto used the measured choice
    opts = {"tile_m": plan.tile_m, "tile_n": plan.tile_n,
            "hybrid_sk_waves": 1 if (plan.mode == 3 and plan.sk_tiles > plan.tiles % plan.grid) else 0}
    explicit = sk.gemm_bf16(a, b, bias, out_dtype=torch.float32, mode=int(plan.mode), options=opts)
    sk.stream_status()
    assert torch.equal(auto, explicit)


def test_autotune_fp8_and_mxfp4():
    p = inputs.fp8_problem(1024, 768, 1024, seed=22, integer=True)
    a, b = gu.dev_u8(p["A"]), gu.dev_u8(p["B"])
    plan, ms = sk.autotune("fp8", a, b, out_dtype=torch.float32, reps=2)
    c = sk.gemm_fp8(a, b, out_dtype=torch.float32, mode="auto")
    sk.stream_status()
    want = oracle.round_output(oracle.addmm_fp8(p["A"], p["B"], None), oracle.F32)
    assert np.array_equal(gu.host_bits(c), want.view(np.uint32))
    q = inputs.mxfp4_problem(512, 768, 1024, seed=23, exp_range=1)
    args = [gu.dev_u8(q[k]) for k in ("A", "A_scale", "B", "B_scale")]
    plan, ms = sk.autotune("mxfp4", args[0], args[2], a_scale=args[1], b_scale=args[3],
                           out_dtype=torch.float32, reps=2)
    assert plan.tile_n in (128, 256) and ms > 0
    c = sk.gemm_mxfp4(*args, None, out_dtype=torch.float32, mode="auto")
    sk.stream_status()
    want = oracle.round_output(oracle.addmm_mxfp4(q["A"], q["A_scale"], q["B"], q["B_scale"], None),
                               oracle.F32)
    assert np.array_equal(gu.host_bits(c), want.view(np.uint32))
