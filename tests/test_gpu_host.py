"""GPU parity of the host-buffer entry points (operands and result in host memory, copies
overlapped with the GEMM in row blocks) against the CPU oracle, through the C ABI."""
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


def host_bf16(bits, pin=True):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pin else t.clone()


def host_bias(b, pin=True):
    if b is None:
        return None
    t = torch.from_numpy(b) if b.dtype == np.float32 else \
        torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pin else t.clone()


def host_u8(x, pin=True):
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.pin_memory() if pin else t.clone()


def bits(c):
    return gu.host_bits(c)


@pytest.mark.parametrize("mode", ["dp", "persistent", "streamk", "hybrid"])
@pytest.mark.parametrize("shape", [(1, 16, 64), (300, 136, 272), (1000, 520, 1024),
                                   (2304, 768, 512), (4100, 264, 128)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_bf16_integer_inputs_are_bit_exact(mode, shape, out):
    M, N, K = shape
    p = inputs.bf16_problem(M, N, K, seed=M + N + K, integer=True,
                            bias="f32_int" if out == "f32" else "bf16_int")
    c = sk.gemm_host("bf16", host_bf16(p["A"]), host_bf16(p["B"]), host_bias(p["bias"]),
                     out_dtype=gu.out_torch_dtype(out), mode=mode, num_sms=24)
    want = oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], p["bias"]),
                               oracle.BF16 if out == "bf16" else oracle.F32)
    assert np.array_equal(bits(c), want if out == "bf16" else want.view(np.uint32))


@pytest.mark.parametrize("fmt", ["bf16", "fp8", "mxfp4"])
def test_random_inputs_match_oracle_and_the_device_call(fmt):
    M, N, K = 2560, 512, 1024
    if fmt == "bf16":
        p = inputs.bf16_problem(M, N, K, seed=71, operand_scale="sqrt_k", bias="bf16_uniform")
        c = sk.gemm_host("bf16", host_bf16(p["A"]), host_bf16(p["B"]), host_bias(p["bias"]))
        ref = oracle.addmm_bf16(p["A"], p["B"], p["bias"])
    elif fmt == "fp8":
        p = inputs.fp8_problem(M, N, K, seed=72, operand_scale="sqrt_k", bias="bf16_uniform")
        c = sk.gemm_host("fp8", host_u8(p["A"]), host_u8(p["B"]), host_bias(p["bias"]))
        ref = oracle.addmm_fp8(p["A"], p["B"], p["bias"])
    else:
        p = inputs.mxfp4_problem(M, N, K, seed=73, exp_range=2, bias="bf16_uniform")
        c = sk.gemm_host("mxfp4", host_u8(p["A"]), host_u8(p["B"]), host_bias(p["bias"]),
                         a_scale=host_u8(p["A_scale"]), b_scale=host_u8(p["B_scale"]))
        ref = oracle.addmm_mxfp4(p["A"], p["A_scale"], p["B"], p["B_scale"], p["bias"])
    gu.assert_close(gu.host_values(c), gu.reference(ref, "bf16"), "bf16", fmt)


def test_pageable_host_memory_and_changing_shapes():
    # unpinned buffers copy synchronously but give the same result; shapes may grow and
    # shrink between calls on one stream
    for M, N, K, pin in [(512, 256, 256, False), (3000, 384, 512, True), (128, 64, 64, False)]:
        p = inputs.bf16_problem(M, N, K, seed=M, integer=True, bias="f32_int")
        c = sk.gemm_host("bf16", host_bf16(p["A"], pin), host_bf16(p["B"], pin),
                         host_bias(p["bias"], pin), out_dtype=torch.float32,
                         out=torch.empty((M, N), dtype=torch.float32))
        want = oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), oracle.F32)
        assert np.array_equal(bits(c), want.view(np.uint32))


def test_two_streams_keep_separate_device_copies():
    pa = inputs.bf16_problem(1024, 256, 512, seed=81, integer=True, bias="f32_int")
    pb = inputs.bf16_problem(1024, 256, 512, seed=82, integer=True, bias="f32_int")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs, keep = [], []
    for p, s in ((pa, s1), (pb, s2)):
        outs.append(torch.empty((1024, 256), dtype=torch.float32).pin_memory())
        keep.append((host_bf16(p["A"]), host_bf16(p["B"]), host_bias(p["bias"])))
        a, b, bias = keep[-1]
        st = sk.sk_gemm_bf16_host(a.data_ptr(), b.data_ptr(), bias.data_ptr(), outs[-1].data_ptr(),
                                  sk.SK_F32, 1024, 256, 512, 0, sk.MODES["streamk"], None,
                                  s.cuda_stream)
        assert st == sk.SK_OK
    torch.cuda.synchronize()
    for p, c in zip((pa, pb), outs):
        want = oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), oracle.F32)
        assert np.array_equal(bits(c), want.view(np.uint32))


def test_addmm_8192_cube_from_host_sampled():
    p = inputs.workload("addmm_bf16_8192")
    c = sk.gemm_host("bf16", host_bf16(p["A"]), host_bf16(p["B"]), host_bias(p["bias"]))
    ms, ns = gu.sample_positions(p["M"], p["N"])
    ref = gu.reference(oracle.addmm_bf16_at(p["A"], p["B"], p["bias"], ms, ns), "bf16")
    got = c.float().numpy()[ms, ns].astype(np.float64)
    gu.assert_close(got, ref, "bf16", "host 8192")
