"""GPU parity of the stored-transposed GEMM (sk_gemm_bf16_t) and of the addmm backward
(sk_addmm_backward_bf16: dA = dC B^T, dB = A^T dC, dbias = column sums of dC) against the CPU
oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
import sm_constrained_persistent_gb300 as sk
from sm_constrained_persistent_gb300 import inputs

pytestmark = pytest.mark.gpu
MODES = ["dp", "persistent", "streamk", "hybrid"]
TILES = {"128x128": {"tile_m": 128, "tile_n": 128}, "128x256": {"tile_m": 128, "tile_n": 256},
         "pair256": {"tile_m": 256}}


@pytest.fixture(autouse=True)
def _device(cuda_device):
    yield


def _ints(rng, shape):
    return inputs.to_bf16_bits(rng.integers(-8, 9, shape).astype(np.float32))


@pytest.mark.parametrize("ta", [0, 1])
@pytest.mark.parametrize("tb", [0, 1])
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("tile", list(TILES))
@pytest.mark.parametrize("shape", [(264, 520, 392), (1000, 776, 1000), (128, 128, 64)])
def test_transposed_gemm_integer_bit_exact(ta, tb, mode, tile, shape):
    M, N, K = shape
    rng = np.random.default_rng(M + N + K + 10 * ta + 20 * tb)
    A = _ints(rng, (K, M) if ta else (M, K))
    B = _ints(rng, (N, K) if tb else (K, N))
    c = sk.gemm_bf16_t(gu.dev_bf16(A), gu.dev_bf16(B), trans_a=ta, trans_b=tb,
                       out_dtype=torch.float32, mode=mode, num_sms=10, options=TILES[tile])
    sk.stream_status()
    want = oracle.round_output(oracle.gemm_bf16_t(A, ta, B, tb), oracle.F32)
    assert np.array_equal(gu.host_bits(c), want.view(np.uint32))


@pytest.mark.parametrize("ta", [0, 1])
@pytest.mark.parametrize("tb", [0, 1])
def test_transposed_gemm_random_with_bias(ta, tb):
    M, N, K = 768, 1024, 2048
    rng = np.random.default_rng(7 + ta + 2 * tb)
    A = inputs.to_bf16_bits((rng.standard_normal((K, M) if ta else (M, K)) / K ** 0.5).astype(np.float32))
    B = inputs.to_bf16_bits(rng.standard_normal((N, K) if tb else (K, N)).astype(np.float32))
    bias = inputs.to_bf16_bits(rng.uniform(-1, 1, N).astype(np.float32))
    c = sk.gemm_bf16_t(gu.dev_bf16(A), gu.dev_bf16(B), trans_a=ta, trans_b=tb,
                       bias=gu.dev_bf16(bias), mode="streamk")
    sk.stream_status()
    ref = gu.reference(oracle.gemm_bf16_t(A, ta, B, tb, bias=bias), "bf16")
    gu.assert_close(gu.host_values(c), ref, "bf16", f"ta={ta} tb={tb}")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", [(520, 264, 392), (256, 256, 512), (1040, 1024, 2048)])
def test_backward_integer_inputs_bit_exact(mode, shape):
    M, N, K = shape
    rng = np.random.default_rng(M * 3 + N + K)
    A, B, dC = _ints(rng, (M, K)), _ints(rng, (K, N)), _ints(rng, (M, N))
    da, db, dbias = sk.addmm_backward(gu.dev_bf16(dC), gu.dev_bf16(A), gu.dev_bf16(B),
                                      grad_dtype=torch.float32, mode=mode, num_sms=12)
    sk.stream_status()
    rA, rB, rb = oracle.addmm_backward_bf16(dC, A, B)
    assert np.array_equal(gu.host_values(da), rA)
    assert np.array_equal(gu.host_values(db), rB)
    assert np.array_equal(gu.host_values(dbias), rb)


def test_backward_random_bf16_grads_and_skipped_outputs():
    M, N, K = 1536, 1024, 768
    rng = np.random.default_rng(21)
    A = inputs.to_bf16_bits((rng.standard_normal((M, K)) / K ** 0.5).astype(np.float32))
    B = inputs.to_bf16_bits((rng.standard_normal((K, N)) / K ** 0.5).astype(np.float32))
    dC = inputs.to_bf16_bits(rng.standard_normal((M, N)).astype(np.float32))
    rA, rB, rb = oracle.addmm_backward_bf16(dC, A, B)
    da, db, dbias = sk.addmm_backward(gu.dev_bf16(dC), gu.dev_bf16(A), gu.dev_bf16(B))
    sk.stream_status()
    gu.assert_close(gu.host_values(da), gu.reference(rA, "bf16"), "bf16", "dA")
    gu.assert_close(gu.host_values(db), gu.reference(rB, "bf16"), "bf16", "dB")
    gu.assert_close(gu.host_values(dbias), gu.reference(rb, "bf16"), "bf16", "dbias")
    for need in (("a",), ("b",), ("bias",), ("a", "bias")):
        outs = sk.addmm_backward(gu.dev_bf16(dC), gu.dev_bf16(A), gu.dev_bf16(B), need=need)
        sk.stream_status()
        for name, got, ref in zip("a b bias".split(), outs, (rA, rB, rb)):
            assert (got is None) == (name not in need)
            if got is not None:
                gu.assert_close(gu.host_values(got), gu.reference(ref, "bf16"), "bf16", name)


def test_backward_of_the_8192_cube_sampled():
    p = inputs.workload("addmm_bf16_8192")
    rng = np.random.default_rng(5)
    dC = inputs.to_bf16_bits(rng.standard_normal((8192, 8192)).astype(np.float32))
    dCd, Ad, Bd = gu.dev_bf16(dC), gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"])
    da, db, dbias = sk.addmm_backward(dCd, Ad, Bd, grad_dtype=torch.float32)
    sk.stream_status()
    ms, ns = gu.sample_positions(8192, 8192, n_random=1024, n_rows=2, n_cols=2)
    idx = (torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda())
    # dA (M x K) = dC B^T; dB (K x N) = A^T dC
    refA = oracle.gemm_bf16_t_at(dC, 0, p["B"], 1, ms, ns)
    refB = oracle.gemm_bf16_t_at(p["A"], 1, dC, 0, ms, ns)
    gu.assert_close(da[idx].cpu().numpy().astype(np.float64), gu.reference(refA, "f32"), "f32", "dA")
    gu.assert_close(db[idx].cpu().numpy().astype(np.float64), gu.reference(refB, "f32"), "f32", "dB")
    refb = oracle.addmm_backward_bf16(dC[:, :64].copy(), p["A"][:, :8].copy(), p["B"][:8, :64].copy())[2]
    gu.assert_close(gu.host_values(dbias)[:64], gu.reference(refb, "f32"), "f32", "dbias")


def test_backward_argument_checks():
    P = 0x100000
    assert sk.sk_addmm_backward_bf16(None, P, P, P, P, P, 1, 64, 64, 64, 0, 2, None) == sk.SK_ERR_INVALID_ARG
    assert sk.sk_addmm_backward_bf16(P, P, P, None, None, None, 1, 64, 64, 64, 0, 2, None) == sk.SK_ERR_INVALID_ARG
    assert sk.sk_addmm_backward_bf16(P, P, P, P, P, P, 1, 64, 60, 64, 0, 2, None) == sk.SK_ERR_INVALID_ARG
    assert sk.sk_gemm_bf16_t(P, 2, P, 0, None, P, 1, 64, 64, 64, 0, 2, None, None) == sk.SK_ERR_INVALID_ARG
