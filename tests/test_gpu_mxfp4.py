"""GPU parity of the MXFP4 addmm path against the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
import sm_constrained_persistent_gb300 as sk
from sm_constrained_persistent_gb300 import inputs

pytestmark = pytest.mark.gpu
MODES = ["dp", "persistent", "streamk", "hybrid"]


@pytest.fixture(autouse=True)
def _device(cuda_device):
    yield


TILES = {"128x128": {"tile_m": 128}, "pair256": {"tile_m": 256}}


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", [(128, 128, 256), (200, 136, 288), (300, 77, 96), (1, 1, 32),
                                   (257, 383, 1056), (64, 1000, 512), (640, 520, 800)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("tile", list(TILES))
def test_small_scale_range_is_bit_exact(mode, shape, out, tile):
    # scale exponents in [-1, 1]: every partial sum is exact in fp32 at these K, so the only
    # rounding is the final one (an fp32 bias is added in that same single rounding; a bf16
    # output gets no bias here, since fp32 add then bf16 cast would round twice)
    M, N, K = shape
    p = inputs.mxfp4_problem(M, N, K, seed=M * 3 + N * 5 + K, exp_range=1,
                             bias="none" if out == "bf16" else "f32_normal")
    c = gu.run_mxfp4(p, out=out, mode=mode, num_sms=12, options=TILES[tile])
    want = oracle.round_output(
        oracle.addmm_mxfp4(p["A"], p["A_scale"], p["B"], p["B_scale"], p["bias"]),
        oracle.BF16 if out == "bf16" else oracle.F32)
    assert np.array_equal(gu.host_bits(c), want if out == "bf16" else want.view(np.uint32))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("num_sms", [1, 3, 17, 0])
@pytest.mark.parametrize("tile", ["auto", "128x128"])
def test_full_scale_range_matches_oracle(mode, num_sms, tile):
    p = inputs.mxfp4_problem(768, 520, 2048, seed=41, exp_range=4, bias="bf16_uniform")
    c = gu.run_mxfp4(p, out="bf16", mode=mode, num_sms=num_sms,
                     options=None if tile == "auto" else TILES[tile])
    ref = gu.reference(oracle.addmm_mxfp4(p["A"], p["A_scale"], p["B"], p["B_scale"], p["bias"]),
                       "bf16")
    gu.assert_close(gu.host_values(c), ref, "bf16", f"{mode}/{num_sms}")


@pytest.mark.parametrize("tile", list(TILES))
def test_nan_scale_propagates_to_its_column_only(tile):
    p = inputs.mxfp4_problem(512, 512, 512, seed=9, exp_range=2)
    p["B_scale"][300, 3] = 255
    c = gu.host_values(gu.run_mxfp4(p, out="f32", mode="streamk", num_sms=6, options=TILES[tile]))
    assert np.all(np.isnan(c[:, 300]))
    assert not np.isnan(np.delete(c, 300, axis=1)).any()


def test_mxfp4_equals_bf16_path_on_decoded_operands():
    # the cross-format identity, GPU against GPU: decoded MX values are exact in bf16
    M, N, K = 256, 384, 512
    p = inputs.mxfp4_problem(M, N, K, seed=13, exp_range=1, bias="f32_normal")
    table = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                      -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0], dtype=np.float32)

    def decode(codes, scales):
        lo, hi = codes & 0xF, codes >> 4
        vals = np.empty((codes.shape[0], K), dtype=np.float32)
        vals[:, 0::2], vals[:, 1::2] = table[lo], table[hi]
        return vals * np.exp2(np.repeat(scales.astype(np.float32) - 127, 32, axis=1))

    q = {"A": inputs.to_bf16_bits(decode(p["A"], p["A_scale"])),
         "B": inputs.to_bf16_bits(decode(p["B"], p["B_scale"]).T.copy()), "bias": p["bias"]}
    mx = gu.host_bits(gu.run_mxfp4(p, out="f32", mode="streamk", num_sms=7))
    bf = gu.host_bits(gu.run_bf16(q, out="f32", mode="streamk", num_sms=7, options={"tile_n": 128}))
    assert np.array_equal(mx, bf)


def test_repeated_calls_reuse_the_scale_workspace():
    ps = [inputs.mxfp4_problem(512, 512, 1024, seed=s, exp_range=1) for s in (1, 2)]
    for _ in range(2):
        for p in ps:
            c = gu.run_mxfp4(p, out="f32", mode="streamk", num_sms=19)
            want = oracle.round_output(oracle.addmm_mxfp4(p["A"], p["A_scale"], p["B"], p["B_scale"]),
                                       oracle.F32)
            assert np.array_equal(gu.host_bits(c), want.view(np.uint32))


def test_addmm_mxfp4_8192_cube_sampled():
    p = inputs.workload("addmm_mxfp4_8192")
    ms, ns = gu.sample_positions(p["M"], p["N"])
    ref = gu.reference(oracle.addmm_mxfp4_at(p["A"], p["A_scale"], p["B"], p["B_scale"], p["bias"],
                                             ms, ns), "bf16")
    a, sa = gu.dev_u8(p["A"]), gu.dev_u8(p["A_scale"])
    b, sb = gu.dev_u8(p["B"]), gu.dev_u8(p["B_scale"])
    bias = gu.dev_bias(p["bias"])
    for mode in MODES:
        c = sk.gemm_mxfp4(a, sa, b, sb, bias, mode=mode)
        sk.stream_status()
        got = c.float()[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()]
        gu.assert_close(got.cpu().numpy().astype(np.float64), ref, "bf16", mode)


def test_cuda_graph_replay_of_an_mxfp4_streamk_call():
    # the scale re-layout buffer and the Stream-K slots are reserved before capture
    M, N, K = 768, 512, 2048
    s = torch.cuda.Stream()
    a = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    b = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
    asc = torch.empty((M, K // 32), dtype=torch.uint8, device="cuda")
    bsc = torch.empty((N, K // 32), dtype=torch.uint8, device="cuda")
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    assert sk.sk_workspace_reserve(0, s.cuda_stream, 152, M, N, K) == sk.SK_OK
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sk.gemm_mxfp4(a, asc, b, bsc, None, out=c, mode="streamk", stream=s)
    for seed in (1, 2):
        p = inputs.mxfp4_problem(M, N, K, seed=seed, exp_range=1)
        for dst, src in ((a, "A"), (b, "B"), (asc, "A_scale"), (bsc, "B_scale")):
            dst.copy_(gu.dev_u8(p[src]))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert sk.sk_stream_status(s.cuda_stream) == sk.SK_OK
        want = oracle.round_output(
            oracle.addmm_mxfp4(p["A"], p["A_scale"], p["B"], p["B_scale"], None), oracle.F32)
        assert np.array_equal(gu.host_bits(c), want.view(np.uint32))
