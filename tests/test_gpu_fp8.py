"""GPU parity of the fp8 (E4M3) addmm path against the CPU oracle, through the C ABI."""
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


def run_fp8(p, out="bf16", mode="streamk", num_sms=0, options=None, stream=None):
    c = sk.gemm_fp8(gu.dev_u8(p["A"]), gu.dev_u8(p["B"]), gu.dev_bias(p["bias"]),
                    out_dtype=gu.out_torch_dtype(out), num_sms=num_sms, mode=mode,
                    options=options, stream=stream)
    sk.stream_status(stream)
    return c


def _want_bits(p, out):
    want = oracle.round_output(oracle.addmm_fp8(p["A"], p["B"], p["bias"]),
                               oracle.BF16 if out == "bf16" else oracle.F32)
    return want if out == "bf16" else want.view(np.uint32)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", [(128, 128, 128), (200, 144, 272), (300, 80, 96), (1, 16, 16),
                                   (257, 384, 1056), (64, 1008, 512), (640, 528, 800)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("tile", list(TILES))
def test_integer_inputs_are_bit_exact(mode, shape, out, tile):
    # integers in [-8, 8] are exact in E4M3 and every partial sum is exact in fp32 at these K;
    # the bias is an integer too, so the single final rounding is the only one
    M, N, K = shape
    p = inputs.fp8_problem(M, N, K, seed=M + 7 * N + 3 * K, integer=True,
                           bias="f32_int" if out == "f32" else "none")
    c = run_fp8(p, out=out, mode=mode, num_sms=12, options=TILES[tile])
    assert np.array_equal(gu.host_bits(c), _want_bits(p, out))


@pytest.mark.parametrize("shape,num_sms", [((300, 272, 16400), 16), ((300, 272, 16400), 64),
                                           ((520, 784, 8192), 152), ((512, 512, 16384), 152)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_split_pair_tiles_finished_by_several_pairs_are_bit_exact(shape, num_sms, out):
    # where at least two pairs have their whole Stream-K range in one tile, they finish a share
    # of its columns with the tile's owner (3 to 22 pairs per tile here)
    M, N, K = shape
    p = inputs.fp8_problem(M, N, K, seed=M + N + K, integer=True,
                           bias="f32_int" if out == "f32" else "none")
    for _ in range(2):
        c = run_fp8(p, out=out, mode="streamk", num_sms=num_sms, options=TILES["pair256"])
        assert np.array_equal(gu.host_bits(c), _want_bits(p, out))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("num_sms", [1, 3, 17, 0])
@pytest.mark.parametrize("tile", ["auto", "128x128", "pair256"])
def test_random_inputs_match_oracle(mode, num_sms, tile):
    p = inputs.fp8_problem(768, 528, 2048, seed=43, operand_scale="sqrt_k", bias="bf16_uniform")
    if tile == "pair256" and num_sms == 1:     # a pair tile needs two SMs
        with pytest.raises(sk.SkError):
            run_fp8(p, mode=mode, num_sms=1, options=TILES[tile])
        return
    c = run_fp8(p, out="bf16", mode=mode, num_sms=num_sms,
                options=None if tile == "auto" else TILES[tile])
    ref = gu.reference(oracle.addmm_fp8(p["A"], p["B"], p["bias"]), "bf16")
    gu.assert_close(gu.host_values(c), ref, "bf16", f"{mode}/{num_sms}/{tile}")


def test_float8_tensors_and_uint8_codes_give_the_same_result():
    p = inputs.fp8_problem(256, 256, 512, seed=5, operand_scale="sqrt_k", bias="f32_normal")
    a, b = gu.dev_u8(p["A"]), gu.dev_u8(p["B"])
    bias = gu.dev_bias(p["bias"])
    c8 = sk.gemm_fp8(a.view(torch.float8_e4m3fn), b.view(torch.float8_e4m3fn), bias,
                     out_dtype=torch.float32, num_sms=5)
    cu = sk.gemm_fp8(a, b, bias, out_dtype=torch.float32, num_sms=5)
    sk.stream_status()
    assert np.array_equal(gu.host_bits(c8), gu.host_bits(cu))
    ref = gu.reference(oracle.addmm_fp8(p["A"], p["B"], p["bias"]), "f32")
    gu.assert_close(gu.host_values(cu), ref, "f32")


@pytest.mark.parametrize("tile", list(TILES))
def test_nan_codes_propagate_to_their_row_and_column_only(tile):
    p = inputs.fp8_problem(512, 512, 512, seed=9, operand_scale="sqrt_k")
    p["B"][100, 300] = 0x7F          # S.1111.111 = NaN
    p["A"][37, 200] = 0xFF
    c = gu.host_values(run_fp8(p, out="f32", mode="streamk", num_sms=6, options=TILES[tile]))
    assert np.all(np.isnan(c[:, 300])) and np.all(np.isnan(c[37, :]))
    rest = np.delete(np.delete(c, 300, axis=1), 37, axis=0)
    assert not np.isnan(rest).any()


def test_extremes_stay_finite_and_subnormals_count():
    # 448 * 448 * 128 is exact and finite in fp32; products of the smallest subnormal (2^-9)
    # are exact in fp32 and must not be flushed to zero
    M, N, K = 128, 128, 256
    A = np.zeros((M, K), dtype=np.uint8)
    B = np.zeros((K, N), dtype=np.uint8)
    A[:64, :128] = 0x7E              # 448 in the first rows
    B[:128, :] = 0x7E
    A[64:, 128:] = 0x01              # 2^-9 in the others
    B[128:, :64] = 0x01
    p = {"A": A, "B": B, "bias": None}
    c = gu.host_bits(run_fp8(p, out="f32", mode="streamk", num_sms=2, options=TILES["128x128"]))
    assert np.array_equal(c, _want_bits(p, "f32"))
    v = c.view(np.float32)
    assert v[64, 0] == 2.0 ** -11 and v[0, 0] == 128 * 448.0 ** 2


def test_fp8_equals_bf16_path_on_decoded_operands():
    # the cross-format identity, GPU against GPU: E4M3 values are exact in bf16; with three
    # exponents the partial sums are exact in fp32, so both paths give the same bits
    M, N, K = 256, 384, 512
    rng = np.random.default_rng(17)

    def draw(shape):
        return rng.integers(-15, 16, shape) / 8.0 * np.exp2(rng.integers(-1, 2, shape))

    Af, Bf = draw((M, K)).astype(np.float32), draw((K, N)).astype(np.float32)
    bias = rng.standard_normal(N).astype(np.float32)
    p = {"A": inputs.to_e4m3_codes(Af), "B": inputs.to_e4m3_codes(Bf), "bias": bias}
    q = {"A": inputs.to_bf16_bits(Af), "B": inputs.to_bf16_bits(Bf), "bias": bias}
    f8 = gu.host_bits(run_fp8(p, out="f32", mode="streamk", num_sms=7))
    bf = gu.host_bits(gu.run_bf16(q, out="f32", mode="streamk", num_sms=7,
                                  options={"tile_n": 128}))
    assert np.array_equal(f8, bf)


def test_addmm_fp8_8192_cube_sampled():
    p = inputs.workload("addmm_fp8_8192")
    ms, ns = gu.sample_positions(p["M"], p["N"])
    ref = gu.reference(oracle.addmm_fp8_at(p["A"], p["B"], p["bias"], ms, ns), "bf16")
    a, b, bias = gu.dev_u8(p["A"]), gu.dev_u8(p["B"]), gu.dev_bias(p["bias"])
    for mode in MODES:
        c = sk.gemm_fp8(a, b, bias, mode=mode)
        sk.stream_status()
        got = c.float()[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()]
        gu.assert_close(got.cpu().numpy().astype(np.float64), ref, "bf16", mode)
        del c


def test_cuda_graph_replay_of_an_fp8_streamk_call():
    M, N, K = 768, 512, 2048
    s = torch.cuda.Stream()
    a = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    b = torch.empty((K, N), dtype=torch.uint8, device="cuda")
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    assert sk.sk_workspace_reserve(0, s.cuda_stream, 152) == sk.SK_OK
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sk.gemm_fp8(a, b, None, out=c, mode="streamk", stream=s)
    for seed in (1, 2):
        p = inputs.fp8_problem(M, N, K, seed=seed, integer=True)
        a.copy_(gu.dev_u8(p["A"]))
        b.copy_(gu.dev_u8(p["B"]))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert sk.sk_stream_status(s.cuda_stream) == sk.SK_OK
        assert np.array_equal(gu.host_bits(c), _want_bits(p, "f32"))
