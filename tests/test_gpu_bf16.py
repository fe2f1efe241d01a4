"""GPU parity of the bf16 addmm path against the CPU oracle, through the C ABI.

Covers every schedule (data-parallel, SM-constrained persistent, Stream-K, hybrid), both CTA
tile widths, fp32 and bf16 outputs, ragged shapes, a num_sms sweep, repeated launches, two
streams, CUDA-graph replay, a Stream-K wait that is made to run out, and the full-size
workloads on sampled outputs."""
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


# ---- the 256 x 256 x 512 fp32-output addmm: Stream-K over 3 CTAs, tiles split in K ----------

@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("num_sms", [3, 0])
def test_addmm_256_fp32_out_matches_oracle(mode, num_sms):
    p = inputs.workload("addmm_bf16_256x256x512_f32out")
    c = gu.run_bf16(p, out="f32", mode=mode, num_sms=num_sms)
    ref = gu.reference(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), "f32")
    gu.assert_close(gu.host_values(c), ref, "f32", f"{mode}/{num_sms}")


def test_addmm_256_streamk_over_3_ctas_splits_two_tiles():
    plan = sk.sk_plan(0, 256, 256, 512, 3, "streamk", torch.cuda.get_device_properties(0).multi_processor_count)
    segs = sk.sk_plan_segments(plan)
    assert plan.grid == 3 and plan.tile_n == 128
    assert (segs[:, 4] == 1).sum() == 2 and (segs[:, 4] == 2).sum() == 2


# ---- exact integer inputs: bit-exact in every schedule --------------------------------------

TILES = {"128x128": {"tile_m": 128, "tile_n": 128}, "128x256": {"tile_m": 128, "tile_n": 256},
         "pair256": {"tile_m": 256}}


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", [(200, 136, 200), (1, 8, 8), (128, 128, 64), (129, 264, 72),
                                   (384, 1024, 512), (640, 256, 8), (520, 776, 1000)])
@pytest.mark.parametrize("tile", list(TILES))
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_integer_inputs_are_bit_exact(mode, shape, tile, out):
    M, N, K = shape
    p = inputs.bf16_problem(M, N, K, seed=M + 7 * N + 13 * K, integer=True,
                            bias="bf16_int" if out == "bf16" else "f32_int")
    c = gu.run_bf16(p, out=out, mode=mode, num_sms=10, options=TILES[tile])
    want = oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], p["bias"]),
                               oracle.BF16 if out == "bf16" else oracle.F32)
    want_bits = want if out == "bf16" else want.view(np.uint32)
    assert np.array_equal(gu.host_bits(c), want_bits)


@pytest.mark.parametrize("mode", ["persistent", "streamk", "hybrid"])
@pytest.mark.parametrize("num_sms", [1, 2, 3, 7, 16, 64, 151, 152, 0, 1000])
@pytest.mark.parametrize("tile", ["auto", "pair256"])
def test_num_sms_sweep_integer_bit_exact(mode, num_sms, tile):
    if tile == "pair256" and 0 < num_sms < 2:
        pytest.skip("a pair needs two SMs")
    p = inputs.bf16_problem(1040, 776, 1000, seed=77, integer=True, bias="bf16_int")
    c = gu.run_bf16(p, out="bf16", mode=mode, num_sms=num_sms,
                    options=None if tile == "auto" else TILES[tile])
    want = oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), oracle.BF16)
    assert np.array_equal(gu.host_bits(c), want)


def test_no_bias_and_zero_a_give_bias_rows():
    M, N, K = 300, 264, 136
    p = inputs.bf16_problem(M, N, K, seed=3, bias="bf16_uniform")
    p["A"] = np.zeros_like(p["A"])
    for mode in MODES:
        c = gu.run_bf16(p, out="bf16", mode=mode, num_sms=7)
        assert np.array_equal(gu.host_bits(c), np.broadcast_to(p["bias"], (M, N)))
    p["bias"] = None
    c = gu.run_bf16(p, out="f32", mode="streamk", num_sms=7)
    assert not gu.host_values(c).any()


# ---- random inputs --------------------------------------------------------------------------

@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("tile", list(TILES))
def test_random_inputs_match_oracle(mode, tile):
    p = inputs.bf16_problem(640, 896, 1544, seed=5, operand_scale="sqrt_k", bias="bf16_uniform")
    c = gu.run_bf16(p, out="bf16", mode=mode, num_sms=0, options=TILES[tile])
    ref = gu.reference(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), "bf16")
    gu.assert_close(gu.host_values(c), ref, "bf16", mode)


def test_streamk_and_dp_outputs_agree():
    p = inputs.bf16_problem(768, 512, 4096, seed=6, operand_scale="sqrt_k", bias="f32_normal")
    outs = {m: gu.host_values(gu.run_bf16(p, out="f32", mode=m, num_sms=0)) for m in MODES}
    for m in MODES:
        gu.assert_close(outs[m], outs["dp"], "f32", f"{m} vs dp")


# ---- launch hygiene -------------------------------------------------------------------------

def test_repeated_streamk_launches_on_one_stream_are_identical():
    p = inputs.bf16_problem(512, 512, 2048, seed=8, bias="bf16_uniform")
    a, b, bias = gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"]), gu.dev_bias(p["bias"])
    outs = [sk.gemm_bf16(a, b, bias, mode="streamk", num_sms=37) for _ in range(6)]
    sk.stream_status()
    first = gu.host_bits(outs[0])
    for o in outs[1:]:
        assert np.array_equal(gu.host_bits(o), first)
    ref = gu.reference(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), "bf16")
    gu.assert_close(gu.host_values(outs[0]), ref, "bf16")


def test_two_streams_run_concurrently_with_separate_workspaces():
    ps = [inputs.bf16_problem(640, 512, 3072, seed=s, bias="bf16_uniform") for s in (11, 12)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    devs = [(gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"]), gu.dev_bias(p["bias"])) for p in ps]
    torch.cuda.synchronize()
    outs = []
    for _ in range(3):
        for (a, b, bias), s in zip(devs, streams):
            with torch.cuda.stream(s):
                outs.append(sk.gemm_bf16(a, b, bias, mode="streamk", num_sms=60, stream=s))
    for s in streams:
        sk.stream_status(s)
    for i, o in enumerate(outs):
        p = ps[i % 2]
        ref = gu.reference(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), "bf16")
        gu.assert_close(gu.host_values(o), ref, "bf16", f"call {i}")


def test_cuda_graph_replay_reuses_the_workspace():
    # A captured launch keeps one flag epoch; the owners reset consumed flags, so every
    # replay must still wait for fresh partials.
    M, N, K = 512, 768, 2048
    s = torch.cuda.Stream()
    a = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    b = torch.empty((K, N), dtype=torch.bfloat16, device="cuda")
    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert sk.sk_workspace_reserve(0, s.cuda_stream, 152) == sk.SK_OK
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sk.gemm_bf16(a, b, None, out=c, mode="streamk", num_sms=0, stream=s)
    for seed in (1, 2, 3):
        p = inputs.bf16_problem(M, N, K, seed=seed, integer=True)
        a.copy_(gu.dev_bf16(p["A"]))
        b.copy_(gu.dev_bf16(p["B"]))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert sk.sk_stream_status(s.cuda_stream) == sk.SK_OK
        want = oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], None), oracle.BF16)
        assert np.array_equal(gu.host_bits(c), want)


def test_capture_without_reserved_workspace_is_refused():
    s = torch.cuda.Stream()
    a = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    c = torch.empty((256, 256), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    st = None
    with torch.cuda.graph(g, stream=s):
        st = sk.sk_gemm_bf16(a.data_ptr(), a.data_ptr(), None, c.data_ptr(), 1, 256, 256, 256,
                             0, 2, s.cuda_stream)
    assert st == sk.SK_ERR_UNSUPPORTED


def test_pair_streamk_wait_that_runs_out_reports_timeout():
    # 2048 x 256 x 4096 on 3 pairs: pair 1 (CTAs 2, 3) continues the tile pair 0 owns; CTA 3
    # never publishes, so CTA 1 (the rank-1 half of the owner) times out.
    p = inputs.bf16_problem(2048, 256, 4096, seed=4, bias="bf16_uniform")
    a, b, bias = gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"]), gu.dev_bias(p["bias"])
    plan = sk.sk_plan(0, 2048, 256, 4096, 6, "streamk", 152, {"tile_m": 256})
    segs = sk.sk_plan_segments(plan)
    assert plan.ctas_per_tile == 2 and plan.grid == 3
    contrib = segs[(segs[:, 0] == 1) & (segs[:, 4] == 2)]   # pair 1's contribution ...
    owner = segs[(segs[:, 0] == 0) & (segs[:, 4] == 1)]     # ... to the tile pair 0 shares
    assert len(contrib) == 1 and len(owner) == 1 and contrib[0, 1] == owner[0, 1]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        sk.gemm_bf16(a, b, bias, mode="streamk", num_sms=6, stream=s,
                     options={"tile_m": 256, "inject_faults": 1, "drop_release_cta": 3,
                              "spin_timeout_ns": 20_000_000})
    assert sk.sk_stream_status(s.cuda_stream) == sk.SK_ERR_TIMEOUT
    c = gu.run_bf16(p, out="bf16", mode="streamk", num_sms=6, stream=s, options={"tile_m": 256})
    ref = gu.reference(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), "bf16")
    gu.assert_close(gu.host_values(c), ref, "bf16")


def test_device_caps_write_only_their_structure():
    # the structure sits between canary bytes; the call must leave them untouched
    import ctypes
    size = ctypes.sizeof(sk.DeviceCaps)
    buf = (ctypes.c_uint8 * (size + 256))()
    ctypes.memset(buf, 0xA5, size + 256)
    st = sk.lib().sk_device_caps(0, ctypes.cast(ctypes.byref(buf, 0), ctypes.POINTER(sk.DeviceCaps)))
    assert st == sk.SK_OK
    assert bytes(buf[size:]) == b"\xa5" * 256


def test_device_caps_report_the_pair_capacity():
    caps = sk.sk_device_caps(0)
    assert caps["cc"] == (10, 3)
    assert caps["setup_error"] == [0] * 5
    assert all(n >= 1 for n in caps["ctas_per_sm"])
    assert all(2 * n <= caps["sm_count"] and n >= 1 for n in caps["max_pair_clusters"])
    assert caps["fp8_setup_error"] == [0] * 3
    assert all(n >= 1 for n in caps["fp8_ctas_per_sm"])
    assert 1 <= caps["fp8_max_pair_clusters"] and 2 * caps["fp8_max_pair_clusters"] <= caps["sm_count"]


def test_streamk_wait_that_runs_out_reports_timeout():
    # CTA 1 contributes to tile 1, owned by CTA 0; it is told never to publish its partial.
    p = inputs.workload("addmm_bf16_256x256x512_f32out")
    a, b, bias = gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"]), gu.dev_bias(p["bias"])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        sk.gemm_bf16(a, b, bias, out_dtype=torch.float32, mode="streamk", num_sms=3, stream=s,
                     options={"inject_faults": 1, "drop_release_cta": 1,
                              "spin_timeout_ns": 20_000_000})
    assert sk.sk_stream_status(s.cuda_stream) == sk.SK_ERR_TIMEOUT
    assert sk.sk_stream_status(s.cuda_stream) == sk.SK_OK      # cleared once read
    c = gu.run_bf16(p, out="f32", mode="streamk", num_sms=3, stream=s)   # recovers
    ref = gu.reference(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), "f32")
    gu.assert_close(gu.host_values(c), ref, "f32")


# ---- full-size workloads, sampled outputs -------------------------------------------------

def _sampled_check(p, out, modes, num_sms_list=(0,)):
    ms, ns = gu.sample_positions(p["M"], p["N"])
    ref = gu.reference(oracle.addmm_bf16_at(p["A"], p["B"], p["bias"], ms, ns), out)
    a, b, bias = gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"]), gu.dev_bias(p["bias"])
    for mode in modes:
        for ns_ in num_sms_list:
            c = sk.gemm_bf16(a, b, bias, out_dtype=gu.out_torch_dtype(out), mode=mode, num_sms=ns_)
            sk.stream_status()
            got = c.float()[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()]
            gu.assert_close(got.cpu().numpy().astype(np.float64), ref, out, f"{mode}/{ns_}")
            del c


def test_addmm_8192_cube_sampled():
    _sampled_check(inputs.workload("addmm_bf16_8192"), "bf16", MODES)


def test_wave_quantised_1920x1920x16384_sampled():
    _sampled_check(inputs.workload("gemm_bf16_1920x1920x16384"), "bf16", MODES)


def test_4096_cube_num_sms_sweep_sampled():
    _sampled_check(inputs.workload("gemm_bf16_4096"), "bf16", ["persistent", "streamk"],
                   (1, 16, 32, 64, 128, 0))


def test_skinny_64x14336x4096_num_sms_sweep_sampled():
    _sampled_check(inputs.workload("gemm_bf16_skinny_64x14336x4096"), "bf16",
                   ["dp", "persistent", "streamk", "hybrid"], (1, 16, 32, 64, 128, 0))


# ---- matrices of at most 64 rows (one partly filled row of tiles) ---------------------------

@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", [(1, 136, 512), (17, 1000, 1088), (64, 256, 4096),
                                   (64, 14336, 256), (63, 8, 64)])
@pytest.mark.parametrize("num_sms", [0, 5])
def test_at_most_64_rows_integer_inputs_are_bit_exact(mode, shape, num_sms):
    M, N, K = shape
    p = inputs.bf16_problem(M, N, K, seed=M * 7 + N + K, integer=True, bias="f32_int")
    c = gu.run_bf16(p, out="f32", mode=mode, num_sms=num_sms, options={"tile_n": 128})
    want = oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), oracle.F32)
    assert np.array_equal(gu.host_bits(c), want.view(np.uint32))


def test_at_most_64_rows_random_bf16_output_matches_oracle():
    p = inputs.bf16_problem(48, 2048, 8192, seed=12, operand_scale="sqrt_k", bias="bf16_uniform")
    for mode in MODES:
        c = gu.run_bf16(p, out="bf16", mode=mode)
        ref = gu.reference(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), "bf16")
        gu.assert_close(gu.host_values(c), ref, "bf16", mode)


# ---- tall stages (128 K per stage) for at most 64 rows of A ----------------------------------

@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", [(64, 14336, 4104), (33, 1000, 136), (1, 256, 8), (64, 96, 4096),
                                   (64, 8, 64), (17, 2000, 1032)])
@pytest.mark.parametrize("tile_n", [96, 128])
@pytest.mark.parametrize("num_sms", [0, 7, 37])
def test_tall_stages_are_bit_exact_and_equal_64k_stages(mode, shape, tile_n, num_sms):
    M, N, K = shape
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    opts = {"tile_m": 128, "tile_n": tile_n}
    plan = sk.sk_plan(0, M, N, K, num_sms, mode, sms, opts)
    assert plan.tile_k == 128 and plan.iters == -(-K // 128)
    p = inputs.bf16_problem(M, N, K, seed=M + 5 * N + 3 * K + tile_n, integer=True, bias="f32_int")
    want = oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), oracle.F32)
    tall = gu.run_bf16(p, out="f32", mode=mode, num_sms=num_sms, options=opts)
    assert np.array_equal(gu.host_bits(tall), want.view(np.uint32))
    short = gu.run_bf16(p, out="f32", mode=mode, num_sms=num_sms, options=dict(opts, tile_k=64))
    assert np.array_equal(gu.host_bits(short), gu.host_bits(tall))


def test_tall_stages_random_bf16_output_matches_oracle():
    p = inputs.bf16_problem(64, 3000, 8200, seed=21, operand_scale="sqrt_k", bias="bf16_uniform")
    for mode in MODES:
        for tile_n in (96, 128):
            c = gu.run_bf16(p, out="bf16", mode=mode, options={"tile_m": 128, "tile_n": tile_n})
            ref = gu.reference(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), "bf16")
            gu.assert_close(gu.host_values(c), ref, "bf16", f"tall/{mode}/{tile_n}")


# ---- the two-tile hybrid (full waves added to the Stream-K region) --------------------------

@pytest.mark.parametrize("shape", [(2304, 2304, 1024), (1000, 3000, 640), (520, 776, 1000)])
@pytest.mark.parametrize("tile", ["128x128", "pair256"])
@pytest.mark.parametrize("num_sms,waves", [(0, 1), (14, 1), (14, 2)])
def test_two_tile_hybrid_integer_inputs_are_bit_exact(shape, tile, num_sms, waves):
    M, N, K = shape
    p = inputs.bf16_problem(M, N, K, seed=M + N + waves, integer=True, bias="f32_int")
    c = gu.run_bf16(p, out="f32", mode="hybrid", num_sms=num_sms,
                    options=dict(TILES[tile], hybrid_sk_waves=waves))
    want = oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), oracle.F32)
    assert np.array_equal(gu.host_bits(c), want.view(np.uint32))


def test_whole_tile_grids_are_captured_beyond_the_reserved_grid():
    # data-parallel and persistent launches split no tile: they need no Stream-K flags or
    # slots, so a grid larger than the one reserved is still captured
    M = N = 2048
    K = 512
    s = torch.cuda.Stream()
    a = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    b = torch.empty((K, N), dtype=torch.bfloat16, device="cuda")
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    assert sk.sk_workspace_reserve(0, s.cuda_stream, 8) == sk.SK_OK
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sk.gemm_bf16(a, b, None, out=c, out_dtype=torch.float32, mode="dp",
                     options={"tile_m": 128, "tile_n": 128}, stream=s)   # 256 CTAs
    p = inputs.bf16_problem(M, N, K, seed=4, integer=True)
    a.copy_(gu.dev_bf16(p["A"]))
    b.copy_(gu.dev_bf16(p["B"]))
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    want = oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], None), oracle.F32)
    assert np.array_equal(gu.host_bits(c), want.view(np.uint32))


@pytest.mark.parametrize("mode", ["streamk", "hybrid"])
@pytest.mark.parametrize("shape,tile,num_sms", [
    ((512, 512, 8192), "pair256", 0),      # 4 pair tiles on 76 pairs: ~19 pieces per tile
    ((1920, 1920, 2048), "pair256", 0),    # 64 tiles on 76 pairs: pairs working inside one tile
    ((1920, 1920, 2048), "pair256", 90),   # 45 pairs
    ((640, 640, 4096), "128x256", 0),      # 15 tiles on 152 CTAs: ~10 pieces per tile
    ((512, 512, 8192), "128x128", 0),      # 16 tiles on 152 CTAs
    ((1920, 1920, 2048), "128x128", 7),    # long ranges over many tiles on 7 CTAs
])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_streamk_fixup_with_many_and_late_contributors_is_bit_exact(mode, shape, tile, num_sms, out):
    # Every partial must be added exactly once, whether the owner summed it into its idle
    # accumulator during its k-loop or read it in its drain: exact on integer inputs.
    M, N, K = shape
    p = inputs.bf16_problem(M, N, K, seed=M + N + K + num_sms, integer=True,
                            bias="bf16_int" if out == "bf16" else "f32_int")
    plan = sk.sk_plan(0, M, N, K, num_sms, mode, torch.cuda.get_device_properties(0).multi_processor_count,
                      TILES[tile])
    assert plan.sk_tiles > 0
    want = oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], p["bias"]),
                               oracle.BF16 if out == "bf16" else oracle.F32)
    want_bits = want if out == "bf16" else want.view(np.uint32)
    for _ in range(2):   # the second launch finds the first one's flags (cleared or left set)
        c = gu.run_bf16(p, out=out, mode=mode, num_sms=num_sms, options=TILES[tile])
        assert np.array_equal(gu.host_bits(c), want_bits)


# ---- split pair tiles finished by several pairs ---------------------------------------------

def finishing_parties(plan):
    """{tile: number of pairs that finish its columns} for the split tiles of a Stream-K plan
    without whole tiles: the owner plus each contributor whose only piece is its piece of the
    tile, when there are at least two such contributors; else the owner alone."""
    segs = sk.sk_plan_segments(plan)
    pieces = np.bincount(segs[:, 0], minlength=plan.grid)
    out = {}
    for tile in np.unique(segs[segs[:, 4] == 1, 1]):
        contrib = segs[(segs[:, 1] == tile) & (segs[:, 4] == 2), 0]
        finishers = int((pieces[contrib] == 1).sum())
        out[int(tile)] = 1 + finishers if finishers >= 2 else 1
    return out


@pytest.mark.parametrize("shape,num_sms,parties", [
    ((300, 264, 8200), 16, {1, 3}),        # ragged M, N and K
    ((300, 264, 8200), 40, {4, 5, 6}),
    ((300, 264, 8200), 64, {7, 8, 9}),     # more parties than the tile's eight column chunks
    ((520, 776, 4096), 152, {5, 6, 7}),
    ((256, 256, 16384), 152, {76}),        # one tile, every pair on it
])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_tiles_finished_by_several_pairs_are_bit_exact(shape, num_sms, parties, out):
    M, N, K = shape
    plan = sk.sk_plan(0, M, N, K, num_sms, "streamk", torch.cuda.get_device_properties(0).multi_processor_count,
                      TILES["pair256"])
    assert plan.ctas_per_tile == 2 and set(finishing_parties(plan).values()) == parties
    p = inputs.bf16_problem(M, N, K, seed=M + N + K + num_sms, integer=True,
                            bias="bf16_int" if out == "bf16" else "f32_int")
    want = oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], p["bias"]),
                               oracle.BF16 if out == "bf16" else oracle.F32)
    want_bits = want if out == "bf16" else want.view(np.uint32)
    for _ in range(2):
        c = gu.run_bf16(p, out=out, mode="streamk", num_sms=num_sms, options=TILES["pair256"])
        assert np.array_equal(gu.host_bits(c), want_bits)


@pytest.mark.parametrize("bias,out", [("bf16_uniform", "bf16"), ("none", "bf16"), ("f32_normal", "f32")])
def test_tiles_finished_by_several_pairs_random_inputs_match_oracle(bias, out):
    p = inputs.bf16_problem(512, 512, 8192, seed=31, operand_scale="sqrt_k", bias=bias)
    c = gu.run_bf16(p, out=out, mode="streamk", num_sms=38, options=TILES["pair256"])
    ref = gu.reference(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), out)
    gu.assert_close(gu.host_values(c), ref, out)


@pytest.mark.parametrize("dropped", ["finisher", "owner"])
def test_shared_finish_wait_that_runs_out_reports_timeout(dropped):
    # 512 x 512 x 4096 on 10 pairs: two split tiles are finished by their owner and two
    # finishers.  A dropped finisher leaves the owner and the other finisher waiting for its
    # partial; a dropped owner leaves the finishers waiting for the owner's share.
    M, N, K = 512, 512, 4096
    opts = dict(TILES["pair256"])
    plan = sk.sk_plan(0, M, N, K, 20, "streamk", torch.cuda.get_device_properties(0).multi_processor_count, opts)
    parties = finishing_parties(plan)
    assert set(parties.values()) == {1, 3}
    segs = sk.sk_plan_segments(plan)
    tile = min(t for t, n in parties.items() if n == 3)
    owner = int(segs[(segs[:, 1] == tile) & (segs[:, 4] == 1), 0][0])
    drop_pair = owner if dropped == "owner" else owner + 1
    p = inputs.bf16_problem(M, N, K, seed=9, integer=True, bias="bf16_int")
    a, b, bias = gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"]), gu.dev_bias(p["bias"])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        sk.gemm_bf16(a, b, bias, mode="streamk", num_sms=20, stream=s,
                     options={**opts, "inject_faults": 1, "drop_release_cta": 2 * drop_pair,
                              "spin_timeout_ns": 20_000_000})
    assert sk.sk_stream_status(s.cuda_stream) == sk.SK_ERR_TIMEOUT
    c = gu.run_bf16(p, out="bf16", mode="streamk", num_sms=20, stream=s, options=opts)
    want = oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), oracle.BF16)
    assert np.array_equal(gu.host_bits(c), want)


# ---- 96-wide tiles (one row of tiles streaming B over more SMs) -----------------------------

@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", [(64, 14336, 512), (128, 96, 64), (100, 200, 136), (1, 8, 8),
                                   (128, 1000, 1024), (300, 776, 520)])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_96_wide_tiles_integer_inputs_are_bit_exact(mode, shape, out):
    M, N, K = shape
    p = inputs.bf16_problem(M, N, K, seed=M + 3 * N + 5 * K, integer=True,
                            bias="bf16_int" if out == "bf16" else "f32_int")
    c = gu.run_bf16(p, out=out, mode=mode, num_sms=37, options={"tile_m": 128, "tile_n": 96})
    want = oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], p["bias"]),
                               oracle.BF16 if out == "bf16" else oracle.F32)
    assert np.array_equal(gu.host_bits(c), want.view(np.uint16 if out == "bf16" else np.uint32))


@pytest.mark.parametrize("mode", ["persistent", "streamk", "hybrid"])
def test_96_wide_tiles_skinny_shape_matches_oracle(mode):
    p = inputs.workload("gemm_bf16_skinny_64x14336x4096")
    c = gu.run_bf16(p, out="bf16", mode=mode, options={"tile_m": 128, "tile_n": 96})
    plan = sk.sk_plan(0, 64, 14336, 4096, 0, mode, torch.cuda.get_device_properties(0).multi_processor_count,
                      {"tile_m": 128, "tile_n": 96})
    assert plan.tile_n == 96 and plan.tiles == 150
    ref = gu.reference(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), "bf16")
    gu.assert_close(gu.host_values(c), ref, "bf16", f"skinny/{mode}/96")


def test_96_wide_tiles_only_for_plain_bf16():
    a = torch.zeros((128, 128), dtype=torch.bfloat16, device="cuda")
    c = torch.empty((128, 128), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    opts = {"tile_m": 128, "tile_n": 96}
    st = sk.sk_gemm_bf16_t(a.data_ptr(), 1, a.data_ptr(), 0, None, c.data_ptr(), sk.SK_BF16,
                           128, 128, 128, 0, sk.MODES["persistent"], opts, stream)
    assert st == sk.SK_ERR_INVALID_ARG
    u = torch.zeros((128, 128), dtype=torch.uint8, device="cuda")
    st = sk.sk_gemm_fp8_ex(u.data_ptr(), u.data_ptr(), None, c.data_ptr(), sk.SK_BF16, 128, 128,
                           128, 0, sk.MODES["persistent"], opts, stream)
    assert st == sk.SK_ERR_INVALID_ARG
