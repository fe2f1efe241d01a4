"""CPU checks of the C-ABI library: it builds, loads, exports every function the header
declares, rejects bad arguments before touching CUDA, and its scheduler (the code the kernels
run) produces the same work split as the oracle's independent restatement."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import sm_constrained_persistent_gb300 as sk
from sm_constrained_persistent_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return sk.lib()


def _declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(sk_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ["sk_gemm_bf16", "sk_gemm_mxfp4", "sk_stream_status", "sk_workspace_reserve",
                     "sk_workspace_release_all", "sk_workspace_release", "sk_status_string",
                     "sk_plan", "sk_plan_segments",
                     "sk_gemm_bf16_ex", "sk_gemm_mxfp4_ex", "sk_gemm_fp8", "sk_gemm_fp8_ex",
                     "sk_gemm_bf16_host", "sk_gemm_fp8_host", "sk_gemm_mxfp4_host",
                     "sk_autotune"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(7):
        assert sk.sk_status_string(code)
    assert sk.sk_status_string(99) == "unknown status"


P = 0x100000  # a 16-byte aligned fake device address: never dereferenced by these tests


@pytest.mark.parametrize("args", [
    dict(A=None), dict(B=None), dict(C=None),
    dict(A=P + 8), dict(B=P + 2), dict(C=P + 4), dict(bias=P + 1),
    dict(M=0), dict(N=0), dict(K=0), dict(M=-5), dict(K=2 ** 31),
    dict(K=100), dict(N=100),            # bf16 needs 16-byte row pitches
    dict(out_dtype=2), dict(mode=5), dict(mode=-1),
])
def test_bf16_bad_arguments_are_rejected_before_cuda(lib, args):
    a = dict(A=P, B=P, bias=None, C=P, out_dtype=1, M=64, N=64, K=64, num_sms=0, mode=2)
    a.update(args)
    st = sk.sk_gemm_bf16(a["A"], a["B"], a["bias"], a["C"], a["out_dtype"], a["M"], a["N"],
                         a["K"], a["num_sms"], a["mode"], None)
    assert st == sk.SK_ERR_INVALID_ARG


@pytest.mark.parametrize("args", [
    dict(A_scale=None), dict(B_scale=None), dict(K=48), dict(K=16), dict(tile_n=256),
    dict(tile_n=64),
])
def test_mxfp4_bad_arguments_are_rejected_before_cuda(lib, args):
    a = dict(A=P, A_scale=P, B=P, B_scale=P, C=P, M=10, N=30, K=64, tile_n=0)
    a.update(args)
    opts = {"tile_n": a["tile_n"]}
    st = sk.sk_gemm_mxfp4_ex(a["A"], a["A_scale"], a["B"], a["B_scale"], None, a["C"], 1,
                             a["M"], a["N"], a["K"], 0, 2, opts, None)
    assert st == sk.SK_ERR_INVALID_ARG


@pytest.mark.parametrize("args", [
    dict(A=None), dict(B=None), dict(C=None), dict(A=P + 1), dict(B=P + 8),
    dict(K=8), dict(K=40), dict(N=24), dict(M=0), dict(out_dtype=3), dict(mode=7),
    dict(tile_n=64), dict(tile_m=256, tile_n=128),
])
def test_fp8_bad_arguments_are_rejected_before_cuda(lib, args):
    a = dict(A=P, B=P, C=P, M=10, N=32, K=64, out_dtype=1, mode=2, tile_n=0, tile_m=0)
    a.update(args)
    opts = {"tile_n": a["tile_n"], "tile_m": a["tile_m"]}
    st = sk.sk_gemm_fp8_ex(a["A"], a["B"], None, a["C"], a["out_dtype"], a["M"], a["N"], a["K"],
                           0, a["mode"], opts, None)
    assert st == sk.SK_ERR_INVALID_ARG
    if not args.get("tile_n") and not args.get("tile_m"):
        st = sk.sk_gemm_fp8(a["A"], a["B"], None, a["C"], a["out_dtype"], a["M"], a["N"], a["K"],
                            0, a["mode"], None)
        assert st == sk.SK_ERR_INVALID_ARG


@pytest.mark.parametrize("fmt,args", [
    ("bf16", dict(A=None)), ("bf16", dict(C=None)), ("bf16", dict(K=100)), ("bf16", dict(N=20)),
    ("bf16", dict(M=0)), ("bf16", dict(out_dtype=2)), ("fp8", dict(K=40)), ("fp8", dict(N=24)),
    ("mxfp4", dict(K=48)), ("mxfp4", dict(A_scale=None)),
])
def test_host_buffer_calls_reject_bad_arguments_before_copying(lib, fmt, args):
    a = dict(A=P, A_scale=P, B=P, B_scale=P, C=P, M=64, N=64, K=64, out_dtype=1)
    a.update(args)
    common = (a["C"], a["out_dtype"], a["M"], a["N"], a["K"], 0, 2, None, None)
    if fmt == "bf16":
        st = sk.sk_gemm_bf16_host(a["A"], a["B"], None, *common)
    elif fmt == "fp8":
        st = sk.sk_gemm_fp8_host(a["A"], a["B"], None, *common)
    else:
        st = sk.sk_gemm_mxfp4_host(a["A"], a["A_scale"], a["B"], a["B_scale"], None, *common)
    assert st == sk.SK_ERR_INVALID_ARG


def test_valid_call_without_a_gpu_is_unsupported_not_a_crash(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = sk.sk_gemm_bf16(P, P, None, P, 1, 64, 64, 64, 0, 2, None)
    assert st == sk.SK_ERR_UNSUPPORTED
    assert sk.sk_gemm_fp8(P, P, None, P, 1, 64, 64, 64, 0, 2, None) == sk.SK_ERR_UNSUPPORTED


def test_options_validation(lib):
    st = sk.sk_gemm_bf16_ex(P, P, None, P, 1, 64, 64, 64, 0, 2,
                            {"spin_timeout_ns": -1}, None)
    assert st == sk.SK_ERR_INVALID_ARG
    assert sk.sk_workspace_reserve(0, None, 0) == sk.SK_ERR_INVALID_ARG
    st = sk.sk_gemm_bf16_ex(P, P, None, P, 1, 64, 64, 64, 0, 3, {"hybrid_sk_waves": -1}, None)
    assert st == sk.SK_ERR_INVALID_ARG


@pytest.mark.parametrize("opts", [
    {"resident_limit": -1}, {"sm_record_len": -4}, {"sm_record": P, "sm_record_len": 0},
    {"sm_record": P + 2, "sm_record_len": 64},
])
def test_bad_resident_limit_and_sm_record_are_rejected_before_cuda(lib, opts):
    for fn in (sk.sk_gemm_bf16_ex, sk.sk_gemm_fp8_ex):
        assert fn(P, P, None, P, 1, 64, 64, 64, 0, 2, opts, None) == sk.SK_ERR_INVALID_ARG
    st = sk.sk_gemm_mxfp4_ex(P, P, P, P, None, P, 1, 64, 64, 64, 0, 2, opts, None)
    assert st == sk.SK_ERR_INVALID_ARG


def test_options_struct_matches_the_c_layout(tmp_path):
    """sk_options_t as the binding lays it out (size and field offsets) is the C struct."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    fields = [f[0] for f in sk.Options._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "sk_gemm.h"\n'
                   "int main(void) {\n"
                   '  printf("%zu\\n", sizeof(sk_options_t));\n'
                   + "".join(f'  printf("%zu\\n", offsetof(sk_options_t, {f}));\n' for f in fields)
                   + "  return 0;\n}\n")
    exe = str(tmp_path / "layout")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", exe], check=True)
    got = [int(x) for x in subprocess.run([exe], capture_output=True, text=True,
                                          check=True).stdout.split()]
    want = [ctypes.sizeof(sk.Options)] + [getattr(sk.Options, f).offset for f in fields]
    assert got == want


def test_workspace_bytes_is_host_bookkeeping(lib):
    assert sk.sk_workspace_bytes(-1, None) == -1
    assert sk.sk_workspace_bytes(0, 0x1234) == 0   # a stream with no workspace


def test_workspace_release_without_a_gpu_is_unsupported_not_a_crash(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert sk.sk_workspace_release(0, None) == sk.SK_ERR_UNSUPPORTED


# ---- planning -----------------------------------------------------------------------------

def test_plan_fields_follow_the_schedule_rules(lib):
    # grid capped at the SM count (a request of 133 on a 132-SM part launches 132)
    p = sk.sk_plan(0, 4096, 4096, 4096, 133, "persistent", 132, {"tile_n": 128})
    assert p.grid == 132 and p.tiles == 1024 and p.iters == 64
    p = sk.sk_plan(0, 4096, 4096, 4096, 0, "dp", 148, {"tile_n": 128})
    assert p.grid == 1024
    p = sk.sk_plan(0, 256, 256, 512, 3, "streamk", 148)
    assert (p.tile_n, p.tiles, p.iters, p.grid) == (128, 4, 8, 3)
    assert (p.sk_base, p.sk_extra, p.whole_tiles) == (10, 2, 0)
    p = sk.sk_plan(0, 1920, 1920, 16384, 0, "hybrid", 148, {"tile_m": 128})
    assert p.tiles == 225 and p.sk_tiles == 225 % 148 and p.whole_tiles == 148
    p = sk.sk_plan(1, 8192, 8192, 8192, 0, "streamk", 148, {"tile_m": 128})
    assert (p.tile_n, p.tile_k, p.iters) == (128, 256, 32)
    # fp8: 128-deep k blocks (128 bytes of E4M3 per row per block)
    p = sk.sk_plan(2, 8192, 8192, 8192, 0, "streamk", 148, {"tile_m": 128})
    assert (p.tile_n, p.tile_k, p.iters) == (256, 128, 64)      # wide 1-CTA tiles fill 148 SMs
    p = sk.sk_plan(2, 8192, 8192, 8192, 0, "streamk", 152)
    assert (p.tile_m, p.tile_n, p.tile_k, p.ctas_per_tile, p.grid) == (256, 256, 128, 2, 76)
    with pytest.raises(sk.SkError):
        sk.sk_plan(0, 0, 8, 8, 0, "dp", 148)


def test_auto_mode_picks_a_concrete_plan_from_the_cost_model():
    # choices of the fitted GB300 cost model on shapes of its calibration set (152 SMs)
    cases = {(8192, 8192, 8192): (2, 2), (64, 14336, 4096): (1, 1), (512, 512, 32768): (2, 2),
             (1536, 1536, 1536): (1, 1), (16384, 2048, 2048): (2, 1), (2304, 2304, 8192): (2, 2)}
    for (M, N, K), (ctas_per_tile, mode) in cases.items():
        p = sk.sk_plan(0, M, N, K, 0, "auto", 152)
        assert (p.ctas_per_tile, p.mode) == (ctas_per_tile, mode), (M, N, K)
        assert p.mode in (1, 2, 3)
        rows = sk.sk_plan_segments(p)          # a concrete plan: its segments cover every tile
        assert rows[:, 3].sum() - rows[:, 2].sum() == p.tiles * p.iters
    # one row of tiles streams B through narrow tiles, unless a tile is forced: 128 or 96
    # columns (96 where they put more SMs on B in one wave)
    for (M, N, K) in [(96, 8192, 8192), (64, 14336, 4096), (128, 4096, 11008), (1, 4096, 4096)]:
        p = sk.sk_plan(0, M, N, K, 0, "auto", 152)
        assert p.tile_m == 128 and p.tile_n in (96, 128), (M, N, K)
    p = sk.sk_plan(0, 64, 14336, 4096, 0, "auto", 152)
    assert (p.tile_n, p.mode, p.grid) == (96, 1, 150)
    p = sk.sk_plan(0, 96, 8192, 8192, 0, "auto", 152, {"tile_n": 256})
    assert (p.tile_m, p.tile_n) == (128, 256)
    p = sk.sk_plan(2, 96, 8192, 8192, 0, "auto", 152)        # fp8 follows the same rule
    assert (p.tile_m, p.tile_n) == (128, 128)
    # tiles the options force stay forced; MXFP4 never gets a 128x256 tile
    p = sk.sk_plan(0, 8192, 8192, 8192, 0, "auto", 152, {"tile_m": 128, "tile_n": 128})
    assert (p.tile_m, p.tile_n) == (128, 128)
    for M in (256, 2048, 8192):
        p = sk.sk_plan(1, M, 4096, 4096, 0, "auto", 152)
        assert (p.ctas_per_tile, p.tile_n) in ((2, 256), (1, 128))
    # one SM: no pairs, and still a plan
    p = sk.sk_plan(0, 4096, 4096, 4096, 1, "auto", 152)
    assert p.ctas_per_tile == 1 and p.grid == 1


def test_96_wide_tiles_where_they_put_more_sms_on_one_row_of_tiles():
    # 64 x 14336: 150 tiles of 96 in one wave instead of 112 of 128 on all SMs; not where they
    # add a wave (1, 16, 32, 64 or 128 SMs)
    for ns, want in [(0, 96), (151, 96), (150, 96), (149, 128), (32, 128), (16, 128), (64, 128),
                     (128, 128), (1, 128)]:
        for mode in ("persistent", "dp"):
            p = sk.sk_plan(0, 64, 14336, 4096, ns, mode, 152)
            assert p.tile_n == (want if mode == "persistent" or ns == 0 else p.tile_n), (ns, mode)
    assert sk.sk_plan(0, 64, 14336, 4096, 0, "dp", 152).tile_n == 96
    # Stream-K and hybrid, more than one row of tiles, fp8 and MXFP4 keep 128-wide tiles
    assert sk.sk_plan(0, 64, 14336, 4096, 0, "streamk", 152).tile_n == 128
    assert sk.sk_plan(0, 256, 14336, 4096, 0, "persistent", 152, {"tile_m": 128}).tile_n == 128
    assert sk.sk_plan(2, 64, 14336, 4096, 0, "persistent", 152).tile_n == 128
    assert sk.sk_plan(1, 64, 14336, 4096, 0, "persistent", 152).tile_n == 128
    # forced, and refused where the kernel does not exist
    p = sk.sk_plan(0, 1000, 1000, 64, 0, "streamk", 152, {"tile_n": 96})
    assert (p.tile_m, p.tile_n, p.tiles_n) == (128, 96, 11)
    for fmt, opts in [(1, {"tile_n": 96}), (2, {"tile_n": 96}), (0, {"tile_m": 256, "tile_n": 96})]:
        with pytest.raises(sk.SkError):
            sk.sk_plan(fmt, 1024, 1024, 1024, 0, "persistent", 152, opts)


def test_tall_stages_for_at_most_64_rows_of_a():
    # bf16, one CTA per 96- or 128-wide tile, plain layout, M <= 64: 128 K per stage
    for M in (1, 8, 63, 64):
        for mode, tn in (("persistent", 96), ("streamk", 128), ("dp", 96), ("hybrid", 128)):
            p = sk.sk_plan(0, M, 14336, 4096, 0, mode, 152)
            assert (p.tile_m, p.tile_n, p.tile_k, p.iters) == (128, tn, 128, 32), (M, mode)
    p = sk.sk_plan(0, 64, 14336, 4104, 0, "streamk", 152)
    assert (p.tile_k, p.iters) == (128, 33)                         # a ragged last stage
    # more rows of A, 256-wide tiles, pairs, other formats: the usual stages
    assert sk.sk_plan(0, 65, 14336, 4096, 0, "persistent", 152).tile_k == 64
    assert sk.sk_plan(0, 64, 14336, 4096, 0, "persistent", 152, {"tile_n": 256}).tile_k == 64
    assert sk.sk_plan(2, 64, 14336, 4096, 0, "persistent", 152).tile_k == 128   # fp8's own
    assert sk.sk_plan(1, 64, 14336, 4096, 0, "persistent", 152).tile_k == 256
    # forced either way where it exists, refused where it does not
    p = sk.sk_plan(0, 64, 14336, 4096, 0, "persistent", 152, {"tile_k": 64})
    assert (p.tile_k, p.iters) == (64, 64)
    assert sk.sk_plan(0, 32, 4096, 4096, 0, "persistent", 152, {"tile_k": 128}).tile_k == 128
    for fmt, M, opts in [(0, 65, {"tile_k": 128}), (0, 64, {"tile_k": 128, "tile_n": 256}),
                         (0, 64, {"tile_k": 256}), (2, 64, {"tile_k": 64}),
                         (1, 64, {"tile_k": 128}), (0, 64, {"tile_k": 96})]:
        with pytest.raises(sk.SkError):
            sk.sk_plan(fmt, M, 14336, 4096, 0, "persistent", 152, opts)


def test_pair_plans():
    # large problems go to SM pairs: 256 x 256 tiles, grid counted in pairs
    p = sk.sk_plan(0, 8192, 8192, 8192, 0, "streamk", 152)
    assert (p.tile_m, p.tile_n, p.ctas_per_tile, p.grid, p.tiles) == (256, 256, 2, 76, 1024)
    p = sk.sk_plan(1, 8192, 8192, 8192, 0, "persistent", 152)
    assert (p.tile_m, p.tile_n, p.tile_k, p.iters, p.grid) == (256, 256, 256, 32, 76)
    # num_sms counts SMs: an odd request leaves one SM unused
    p = sk.sk_plan(0, 4096, 4096, 4096, 33, "persistent", 152)
    assert p.ctas_per_tile == 2 and p.grid == 16
    p = sk.sk_plan(0, 4096, 4096, 4096, 0, "dp", 152)
    assert p.grid == 256 and p.ctas_per_tile == 2
    # too few SMs, rows or tiles for a pair: one CTA per tile
    assert sk.sk_plan(0, 4096, 4096, 4096, 1, "persistent", 152).ctas_per_tile == 1
    assert sk.sk_plan(0, 4096, 4096, 4096, 3, "streamk", 152).ctas_per_tile == 1
    assert sk.sk_plan(0, 64, 14336, 4096, 0, "streamk", 152).ctas_per_tile == 1
    assert sk.sk_plan(0, 256, 256, 512, 0, "streamk", 152).ctas_per_tile == 1
    # forced choices
    assert sk.sk_plan(0, 256, 256, 512, 0, "dp", 152, {"tile_m": 256}).ctas_per_tile == 2
    assert sk.sk_plan(0, 8192, 8192, 8192, 0, "dp", 152, {"tile_n": 128}).ctas_per_tile == 1
    for bad in [{"tile_m": 256, "tile_n": 128}, {"tile_m": 64}]:
        with pytest.raises(sk.SkError):
            sk.sk_plan(0, 1024, 1024, 1024, 0, "dp", 152, bad)
    with pytest.raises(sk.SkError):
        sk.sk_plan(0, 1024, 1024, 1024, 1, "dp", 152, {"tile_m": 256})


@pytest.mark.parametrize("mode", ["dp", "persistent", "streamk", "hybrid"])
@pytest.mark.parametrize("shape", [(8192, 8192, 8192), (1920, 1920, 16384), (300, 264, 200),
                                   (1000, 3000, 640)])
@pytest.mark.parametrize("g", [2, 7, 33, 0])
def test_pair_scheduler_matches_oracle_restatement(mode, shape, g):
    M, N, K = shape
    plan = sk.sk_plan(0, M, N, K, g, mode, 152, {"tile_m": 256})
    assert plan.ctas_per_tile == 2
    got = sk.sk_plan_segments(plan)
    want = oracle.schedule(sk.MODES[mode], plan.tiles, plan.iters, plan.grid)
    assert np.array_equal(got[:, :5], want)


@pytest.mark.parametrize("shape", [(2304, 2304, 8192), (8192, 8192, 8192), (1000, 3000, 640)])
@pytest.mark.parametrize("g", [7, 33, 0])
@pytest.mark.parametrize("tile_m,waves", [(256, 1), (128, 1), (128, 2)])
def test_two_tile_hybrid_matches_oracle_restatement(shape, g, tile_m, waves):
    M, N, K = shape
    plan = sk.sk_plan(0, M, N, K, g, "hybrid", 152, {"tile_m": tile_m, "hybrid_sk_waves": waves})
    got = sk.sk_plan_segments(plan)
    want = oracle.schedule(sk.MODES["hybrid"], plan.tiles, plan.iters, plan.grid, waves)
    assert np.array_equal(got[:, :5], want)
    assert plan.sk_tiles == min(plan.tiles, plan.tiles % plan.grid + waves * plan.grid)


def _same_split(mode, M, N, K, g_req, sms, tile_n):
    plan = sk.sk_plan(0, M, N, K, g_req, mode, sms, {"tile_n": tile_n})
    got = sk.sk_plan_segments(plan)
    want = oracle.schedule(sk.MODES[mode], plan.tiles, plan.iters, plan.grid)
    assert np.array_equal(got[:, :5], want), (mode, M, N, K, g_req, sms)
    return plan, got


@pytest.mark.parametrize("mode", ["dp", "persistent", "streamk", "hybrid"])
@pytest.mark.parametrize("shape", [(256, 256, 512), (1920, 1920, 16384), (64, 14336, 4096),
                                   (200, 136, 200), (128, 128, 64), (4096, 4096, 4096)])
@pytest.mark.parametrize("g", [1, 3, 7, 16, 132, 0])
def test_kernel_scheduler_matches_oracle_restatement(lib, mode, shape, g):
    M, N, K = shape
    _same_split(mode, M, N, K, g, 148, 128)


@pytest.mark.parametrize("mode", ["dp", "persistent", "streamk", "hybrid"])
@pytest.mark.parametrize("M,N,K,group,g", [(8192, 8192, 8192, 16, 152), (1920, 1920, 16384, 16, 152),
                                           (1000, 3000, 640, 5, 37), (128, 256, 64, 1, 3),
                                           (640, 128, 4096, 3, 7), (256, 256, 512, 16, 3),
                                           (2048, 512, 128, 4, 148)])
@pytest.mark.parametrize("tile_m", [128, 256])
def test_raster_is_a_bijection_onto_the_tile_grid(lib, mode, M, N, K, group, g, tile_m):
    if tile_m == 256 and g < 2:
        pytest.skip("pairs need two SMs")
    opts = {"raster_group": group, "tile_m": tile_m}
    if tile_m == 128:
        opts["tile_n"] = 128
    plan = sk.sk_plan(0, M, N, K, g, mode, 152, opts)
    segs = sk.sk_plan_segments(plan)
    owned = segs[segs[:, 2] == 0]          # the piece holding k = 0 of each tile
    cells = list(map(tuple, owned[:, 5:7].tolist()))
    assert len(cells) == plan.tiles == len(set(cells))
    assert set(cells) == {(i, j) for i in range(plan.tiles_m) for j in range(plan.tiles_n)}
    # every piece of a tile maps to the same cell
    cell_of = {int(t): (int(a), int(b)) for t, a, b in owned[:, [1, 5, 6]].tolist()}
    for t, a, b in segs[:, [1, 5, 6]].tolist():
        assert cell_of[t] == (a, b)


def _raster_pos(plan, tm, tn):
    group = tm // plan.raster_group
    first = group * plan.raster_group
    rows = min(plan.tiles_m - first, plan.raster_group)
    return first * plan.tiles_n + tn * rows + (tm - first)


@pytest.mark.parametrize("M,N,K,g", [(8192, 8192, 8192, 152), (4096, 4096, 4096, 152),
                                     (1920, 1920, 16384, 152), (3000, 2000, 1000, 37)])
def test_streamk_tiles_worked_on_together_form_one_raster_block(lib, M, N, K, g):
    plan = sk.sk_plan(0, M, N, K, g, "streamk", 152, {"tile_n": 128})
    segs = sk.sk_plan_segments(plan)
    f = plan.sk_base // plan.iters
    for cta in range(plan.grid):
        mine = segs[(segs[:, 0] == cta) & (segs[:, 2] == 0)]
        for tau, row in enumerate(mine.tolist()):
            pos = _raster_pos(plan, row[5], row[6]) - plan.whole_tiles
            if tau < f:
                assert pos == tau * plan.grid + cta
            else:
                assert f * plan.grid <= pos < plan.tiles - plan.whole_tiles


def test_streamk_256_cube_split_matches_golden(lib):
    want = np.loadtxt(os.path.join(ROOT, "tests", "golden", "streamk_256x256x512_g3.txt"),
                      dtype=np.int64)
    plan = sk.sk_plan(0, 256, 256, 512, 3, "streamk", 148)
    got = sk.sk_plan_segments(plan)
    assert np.array_equal(got[:, :5], want)


def test_streamk_regions_of_2_31_iterations_are_refused():
    # the kernels' schedule arithmetic runs in 32 bits: a Stream-K region of 2^31 or more tile
    # k-iterations is refused; persistent plans of the same problem and the automatic choice
    # (which skips refused candidates) stay available
    big, tiles = (131072, 131072, 131072), {"tile_m": 128, "tile_n": 128}
    for mode in ("streamk", "hybrid"):
        with pytest.raises(sk.SkError) as e:
            sk.sk_plan(0, *big, 0, mode, 152, dict(tiles, hybrid_sk_waves=10 ** 6))
        assert e.value.status == sk.SK_ERR_UNSUPPORTED
    p = sk.sk_plan(0, *big, 0, "persistent", 152, tiles)
    assert p.tiles == 1024 * 1024
    p = sk.sk_plan(0, *big, 0, "auto", 152)
    assert p.sk_tiles * p.iters < 2 ** 31
    p = sk.sk_plan(0, 65536, 65536, 512000, 0, "streamk", 152, tiles)   # just below the limit
    assert p.sk_tiles * p.iters == 262144 * 8000 < 2 ** 31 and p.mode == 2
    with pytest.raises(sk.SkError):                                       # at it: 2^18 x 2^13
        sk.sk_plan(0, 65536, 65536, 524288, 0, "streamk", 152, tiles)


def test_auto_cost_constants_are_the_fit_of_the_shipped_sweep():
    pytest.importorskip("scipy")
    from sm_constrained_persistent_gb300 import tuning
    coef, quality = tuning.fit(tuning.load())
    src = open(os.path.join(ROOT, "sm_constrained_persistent_gb300", "csrc", "sk_api.cu")).read()
    m = re.search(r"kCost = \{\{([^}]*)\}, ([^;]*)\};", src)
    iters = [float(v) for v in m.group(1).split(",")]
    rest = [float(v) for v in m.group(2).rstrip("}").split(",")]
    assert iters == [coef["t_iter_pair"], coef["t_iter_128x256"], coef["t_iter_128x128"]]
    assert rest == [coef["t_piece"], coef["t_split"], coef["t_part"], coef["t_launch"],
                    coef["t_split_shared"], coef["t_part_shared"]]
    assert quality["mean_loss"] < 0.02 and quality["max_loss"] < 0.15


def test_auto_choice_is_the_cheapest_candidate_of_the_documented_estimate():
    # tuning.plan_cost restates the estimate; the library's automatic plan must be its first
    # cheapest candidate (tiles 256x256, 128x256, 128x128, 128x96 in that order, each under
    # persistent, Stream-K and hybrid, with the planner's rules for one row of tiles)
    pytest.importorskip("scipy")
    from sm_constrained_persistent_gb300 import tuning
    coef, _ = tuning.fit(tuning.load())
    tiles = [(256, 256), (128, 256), (128, 128), (128, 96)]
    shapes = [(8192, 8192, 8192), (1920, 1920, 16384), (512, 512, 16384), (64, 14336, 4096),
              (96, 8192, 8192), (3000, 1000, 7000), (256, 4096, 4096), (1024, 2048, 8192),
              (4096, 4096, 1024), (640, 2560, 16384), (1, 4096, 4096), (7168, 7168, 1536)]
    for fmt in (0, 1, 2):
        for (M, N, K) in shapes:
            if fmt == 1 and (K % 32 or N % 2):
                continue
            best = None
            for tm, tn in tiles:
                if M <= 128 and (tm, tn) in ((128, 256), (256, 256)):
                    continue
                if tn == 96 and (fmt != 0 or M > 128):
                    continue
                for mode in ("persistent", "streamk", "hybrid"):
                    try:
                        p = sk.sk_plan(fmt, M, N, K, 0, mode, 152, {"tile_m": tm, "tile_n": tn})
                    except sk.SkError:
                        continue
                    c = tuning.plan_cost(p, coef, fmt)
                    if best is None or c < best[0]:
                        best = (c, p)
            auto = sk.sk_plan(fmt, M, N, K, 0, "auto", 152)
            want = best[1]
            assert (auto.mode, auto.tile_m, auto.tile_n, auto.grid) == \
                (want.mode, want.tile_m, want.tile_n, want.grid), (fmt, M, N, K)


def test_tensor_pipe_probes_compile_for_sm103a():
    """The measurement programs behind the kernels' MMA-kind and scale-copy choices build."""
    import shutil
    if shutil.which("nvcc") is None:
        pytest.skip("no nvcc")
    from sm_constrained_persistent_gb300 import probes
    for name in probes.PROBES:
        assert os.path.exists(probes.build(name))
