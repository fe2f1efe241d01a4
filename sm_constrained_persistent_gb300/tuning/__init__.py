"""Calibration of the automatic schedule and tile choice (SK_MODE_AUTO).

`sweep()` times a list of bf16 shapes under every schedule and tile kind on the current GPU;
`fit()` fits the cost model's constants (the `kCost` table in csrc/sk_api.cu) to such timings
by non-negative least squares on the relative error, and reports how close the cheapest
estimate comes to the fastest configuration.  `gb300_bf16_sweep.json` holds the timings the
shipped constants were fitted to.
"""
from __future__ import annotations

import json
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# 64-K stages throughout: the shipped timings predate the tall (128-K) stages that problems of
# at most 64 rows now get, and the fit prices those through its own scale.
TILES = {"pair": {"tile_m": 256, "tile_k": 64}, "128x256": {"tile_m": 128, "tile_n": 256, "tile_k": 64},
         "128x128": {"tile_m": 128, "tile_n": 128, "tile_k": 64}}
MODES = ["dp", "persistent", "streamk", "hybrid"]


def load(path=os.path.join(HERE, "gb300_bf16_sweep.json")):
    with open(path) as f:
        return json.load(f)["times"]


def sweep(shapes, steps=10, warmup=3, seed=99):
    """{"MxNxK": {tile: {mode: ms}}} for bf16 N(0,1)/sqrt(K) operands on the current device."""
    import numpy as np
    import torch
    import sm_constrained_persistent_gb300 as sk
    from sm_constrained_persistent_gb300 import inputs
    flush_w = torch.empty(64 << 20, dtype=torch.float32, device="cuda")
    flush_r = torch.ones((64 << 10, 1024), dtype=torch.float32, device="cuda")
    flush_o = torch.empty(1024, dtype=torch.float32, device="cuda")
    out = {}
    for (M, N, K) in shapes:
        p = inputs.bf16_problem(M, N, K, seed=seed, operand_scale="sqrt_k")
        a = torch.from_numpy(p["A"].view(np.int16)).view(torch.bfloat16).cuda()
        b = torch.from_numpy(p["B"].view(np.int16)).view(torch.bfloat16).cuda()
        c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        res = {}
        for tname, opt in TILES.items():
            if tname == "pair" and M <= 128:
                continue
            res[tname] = {}
            for mode in MODES:
                for _ in range(warmup):
                    sk.gemm_bf16(a, b, out=c, mode=mode, options=opt)
                total = 0.0
                for _ in range(steps):
                    flush_w.fill_(1.0)
                    torch.amax(flush_r, dim=0, out=flush_o)
                    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    s.record()
                    sk.gemm_bf16(a, b, out=c, mode=mode, options=opt)
                    e.record()
                    torch.cuda.synchronize()
                    total += s.elapsed_time(e)
                sk.stream_status()
                res[tname][mode] = total / steps
        out[f"{M}x{N}x{K}"] = res
    return out


def _features(M, N, K, tile, mode, sm_count):
    import sm_constrained_persistent_gb300 as sk
    p = sk.sk_plan(0, M, N, K, 0, mode, sm_count, TILES[tile])
    g, T, I = p.grid, p.tiles, p.iters
    kind = ["pair", "128x256", "128x128"].index(tile)
    x = [0.0] * 10
    if mode in ("dp", "persistent"):
        workers = min(g, sm_count // p.ctas_per_tile)
        waves = math.ceil(T / workers)
        x[kind], x[3] = waves * I, waves
        x[7] = waves if mode == "dp" else 0
    else:
        skT, whole = p.sk_tiles, p.whole_tiles
        per = math.ceil(skT * I / g) if skT else 0
        x[kind] = per + math.ceil(whole / g) * I
        x[3] = math.ceil(whole / g) + (math.ceil(per / I) + 1 if skT else 0)
        split = 1.0 if skT and (per % I != 0 or (skT * I) % g != 0) else 0.0
        sharers = math.ceil(I / per) if skT else 0
        # SM pairs (bf16, fp8) finish a split tile together with the contributors that hold
        # nothing else, where the tile has at least two of them: a fix-up of its own price
        if shared_finish(p):
            x[8], x[9] = split, sharers
        else:
            x[4], x[5] = split, sharers
    x[6] = 1.0
    return x


def shared_finish(p, format=0):
    """Whether a plan's split tiles are mostly finished by their owners and the contributors
    that hold nothing else (the SM-pair kernels, bf16 and fp8): a Stream-K region covering the
    whole grid's work, ranges at most a third of a tile."""
    if p.ctas_per_tile != 2 or format == 1 or p.sk_tiles == 0 or p.whole_tiles != 0:
        return False
    per = math.ceil(p.sk_tiles * p.iters / max(p.grid, 1))
    return math.ceil(p.iters / per) >= 3


def fit(times, sm_count=152):
    """Constants (us): per-k-iteration time of a pair / 128x256 / 128x128 tile, per piece,
    per split region, per CTA sharing a split tile, launch, the data-parallel per-wave cost
    (which only keeps data-parallel rows from biasing the others), and the split-region and
    per-sharing-CTA costs where SM pairs share the finish of their split tiles.  Also returns the mean and
    the largest loss of picking the cheapest estimate among persistent / Stream-K / hybrid."""
    import numpy as np
    from scipy.optimize import nnls
    rows = []
    for shape, res in times.items():
        M, N, K = map(int, shape.split("x"))
        for tile, modes in res.items():
            for mode, ms in modes.items():
                rows.append((shape, tile, mode, ms * 1000.0, _features(M, N, K, tile, mode, sm_count)))
    X = np.array([r[4] for r in rows])
    y = np.array([r[3] for r in rows])
    coef, _ = nnls(X / y[:, None], np.ones_like(y))
    pred = X @ coef
    losses = []
    for shape in times:
        rs = [(r, p) for r, p in zip(rows, pred) if r[0] == shape]
        best = min(r[3] for r, _ in rs)
        M = int(shape.split("x")[0])
        # the planner's candidates: no data-parallel, and no 128x256 tile for one row of tiles
        pick = min(((r, p) for r, p in rs if r[2] != "dp" and not (M <= 128 and r[1] == "128x256")),
                   key=lambda t: t[1])[0]
        losses.append(pick[3] / best - 1.0)
    names = ["t_iter_pair", "t_iter_128x256", "t_iter_128x128", "t_piece", "t_split", "t_part",
             "t_launch", "t_dp_wave", "t_split_shared", "t_part_shared"]
    return dict(zip(names, (round(float(c), 4) for c in coef))), \
        {"mean_loss": float(np.mean(losses)), "max_loss": float(np.max(losses))}


# The per-iteration scales of the estimate that are not fitted: MXFP4 and 96-wide k-iterations
# against bf16 ones, and a tall (128-K) stage against two 64-K ones.
MX_ITER_SCALE = 1.45
N96_ITER_SCALE = 0.94
TALL_ITER_SCALE = 0.97


def plan_cost(p, coef, format=0):
    """The automatic choice's estimate (us) of a plan `p` (an sk_plan_t) under the fitted
    constants `coef` (fit()'s first result): the cost the library minimises over its candidates."""
    kind = 0 if p.ctas_per_tile == 2 else (1 if p.tile_n == 256 else 2)
    t_iter = [coef["t_iter_pair"], coef["t_iter_128x256"], coef["t_iter_128x128"]][kind]
    t_iter *= MX_ITER_SCALE if format == 1 else 1.0
    t_iter *= N96_ITER_SCALE if p.tile_n == 96 else 1.0
    t_iter *= 2.0 * TALL_ITER_SCALE if format == 0 and p.tile_k == 128 else 1.0
    g, T, I = max(p.grid, 1), p.tiles, p.iters
    fixup = 0.0
    if p.mode in (0, 1):
        waves = math.ceil(T / g)
        iters, pieces = waves * I, waves
    else:
        skT, whole = p.sk_tiles, p.whole_tiles
        per = math.ceil(skT * I / g) if skT else 0
        iters = per + math.ceil(whole / g) * I
        pieces = math.ceil(whole / g) + (math.ceil(per / I) + 1 if skT else 0)
        if skT:
            split = per % I != 0 or (skT * I) % g != 0
            shared = shared_finish(p, format)
            fixup = ((coef["t_split_shared"] if shared else coef["t_split"]) if split else 0.0) + \
                (coef["t_part_shared"] if shared else coef["t_part"]) * math.ceil(I / max(per, 1))
    return coef["t_launch"] + iters * t_iter + pieces * coef["t_piece"] + fixup
