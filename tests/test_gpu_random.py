"""Seeded random sweep over shapes, schedules, tile kinds, num_sms and formats: every case
bit-exact against the CPU oracle on exact-integer inputs (so any schedule or tile must give
exactly the same result)."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
import sm_constrained_persistent_gb300 as sk
from sm_constrained_persistent_gb300 import inputs

pytestmark = pytest.mark.gpu
MODES = ["dp", "persistent", "streamk", "hybrid", "auto"]
TILES = [None, {"tile_m": 128, "tile_n": 128}, {"tile_m": 128, "tile_n": 256}, {"tile_m": 256}]


def _cases(n, seed):
    rng = np.random.default_rng(seed)
    for i in range(n):
        fmt = ["bf16", "fp8", "mxfp4"][i % 3]
        align = {"bf16": 8, "fp8": 16, "mxfp4": 32}[fmt]
        M = int(rng.integers(1, 700))
        N = int(rng.integers(1, 90)) * 8 if fmt != "fp8" else int(rng.integers(1, 45)) * 16
        K = int(rng.integers(1, 40)) * align
        mode = MODES[int(rng.integers(0, len(MODES)))]
        tile = TILES[int(rng.integers(0, len(TILES)))]
        if fmt == "mxfp4" and tile == TILES[2]:
            tile = TILES[1]                       # MXFP4 has no 128x256 tile
        num_sms = int(rng.choice([0, 1, 2, 5, 13, 64, 151]))
        if tile is not None and tile.get("tile_m") == 256 and num_sms in (1,):
            num_sms = 2                           # a pair needs two SMs
        out = "f32" if rng.random() < 0.5 else "bf16"
        yield pytest.param(fmt, M, N, K, mode, tile, num_sms, out, int(rng.integers(1 << 30)),
                           id=f"{i}-{fmt}-{M}x{N}x{K}-{mode}-{num_sms}")


@pytest.mark.parametrize("fmt,M,N,K,mode,tile,num_sms,out,seed", list(_cases(72, 2024)))
def test_random_case_is_bit_exact(fmt, M, N, K, mode, tile, num_sms, out, seed):
    odt = torch.float32 if out == "f32" else torch.bfloat16
    if fmt == "bf16":
        p = inputs.bf16_problem(M, N, K, seed=seed, integer=True,
                                bias="f32_int" if out == "f32" else "none")
        c = gu.run_bf16(p, out=out, mode=mode, num_sms=num_sms, options=tile)
        ref = oracle.addmm_bf16(p["A"], p["B"], p["bias"])
    elif fmt == "fp8":
        p = inputs.fp8_problem(M, N, K, seed=seed, integer=True,
                               bias="f32_int" if out == "f32" else "none")
        c = sk.gemm_fp8(gu.dev_u8(p["A"]), gu.dev_u8(p["B"]), gu.dev_bias(p["bias"]),
                        out_dtype=odt, mode=mode, num_sms=num_sms, options=tile)
        sk.stream_status()
        ref = oracle.addmm_fp8(p["A"], p["B"], p["bias"])
    else:
        p = inputs.mxfp4_problem(M, N, K, seed=seed, exp_range=1,
                                 bias="f32_normal" if out == "f32" else "none")
        c = gu.run_mxfp4(p, out=out, mode=mode, num_sms=num_sms, options=tile)
        ref = oracle.addmm_mxfp4(p["A"], p["A_scale"], p["B"], p["B_scale"], p["bias"])
    want = oracle.round_output(ref, oracle.BF16 if out == "bf16" else oracle.F32)
    got = gu.host_bits(c)
    assert np.array_equal(got, want if out == "bf16" else want.view(np.uint32))
