"""The range bookkeeping behind the SM-pair kernels' shared fix-up, on the CPU.

tests/share_check.cu runs sk_range_cta and tile_contributors (sk_schedule.cuh, the code the
kernels run) on plans from the library's planner; every answer is compared with the schedule's
own list of pieces (sk_plan_segments, from the kernels' Cursor):
  - a split tile's owner is the unit holding its first k-iteration (its role-1 piece);
  - its contributors are the units with a role-2 piece of it;
  - a contributor is a finisher exactly when that piece is its only piece in the Stream-K
    region (its whole range lies inside the tile).
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

import sm_constrained_persistent_gb300 as sk
from sm_constrained_persistent_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = [  # (M, N, K, num_sms, mode)
    (1920, 1920, 16384, 0, "streamk"),
    (1024, 1024, 16384, 0, "streamk"),
    (512, 512, 16384, 0, "streamk"),
    (256, 256, 16384, 0, "streamk"),      # one tile, every pair on it
    (300, 264, 8200, 16, "streamk"),
    (300, 264, 8200, 64, "streamk"),
    (520, 776, 4096, 0, "streamk"),
    (8192, 8192, 8192, 0, "streamk"),     # every range spans many tiles: no finishers
    (4096, 4096, 4096, 0, "streamk"),
    (4096, 4096, 4096, 0, "hybrid"),
    (1920, 1920, 16384, 0, "hybrid"),
    (2048, 256, 4096, 6, "streamk"),
    (1040, 776, 1000, 0, "streamk"),
]


@pytest.fixture(scope="module")
def share_check(tmp_path_factory):
    nvcc = shutil.which(os.environ.get("NVCC", "nvcc"))
    if nvcc is None:
        pytest.skip("no nvcc")
    exe = str(tmp_path_factory.mktemp("share") / "share_check")
    subprocess.run([nvcc, *_build.ARCH, "-std=c++17", "-I", _build.CSRC,
                    os.path.join(ROOT, "tests", "share_check.cu"), "-o", exe], check=True)
    return exe


def _plans():
    out = []
    for M, N, K, num_sms, mode in CASES:
        plan = sk.sk_plan(0, M, N, K, num_sms, mode, 152, {"tile_m": 256})
        assert plan.ctas_per_tile == 2
        out.append(((M, N, K, num_sms, mode), plan))
    return out


def test_range_owner_and_contributors_match_the_schedule(share_check):
    plans = _plans()
    stdin = "".join(f"{p.tiles_m} {p.tiles_n} {p.iters} {p.grid} {p.whole_tiles} {p.sk_base} "
                    f"{p.sk_extra}\n" for _, p in plans)
    res = subprocess.run([share_check], input=stdin, capture_output=True, text=True, check=True)
    blocks = res.stdout.split("end\n")
    assert len(blocks) == len(plans) + 1 and blocks[-1] == ""
    seen_finishers = set()
    for (case, plan), block in zip(plans, blocks):
        segs = sk.sk_plan_segments(plan)
        region = segs[segs[:, 1] >= plan.whole_tiles]
        pieces = np.bincount(region[:, 0], minlength=plan.grid)
        got = {}
        for line in block.splitlines():
            t, owner, n_contrib, finishers = map(int, line.split())
            got[t + plan.whole_tiles] = (owner, n_contrib, finishers)
        split = sorted(int(t) for t in np.unique(segs[segs[:, 4] == 1, 1]))
        assert sorted(got) == split, case
        for tile in split:
            owner = int(segs[(segs[:, 1] == tile) & (segs[:, 4] == 1), 0][0])
            contrib = segs[(segs[:, 1] == tile) & (segs[:, 4] == 2), 0]
            finishers = int((pieces[contrib] == 1).sum())
            assert got[tile] == (owner, len(contrib), finishers), (case, tile)
            seen_finishers.add(finishers)
    # the cases reach tiles with no, one, two and many finishers
    assert {0, 1, 2}.issubset(seen_finishers) and max(seen_finishers) >= 20
