"""Pins for the CPU oracle: each check ties it to something other than itself.

* output rounding: nearest-neighbour search over the enumerated bf16 values (a different
  algorithm from the oracle's scale-and-round), and numpy's float64->float32 conversion;
* GEMM: exact rational arithmetic (fractions) on tiny shapes, integer matmul (numpy int64),
  closed forms (A = 0, B = I, all ones) and torch's float64 addmm;
* MX decode: the OCP MX v1.0 E2M1 table and 2^(E-127) for E8M0;
* MXFP4 GEMM: exact rational brute force with the nibbles unpacked here, the cross-format
  identity with the bf16 GEMM of the decoded operands, and scale linearity;
* schedules: coverage, ownership and balance invariants, the hand-derived 3-CTA split, and
  schedule invariance of the result.
"""
import bisect
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from sm_constrained_persistent_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------------------
# helpers written independently of the oracle
# ---------------------------------------------------------------------------------------

def _f32_bits_to_float(bits32):
    return struct.unpack("<f", struct.pack("<I", bits32))[0]


def _bf16_to_float(bits):
    return _f32_bits_to_float((bits & 0xFFFF) << 16)


# All non-negative finite bf16 values in increasing order, plus 2^128 standing for +Inf
# (its pattern 0x7F80 has an even mantissa, so a tie at the top rounds to Inf).
_BF16_POS = [(Fraction(_bf16_to_float(b)), b) for b in range(0x0000, 0x7F80)]
_BF16_POS.append((Fraction(2) ** 128, 0x7F80))
_BF16_KEYS = [v for v, _ in _BF16_POS]


def bf16_nearest_even(x):
    """Nearest bf16 pattern to the exact rational/float x, ties to the even pattern."""
    x = Fraction(x)
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    i = bisect.bisect_left(_BF16_KEYS, a)
    if i < len(_BF16_KEYS) and _BF16_KEYS[i] == a:
        return sign | _BF16_POS[i][1]
    if i >= len(_BF16_KEYS):
        return sign | 0x7F80
    lo_v, lo_b = _BF16_POS[i - 1]
    hi_v, hi_b = _BF16_POS[i]
    dlo, dhi = a - lo_v, hi_v - a
    if dlo < dhi:
        pick = lo_b
    elif dhi < dlo:
        pick = hi_b
    else:
        pick = lo_b if lo_b % 2 == 0 else hi_b
    return sign | pick


def _golden_e2m1():
    table = {}
    with open(os.path.join(GOLDEN, "e2m1_ocp_mx_v1.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            code, val = line.split()
            table[int(code)] = float(val)
    return table


E2M1 = _golden_e2m1()


def _unpack_codes(codes_row_bytes, K):
    """Unpack one row of packed FP4 bytes: even k in the low nibble."""
    out = []
    for byte in codes_row_bytes:
        out.append(int(byte) & 0xF)
        out.append(int(byte) >> 4)
    assert len(out) == K
    return out


# ---------------------------------------------------------------------------------------
# rounding
# ---------------------------------------------------------------------------------------

def test_round_bf16_special_values():
    assert oracle.round_bf16(0.0) == 0x0000
    assert oracle.round_bf16(-0.0) == 0x8000
    assert oracle.round_bf16(float("inf")) == 0x7F80
    assert oracle.round_bf16(float("-inf")) == 0xFF80
    assert oracle.round_bf16(float("nan")) & 0x7F80 == 0x7F80
    assert oracle.round_bf16(float("nan")) & 0x007F != 0
    # 1 + 2^-8 is exactly halfway between 1 and 1 + 2^-7: ties to the even pattern (1.0).
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 0x3F80
    # 1 + 3*2^-8 is halfway between 1+2^-7 (odd) and 1+2^-6 (even).
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82


def test_round_bf16_matches_nearest_neighbour_search():
    rng = np.random.default_rng(7)
    samples = []
    # random magnitudes over the whole bf16 range, subnormals and beyond the top
    for e in range(-140, 130, 3):
        samples.extend(rng.uniform(1.0, 2.0, size=6) * 2.0 ** e)
    # exact halfway points between neighbours (ties), including subnormal and top ones
    for b in list(range(0x0001, 0x0100)) + list(range(0x3F00, 0x3F90)) + [0x7F7E, 0x7F7F]:
        lo, hi = Fraction(_bf16_to_float(b)), Fraction(_bf16_to_float(b + 1)) if b + 1 < 0x7F80 else Fraction(2) ** 128
        samples.append(float((lo + hi) / 2))
        samples.append(float(lo + (hi - lo) / 4))
    samples += [float.fromhex("0x1.fefffffffffffp+127"), float.fromhex("0x1.ff00000000000p+127"),
                float.fromhex("0x1.ff00000000001p+127"), 5e-324, 2.0 ** -134, 2.0 ** -133 * 1.5]
    for s in samples:
        for x in (s, -s):
            assert oracle.round_bf16(x) == bf16_nearest_even(x), x


def test_round_output_f32_matches_numpy():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(1000) * 10.0 ** rng.integers(-40, 40, 1000),
                        [3.4028235677973366e38, 3.4028236e38, 1e-46, -0.0, 0.0]])
    got = oracle.round_output(x, oracle.F32)
    with np.errstate(over="ignore"):
        want = x.astype(np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


# ---------------------------------------------------------------------------------------
# bf16 GEMM
# ---------------------------------------------------------------------------------------

def _dyadic_bf16(rng, shape):
    """bf16 values with 8 significant bits and exponents in [-4, 4] (exact in bf16)."""
    mant = rng.integers(128, 256, size=shape) * rng.choice([-1, 1], size=shape)
    expo = rng.integers(-4, 5, size=shape)
    vals = mant.astype(np.float64) * np.exp2(expo - 7)
    return inputs.to_bf16_bits(vals.astype(np.float32))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (8, 2, 5), (2, 7, 8), (5, 3, 1)])
@pytest.mark.parametrize("bias_kind", ["none", "f32", "bf16"])
def test_bf16_bruteforce_exact_rationals(M, N, K, bias_kind):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    A = _dyadic_bf16(rng, (M, K))
    B = _dyadic_bf16(rng, (K, N))
    bias = None
    if bias_kind == "f32":
        bias = rng.standard_normal(N).astype(np.float32)
    elif bias_kind == "bf16":
        bias = _dyadic_bf16(rng, (N,))
    got64 = oracle.addmm_bf16(A, B, bias)
    got16 = oracle.round_output(got64, oracle.BF16)
    got32 = oracle.round_output(got64, oracle.F32)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(_bf16_to_float(int(A[m, k]))) * Fraction(_bf16_to_float(int(B[k, n])))
                        for k in range(K))
            if bias_kind == "f32":
                exact += Fraction(float(bias[n]))
            elif bias_kind == "bf16":
                exact += Fraction(_bf16_to_float(int(bias[n])))
            assert Fraction(got64[m, n]) == exact
            assert int(got16[m, n]) == bf16_nearest_even(exact)
            assert got32[m, n] == np.float32(float(exact))


def test_bf16_integer_inputs_match_integer_matmul():
    p = inputs.bf16_problem(70, 90, 200, seed=11, integer=True, bias="f32_int")
    Ai = inputs.bf16_bits_to_f32(p["A"]).astype(np.int64)
    Bi = inputs.bf16_bits_to_f32(p["B"]).astype(np.int64)
    want = Ai @ Bi + p["bias"].astype(np.int64)[None, :]
    got = oracle.addmm_bf16(p["A"], p["B"], p["bias"])
    assert np.array_equal(got, want.astype(np.float64))


def test_bias_only_when_a_is_zero():
    rng = np.random.default_rng(5)
    M, N, K = 6, 11, 9
    A = np.zeros((M, K), dtype=np.uint16)
    B = inputs.to_bf16_bits(rng.standard_normal((K, N)).astype(np.float32))
    bias32 = rng.standard_normal(N).astype(np.float32)
    got = oracle.addmm_bf16(A, B, bias32)
    assert np.array_equal(got, np.broadcast_to(bias32.astype(np.float64), (M, N)))
    bias16 = inputs.to_bf16_bits(rng.standard_normal(N).astype(np.float32))
    got = oracle.addmm_bf16(A, B, bias16)
    assert np.array_equal(got, np.broadcast_to(inputs.bf16_bits_to_f32(bias16).astype(np.float64), (M, N)))
    assert np.array_equal(oracle.addmm_bf16(A, B, None), np.zeros((M, N)))


def test_identity_and_all_ones_closed_forms():
    rng = np.random.default_rng(9)
    M, K = 13, 24
    A = inputs.to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    eye = inputs.to_bf16_bits(np.eye(K, dtype=np.float32))
    bias = rng.standard_normal(K).astype(np.float32)
    got = oracle.addmm_bf16(A, eye, bias)
    want = inputs.bf16_bits_to_f32(A).astype(np.float64) + bias.astype(np.float64)[None, :]
    assert np.array_equal(got, want)
    M, N, K = 4, 5, 37
    ones_a = inputs.to_bf16_bits(np.ones((M, K), dtype=np.float32))
    ones_b = inputs.to_bf16_bits(np.ones((K, N), dtype=np.float32))
    bias = np.arange(N, dtype=np.float32) - 2.0
    got = oracle.addmm_bf16(ones_a, ones_b, bias)
    assert np.array_equal(got, np.broadcast_to(K + bias.astype(np.float64), (M, N)))


def test_bias_is_along_n_not_m():
    # M != N so a bias indexed by the row would read out of range or give other values.
    M, N, K = 3, 8, 4
    A = np.zeros((M, K), dtype=np.uint16)
    B = np.zeros((K, N), dtype=np.uint16)
    bias = np.arange(N, dtype=np.float32) * 3.0
    got = oracle.addmm_bf16(A, B, bias)
    for m in range(M):
        assert np.array_equal(got[m], bias.astype(np.float64))


def test_bf16_matches_torch_float64_addmm():
    p = inputs.bf16_problem(96, 80, 136, seed=21, bias="f32_normal")
    A = torch.from_numpy(inputs.bf16_bits_to_f32(p["A"]).astype(np.float64))
    B = torch.from_numpy(inputs.bf16_bits_to_f32(p["B"]).astype(np.float64))
    bias = torch.from_numpy(p["bias"].astype(np.float64))
    want = torch.addmm(bias, A, B).numpy()
    got = oracle.addmm_bf16(p["A"], p["B"], p["bias"])
    scale = (A.abs() @ B.abs()).numpy() + np.abs(p["bias"])[None, :]
    assert np.all(np.abs(got - want) <= 1e-12 * scale)


def test_transposed_operand_is_detected():
    # Non-square, non-symmetric operands: C must equal A @ B, not A @ B^T-like variants.
    rng = np.random.default_rng(12)
    A = inputs.to_bf16_bits(rng.integers(-3, 4, (5, 7)).astype(np.float32))
    B = inputs.to_bf16_bits(rng.integers(-3, 4, (7, 6)).astype(np.float32))
    got = oracle.addmm_bf16(A, B)
    Ai = inputs.bf16_bits_to_f32(A).astype(np.int64)
    Bi = inputs.bf16_bits_to_f32(B).astype(np.int64)
    assert np.array_equal(got, (Ai @ Bi).astype(np.float64))


def test_row_blocks_and_sampled_elements_agree_with_full():
    p = inputs.bf16_problem(40, 33, 64, seed=4, bias="bf16_uniform")
    full = oracle.addmm_bf16(p["A"], p["B"], p["bias"])
    part = oracle.addmm_bf16(p["A"], p["B"], p["bias"], rows=(7, 19))
    assert np.array_equal(part, full[7:19])
    rng = np.random.default_rng(0)
    ms, ns = rng.integers(0, 40, 50), rng.integers(0, 33, 50)
    at = oracle.addmm_bf16_at(p["A"], p["B"], p["bias"], ms, ns)
    assert np.array_equal(at, full[ms, ns])


# ---------------------------------------------------------------------------------------
# MX decode and MXFP4 GEMM
# ---------------------------------------------------------------------------------------

def test_e2m1_decode_matches_ocp_table():
    for code in range(16):
        v = oracle.e2m1_value(code)
        assert v == E2M1[code]
        assert math.copysign(1.0, v) == math.copysign(1.0, E2M1[code]), code


def test_e8m0_decode_is_power_of_two():
    for e in range(255):
        assert oracle.e8m0_value(e) == float(Fraction(2) ** (e - 127))
    assert math.isnan(oracle.e8m0_value(255))


def _mx_exact(codes, scales, K, row, k):
    c = _unpack_codes(codes[row], K)[k]
    return Fraction(E2M1[c]) * Fraction(2) ** (int(scales[row, k // 32]) - 127)


@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (3, 4, 64), (5, 2, 96)])
def test_mxfp4_bruteforce_exact_rationals(M, N, K):
    p = inputs.mxfp4_problem(M, N, K, seed=M + N + K, bias="bf16_uniform")
    got = oracle.addmm_mxfp4(p["A"], p["A_scale"], p["B"], p["B_scale"], p["bias"])
    for m in range(M):
        for n in range(N):
            exact = sum(_mx_exact(p["A"], p["A_scale"], K, m, k) *
                        _mx_exact(p["B"], p["B_scale"], K, n, k) for k in range(K))
            exact += Fraction(_bf16_to_float(int(p["bias"][n])))
            assert Fraction(got[m, n]) == exact


def _decode_mx_to_bf16(codes, scales, K):
    rows = codes.shape[0]
    vals = np.empty((rows, K), dtype=np.float32)
    for r in range(rows):
        unpacked = _unpack_codes(codes[r], K)
        for k in range(K):
            vals[r, k] = E2M1[unpacked[k]] * 2.0 ** (int(scales[r, k // 32]) - 127)
    bits = inputs.to_bf16_bits(vals)
    assert np.array_equal(inputs.bf16_bits_to_f32(bits), vals)  # exact in bf16
    return bits


def test_mxfp4_equals_bf16_gemm_of_decoded_operands():
    M, N, K = 9, 7, 128
    p = inputs.mxfp4_problem(M, N, K, seed=99, bias="f32_normal")
    a_dec = _decode_mx_to_bf16(p["A"], p["A_scale"], K)            # M x K
    b_dec = _decode_mx_to_bf16(p["B"], p["B_scale"], K).T.copy()   # K x N
    mx = oracle.addmm_mxfp4(p["A"], p["A_scale"], p["B"], p["B_scale"], p["bias"])
    bf = oracle.addmm_bf16(a_dec, b_dec, p["bias"])
    assert np.array_equal(mx, bf)


def test_mxfp4_scale_linearity():
    M, N, K = 4, 5, 96
    p = inputs.mxfp4_problem(M, N, K, seed=5)
    base = oracle.addmm_mxfp4(p["A"], p["A_scale"], p["B"], p["B_scale"])
    sa = p["A_scale"].copy()
    sa[2, 1] += 1     # double block 1 (k in [32, 64)) of row 2 of A
    bumped = oracle.addmm_mxfp4(p["A"], sa, p["B"], p["B_scale"])
    assert np.array_equal(np.delete(bumped, 2, axis=0), np.delete(base, 2, axis=0))
    for n in range(N):
        block = sum(_mx_exact(p["A"], p["A_scale"], K, 2, k) * _mx_exact(p["B"], p["B_scale"], K, n, k)
                    for k in range(32, 64))
        assert Fraction(bumped[2, n]) - Fraction(base[2, n]) == block


def test_mxfp4_nan_scale_poisons_exactly_its_row():
    M, N, K = 3, 4, 64
    p = inputs.mxfp4_problem(M, N, K, seed=8)
    sb = p["B_scale"].copy()
    sb[1, 0] = 255
    got = oracle.addmm_mxfp4(p["A"], p["A_scale"], p["B"], sb)
    assert np.all(np.isnan(got[:, 1]))
    assert not np.any(np.isnan(np.delete(got, 1, axis=1)))


def test_mxfp4_sampled_elements_agree_with_full():
    p = inputs.mxfp4_problem(20, 18, 64, seed=2, bias="bf16_uniform")
    full = oracle.addmm_mxfp4(p["A"], p["A_scale"], p["B"], p["B_scale"], p["bias"])
    rng = np.random.default_rng(1)
    ms, ns = rng.integers(0, 20, 40), rng.integers(0, 18, 40)
    at = oracle.addmm_mxfp4_at(p["A"], p["A_scale"], p["B"], p["B_scale"], p["bias"], ms, ns)
    assert np.array_equal(at, full[ms, ns])
    rows = oracle.addmm_mxfp4(p["A"], p["A_scale"], p["B"], p["B_scale"], p["bias"], rows=(3, 11))
    assert np.array_equal(rows, full[3:11])


# ---------------------------------------------------------------------------------------
# schedules
# ---------------------------------------------------------------------------------------

def _check_schedule(mode, T, I, g, hybrid_waves=0):
    segs = oracle.schedule(mode, T, I, g, hybrid_waves)
    whole = {oracle.MODE_STREAMK: 0,
             oracle.MODE_HYBRID: T - min(T, T % g + hybrid_waves * g)}.get(mode, T)
    cover = np.zeros((T, I), dtype=np.int64)
    owners = {}
    per_cta = {}
    for cta, tile, k0, k1, role in segs.tolist():
        assert 0 <= tile < T and 0 <= k0 < k1 <= I
        cover[tile, k0:k1] += 1
        per_cta.setdefault(cta, []).append((tile, k0, k1, role))
        if k0 == 0:
            assert tile not in owners
            owners[tile] = (cta, k1, role)
            assert role == (oracle.ROLE_FULL if k1 == I else oracle.ROLE_OWNER)
        else:
            assert role == oracle.ROLE_CONTRIB
    assert np.all(cover == 1), "every (tile, k-iteration) exactly once"
    assert set(owners) == set(range(T))
    for cta, lst in per_cta.items():
        contribs = [i for i, s in enumerate(lst) if s[3] == oracle.ROLE_CONTRIB]
        owned = [i for i, s in enumerate(lst) if s[3] == oracle.ROLE_OWNER]
        assert len(contribs) <= 1, "a CTA spills at most once"
        assert len(owned) <= 1
        # execution order: the Stream-K region's whole tiles, then the contribution, then
        # the shared owned tile, then the tiles of the whole-tile region
        region = [s for s in lst if s[0] >= whole]
        order = [s[3] for s in region]
        assert order == sorted(order, key=lambda r: {oracle.ROLE_FULL: 0, oracle.ROLE_CONTRIB: 1,
                                                      oracle.ROLE_OWNER: 2}[r])
        assert lst[:len(region)] == region
        # the contribution is the start of the CTA's range: it precedes every other piece
        # of the range in linear order
        if contribs:
            t, k0, k1, _ = lst[contribs[0]]
            assert all((tt, kk0) > (t, k0) for tt, kk0, _, rr in lst if rr != oracle.ROLE_CONTRIB
                       and tt >= t)
    # contributions of a split tile come from the CTAs right after the owner, in order
    for tile, (owner, k1, role) in owners.items():
        if role != oracle.ROLE_OWNER:
            continue
        parts = sorted((cta, k0, kk1) for cta, t, k0, kk1, r in segs.tolist()
                       if t == tile and r == oracle.ROLE_CONTRIB)
        assert [c for c, _, _ in parts] == list(range(owner + 1, owner + 1 + len(parts)))
        pos = k1
        for _, k0, kk1 in parts:
            assert k0 == pos
            pos = kk1
        assert pos == I
    return segs, per_cta


@pytest.mark.parametrize("T,I", [(4, 8), (1, 1), (7, 3), (225, 16), (13, 64), (2, 100)])
@pytest.mark.parametrize("g", [1, 2, 3, 5, 16, 148, 152])
def test_streamk_and_hybrid_schedule_invariants(T, I, g):
    g_sk = min(g, T * I)
    segs, per_cta = _check_schedule(oracle.MODE_STREAMK, T, I, g_sk)
    lens = [sum(k1 - k0 for _, k0, k1, _ in per_cta.get(c, [])) for c in range(g_sk)]
    assert max(lens) - min(lens) <= 1
    assert lens == sorted(lens, reverse=True)   # the longer ranges come first
    segs, per_cta = _check_schedule(oracle.MODE_HYBRID, T, I, g_sk)
    sk_tiles = T % g_sk
    for cta, lst in per_cta.items():
        whole = [t for t, k0, k1, r in lst if t < T - sk_tiles]
        assert whole == list(range(cta, T - sk_tiles, g_sk))
        assert all(k0 == 0 and k1 == I for t, k0, k1, r in lst if t < T - sk_tiles)


@pytest.mark.parametrize("T,I", [(81, 128), (225, 16), (13, 64), (1024, 32), (7, 3)])
@pytest.mark.parametrize("g", [2, 5, 76, 152])
@pytest.mark.parametrize("waves", [1, 2])
def test_two_tile_hybrid_schedule(T, I, g, waves):
    # the hybrid with `waves` full waves added to its Stream-K region: the same invariants,
    # and every CTA's Stream-K share is at least `waves` whole tiles' worth when the tiles
    # allow it
    g = min(g, T * I)
    segs, per_cta = _check_schedule(oracle.MODE_HYBRID, T, I, g, waves)
    sk_tiles = min(T, T % g + waves * g)
    sk_iters = [sum(k1 - k0 for t, k0, k1, _ in per_cta.get(c, []) if t >= T - sk_tiles)
                for c in range(g)]
    assert sum(sk_iters) == sk_tiles * I
    if sk_tiles < T:
        assert min(sk_iters) >= waves * I
    for cta, lst in per_cta.items():
        whole = [t for t, k0, k1, r in lst if t < T - sk_tiles]
        assert whole == list(range(cta, T - sk_tiles, g))
    # waves = 0 is the plain hybrid; enough waves make it Stream-K over every tile
    assert np.array_equal(oracle.schedule(oracle.MODE_HYBRID, T, I, g, 0),
                          oracle.schedule(oracle.MODE_HYBRID, T, I, g))
    assert np.array_equal(oracle.schedule(oracle.MODE_HYBRID, T, I, g, T),
                          oracle.schedule(oracle.MODE_STREAMK, T, I, g))


@pytest.mark.parametrize("T,g", [(1, 1), (10, 3), (1024, 148), (225, 152), (5, 9)])
def test_persistent_and_dp_schedules(T, g):
    segs, per_cta = _check_schedule(oracle.MODE_PERSISTENT, T, 4, min(g, T))
    for cta, lst in per_cta.items():
        assert [t for t, *_ in lst] == list(range(cta, T, min(g, T)))
    segs, per_cta = _check_schedule(oracle.MODE_DP, T, 4, T)
    assert sorted(per_cta) == list(range(T))
    assert all(len(v) == 1 for v in per_cta.values())


def test_streamk_split_of_the_256_cube_over_3_ctas_matches_hand_derivation():
    want = np.loadtxt(os.path.join(GOLDEN, "streamk_256x256x512_g3.txt"), dtype=np.int64)
    got = oracle.schedule(oracle.MODE_STREAMK, 4, 8, 3)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("mode", [oracle.MODE_DP, oracle.MODE_PERSISTENT,
                                  oracle.MODE_STREAMK, oracle.MODE_HYBRID])
@pytest.mark.parametrize("g", [1, 2, 3, 5, 7, 16])
def test_schedule_invariance_of_the_result(mode, g):
    # exact integer inputs: every schedule gives bit-identical binary64 results
    p = inputs.bf16_problem(70, 50, 200, seed=31, integer=True, bias="f32_int")
    plain = oracle.addmm_bf16(p["A"], p["B"], p["bias"])
    sched = oracle.addmm_bf16_scheduled(p["A"], p["B"], p["bias"], mode, 32, 16, 16, g)
    assert np.array_equal(plain, sched)
    # random inputs: equal up to binary64 reassociation
    q = inputs.bf16_problem(40, 30, 100, seed=32, bias="f32_normal")
    plain = oracle.addmm_bf16(q["A"], q["B"], q["bias"])
    sched = oracle.addmm_bf16_scheduled(q["A"], q["B"], q["bias"], mode, 16, 16, 8, g)
    assert np.allclose(sched, plain, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------------------
# stored-transposed GEMM and addmm backward
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("ta", [False, True])
@pytest.mark.parametrize("tb", [False, True])
def test_transposed_gemm_bruteforce_exact_rationals(ta, tb):
    rng = np.random.default_rng(40 + 2 * ta + tb)
    M, N, K = 3, 5, 4
    A = _dyadic_bf16(rng, (K, M) if ta else (M, K))
    B = _dyadic_bf16(rng, (N, K) if tb else (K, N))
    got = oracle.gemm_bf16_t(A, ta, B, tb)
    for m in range(M):
        for n in range(N):
            exact = Fraction(0)
            for k in range(K):
                a = A[k, m] if ta else A[m, k]
                b = B[n, k] if tb else B[k, n]
                exact += Fraction(_bf16_to_float(int(a))) * Fraction(_bf16_to_float(int(b)))
            assert Fraction(got[m, n]) == exact
    ms, ns = np.array([0, 2, 1]), np.array([4, 0, 3])
    assert np.array_equal(oracle.gemm_bf16_t_at(A, ta, B, tb, ms, ns), got[ms, ns])


def test_addmm_backward_matches_torch_autograd_float64():
    p = inputs.bf16_problem(48, 40, 56, seed=17, bias="f32_normal")
    dC = inputs.to_bf16_bits(np.random.default_rng(18).standard_normal((48, 40)).astype(np.float32))
    A = torch.from_numpy(inputs.bf16_bits_to_f32(p["A"]).astype(np.float64)).requires_grad_()
    B = torch.from_numpy(inputs.bf16_bits_to_f32(p["B"]).astype(np.float64)).requires_grad_()
    bias = torch.from_numpy(p["bias"].astype(np.float64)).requires_grad_()
    torch.addmm(bias, A, B).backward(torch.from_numpy(inputs.bf16_bits_to_f32(dC).astype(np.float64)))
    dA, dB, db = oracle.addmm_backward_bf16(dC, p["A"], p["B"])
    assert np.allclose(dA, A.grad.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(dB, B.grad.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(db, bias.grad.numpy(), rtol=1e-12, atol=1e-12)


def test_addmm_backward_integer_closed_forms():
    rng = np.random.default_rng(19)
    M, N, K = 9, 7, 5
    A = rng.integers(-5, 6, (M, K))
    B = rng.integers(-5, 6, (K, N))
    dC = rng.integers(-5, 6, (M, N))
    bits = lambda x: inputs.to_bf16_bits(x.astype(np.float32))
    dA, dB, db = oracle.addmm_backward_bf16(bits(dC), bits(A), bits(B))
    assert np.array_equal(dA, (dC @ B.T).astype(np.float64))
    assert np.array_equal(dB, (A.T @ dC).astype(np.float64))
    assert np.array_equal(db, dC.sum(axis=0).astype(np.float64))
    # the backward GEMMs are the forward GEMM of stored-transposed operands
    assert np.array_equal(dA, oracle.gemm_bf16_t(bits(dC), False, bits(B), True))
    assert np.array_equal(dB, oracle.gemm_bf16_t(bits(A), True, bits(dC), False))


# ---------------------------------------------------------------------------------------
# fp8 (E4M3)
# ---------------------------------------------------------------------------------------

def test_e4m3_decode_matches_torch_float8_and_the_format_limits():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = oracle.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c] and math.copysign(1, v) == math.copysign(1, ref[c]), c
    assert oracle.e4m3_value(0x7E) == 448.0            # largest finite
    assert oracle.e4m3_value(0x01) == 2.0 ** -9         # smallest subnormal
    assert oracle.e4m3_value(0x08) == 2.0 ** -6         # smallest normal
    assert oracle.e4m3_value(0x38) == 1.0 and oracle.e4m3_value(0xC4) == -3.0
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))


def test_fp8_bruteforce_exact_rationals_and_cross_format():
    rng = np.random.default_rng(61)
    M, N, K = 4, 6, 9
    A = rng.integers(0, 256, (M, K)).astype(np.uint8)
    B = rng.integers(0, 256, (K, N)).astype(np.uint8)
    A[(A & 0x7F) == 0x7F] = 0x3C          # no NaN codes
    B[(B & 0x7F) == 0x7F] = 0x44
    bias = rng.standard_normal(N).astype(np.float32)
    got = oracle.addmm_fp8(A, B, bias)

    def dec(c):      # sign, exponent and mantissa fields read by hand, as exact rationals
        c = int(c)
        e, m = (c >> 3) & 15, c & 7
        v = Fraction(m, 512) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        return -v if c & 0x80 else v

    for m in range(M):
        for n in range(N):
            exact = sum(dec(A[m, k]) * dec(B[k, n]) for k in range(K)) + Fraction(float(bias[n]))
            assert Fraction(got[m, n]) == exact
    # decoded E4M3 values are exact in bf16: the fp8 GEMM equals the bf16 GEMM of them
    a16 = inputs.to_bf16_bits(torch.from_numpy(A).view(torch.float8_e4m3fn).float().numpy())
    b16 = inputs.to_bf16_bits(torch.from_numpy(B).view(torch.float8_e4m3fn).float().numpy())
    assert np.array_equal(got, oracle.addmm_bf16(a16, b16, bias))
    ms, ns = np.array([0, 3, 2]), np.array([5, 1, 0])
    assert np.array_equal(oracle.addmm_fp8_at(A, B, bias, ms, ns), got[ms, ns])
    assert np.array_equal(oracle.addmm_fp8(A, B, bias, rows=(1, 3)), got[1:3])


def test_fp8_generator_draws_exact_integers_and_no_nan():
    p = inputs.fp8_problem(64, 48, 96, seed=2, integer=True, bias="f32_int")
    vals = torch.from_numpy(p["A"]).view(torch.float8_e4m3fn).float().numpy()
    assert np.all(vals == np.round(vals)) and np.abs(vals).max() <= 8
    q = inputs.fp8_problem(64, 48, 96, seed=2, operand_scale="sqrt_k")
    assert not np.any((q["A"] & 0x7F) == 0x7F) and not np.any((q["B"] & 0x7F) == 0x7F)
