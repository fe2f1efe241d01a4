"""Seeded synthetic inputs for the addmm GEMM path.

This module only draws random numbers and packs them into the storage formats the library
takes; it does none of the GEMM's arithmetic.  Both the CUDA path and the CPU oracle are fed
from it.  Every generator takes an explicit seed (numpy PCG64).

Storage conventions (host, numpy):
  * bf16 tensors are ``uint16`` arrays of bf16 bit patterns (rounded from fp32 by torch's
    round-to-nearest-even conversion);
  * fp32 tensors are ``float32``;
  * fp8 operands are ``uint8`` OCP E4M3 codes (torch ``float8_e4m3fn`` bit patterns);
  * MXFP4 operands are ``uint8`` code bytes, two E2M1 codes per byte packed along K with the
    even-k element in the low nibble, rows x K/2; their E8M0 scales are ``uint8`` rows x K/32.

The distributions follow the workload descriptions of the addmm/Stream-K benchmarks:
N(0,1) or N(0,1)/sqrt(K) operands rounded to bf16, fp32 N(0,1) or bf16 U(-1,1) bias, and for
MXFP4 codes uniform over all 16 values with scale exponents uniform in [-4, 4].
"""
from __future__ import annotations

import numpy as np
import torch


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), nearest-even, via torch's conversion."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact widening)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal_f32(rng, shape, scale):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return x


def to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    """fp32 array -> OCP FP8 E4M3 codes (uint8), via torch's float8_e4m3fn conversion."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


def fp8_problem(M, N, K, *, seed, operand_scale="unit", bias="none", integer=False):
    """E4M3 A (M,K) and B (K,N) codes plus an optional bias (as bf16_problem's).  A is N(0,1);
    B is N(0,1), or N(0,1)/sqrt(K) for operand_scale "sqrt_k", so that C stays O(1)."""
    rng = np.random.default_rng(seed)
    if integer:
        A = to_e4m3_codes(rng.integers(-8, 9, size=(M, K)).astype(np.float32))
        B = to_e4m3_codes(rng.integers(-8, 9, size=(K, N)).astype(np.float32))
    else:
        s = 1.0 if operand_scale == "unit" else 1.0 / np.sqrt(K)
        A = to_e4m3_codes(_normal_f32(rng, (M, K), 1.0))
        B = to_e4m3_codes(_normal_f32(rng, (K, N), s))
    b = None
    if bias == "f32_normal":
        b = rng.standard_normal(size=N, dtype=np.float32)
    elif bias == "bf16_uniform":
        b = to_bf16_bits(rng.uniform(-1.0, 1.0, size=N).astype(np.float32))
    elif bias == "f32_int":
        b = rng.integers(-8, 9, size=N).astype(np.float32)
    elif bias != "none":
        raise ValueError(bias)
    return {"A": A, "B": B, "bias": b, "M": M, "N": N, "K": K}


def bf16_problem(M, N, K, *, seed, operand_scale="unit", bias="none", integer=False):
    """A (M,K) and B (K,N) bf16 operands plus an optional bias[N].

    operand_scale: "unit" for N(0,1), "sqrt_k" for N(0,1)/sqrt(K).
    bias: "none", "f32_normal" (fp32 N(0,1)), "bf16_uniform" (bf16 U(-1,1)),
          "f32_int" / "bf16_int" (integers in [-8, 8]).
    integer=True draws A and B as integers in [-8, 8] instead (exactly representable; every
    partial sum is exact in fp32 while K * 64 < 2^24).
    """
    rng = np.random.default_rng(seed)
    if integer:
        A = to_bf16_bits(rng.integers(-8, 9, size=(M, K)).astype(np.float32))
        B = to_bf16_bits(rng.integers(-8, 9, size=(K, N)).astype(np.float32))
    else:
        s = 1.0 if operand_scale == "unit" else 1.0 / np.sqrt(K)
        A = to_bf16_bits(_normal_f32(rng, (M, K), s))
        B = to_bf16_bits(_normal_f32(rng, (K, N), s))
    b = None
    if bias == "f32_normal":
        b = rng.standard_normal(size=N, dtype=np.float32)
    elif bias == "bf16_uniform":
        b = to_bf16_bits(rng.uniform(-1.0, 1.0, size=N).astype(np.float32))
    elif bias == "f32_int":
        b = rng.integers(-8, 9, size=N).astype(np.float32)
    elif bias == "bf16_int":
        b = to_bf16_bits(rng.integers(-8, 9, size=N).astype(np.float32))
    elif bias != "none":
        raise ValueError(bias)
    return {"A": A, "B": B, "bias": b, "M": M, "N": N, "K": K}


def mxfp4_problem(M, N, K, *, seed, bias="none", exp_range=4, codes=None):
    """MXFP4 A (M, K/2 bytes) + A_scale (M, K/32) and B (N, K/2 bytes) + B_scale (N, K/32).

    Codes are uniform over 0..15 (each byte = two independent nibbles); scale exponents are
    127 + U{-exp_range..exp_range}, independent per (row, 32-block).  ``codes`` may restrict the
    code values drawn (a sequence of allowed 4-bit codes)."""
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    rng = np.random.default_rng(seed)

    def draw_codes(rows):
        if codes is None:
            lo = rng.integers(0, 16, size=(rows, K // 2), dtype=np.uint8)
            hi = rng.integers(0, 16, size=(rows, K // 2), dtype=np.uint8)
        else:
            allowed = np.asarray(codes, dtype=np.uint8)
            lo = allowed[rng.integers(0, len(allowed), size=(rows, K // 2))]
            hi = allowed[rng.integers(0, len(allowed), size=(rows, K // 2))]
        return (lo | (hi << 4)).astype(np.uint8)

    A = draw_codes(M)
    A_scale = (127 + rng.integers(-exp_range, exp_range + 1, size=(M, K // 32))).astype(np.uint8)
    B = draw_codes(N)
    B_scale = (127 + rng.integers(-exp_range, exp_range + 1, size=(N, K // 32))).astype(np.uint8)
    b = None
    if bias == "bf16_uniform":
        b = to_bf16_bits(rng.uniform(-1.0, 1.0, size=N).astype(np.float32))
    elif bias == "f32_normal":
        b = rng.standard_normal(size=N, dtype=np.float32)
    elif bias != "none":
        raise ValueError(bias)
    return {"A": A, "A_scale": A_scale, "B": B, "B_scale": B_scale, "bias": b,
            "M": M, "N": N, "K": K}


# The benchmark workloads, by name: (format, M, N, K, generator kwargs, output dtype).
WORKLOADS = {
    "addmm_bf16_256x256x512_f32out": ("bf16", 256, 256, 512,
                                      dict(operand_scale="unit", bias="f32_normal"), "f32", 1234),
    "addmm_bf16_8192": ("bf16", 8192, 8192, 8192,
                        dict(operand_scale="sqrt_k", bias="bf16_uniform"), "bf16", 1235),
    "gemm_bf16_1920x1920x16384": ("bf16", 1920, 1920, 16384,
                                  dict(operand_scale="sqrt_k", bias="none"), "bf16", 1236),
    "addmm_mxfp4_8192": ("mxfp4", 8192, 8192, 8192, dict(bias="bf16_uniform"), "bf16", 1237),
    "gemm_bf16_4096": ("bf16", 4096, 4096, 4096,
                       dict(operand_scale="sqrt_k", bias="none"), "bf16", 1238),
    "gemm_bf16_skinny_64x14336x4096": ("bf16", 64, 14336, 4096,
                                       dict(operand_scale="sqrt_k", bias="none"), "bf16", 1238),
    "addmm_fp8_8192": ("fp8", 8192, 8192, 8192,
                       dict(operand_scale="sqrt_k", bias="bf16_uniform"), "bf16", 1239),
    # few tiles, long K: 16 SM-pair tiles for 76 pairs, the case Stream-K exists for
    "gemm_bf16_1024x1024x16384": ("bf16", 1024, 1024, 16384,
                                  dict(operand_scale="sqrt_k", bias="none"), "bf16", 1241),
}


def workload(name, seed=None):
    fmt, M, N, K, kw, out, default_seed = WORKLOADS[name]
    s = default_seed if seed is None else seed
    if fmt == "bf16":
        p = bf16_problem(M, N, K, seed=s, **kw)
    elif fmt == "fp8":
        p = fp8_problem(M, N, K, seed=s, **kw)
    else:
        p = mxfp4_problem(M, N, K, seed=s, **kw)
    p["format"], p["out_dtype"] = fmt, out
    return p
