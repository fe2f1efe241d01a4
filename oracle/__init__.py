"""CPU oracle for the addmm GEMM path (test infrastructure only).

The oracle is plain C++ (``oracle.cpp``) compiled with the host compiler and loaded with
ctypes.  It computes ``C = A @ B + bias[n]`` with exact products, binary64 accumulation in
ascending k, the bias added once, and a single round-to-nearest-even to the output type.
It shares no code with the CUDA library and must only be used by the tests, the smoke check
and the benchmark's CPU-baseline leg; the product path never imports it.

Arrays are numpy: bf16 data is carried as ``uint16`` bit patterns, MXFP4 codes and E8M0
scales as ``uint8``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB_DIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")
_lock = threading.Lock()
_handle = None

MODE_DP, MODE_PERSISTENT, MODE_STREAMK, MODE_HYBRID = 0, 1, 2, 3
ROLE_FULL, ROLE_OWNER, ROLE_CONTRIB = 0, 1, 2
F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with g++ (no fused multiply-add, so results match on every
    host architecture).  Returns the library path."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _lib():
    global _handle
    with _lock:
        if _handle is None:
            lib = ctypes.CDLL(build())
            d, i64, i32, vp = ctypes.c_double, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            lib.oracle_bf16_value.restype = d
            lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
            lib.oracle_e2m1_value.restype = d
            lib.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e8m0_value.restype = d
            lib.oracle_e8m0_value.argtypes = [ctypes.c_uint8]
            lib.oracle_round_bf16.restype = ctypes.c_uint16
            lib.oracle_round_bf16.argtypes = [d]
            lib.oracle_round_output.restype = None
            lib.oracle_round_output.argtypes = [vp, vp, i64, i32]
            lib.oracle_addmm_bf16_rows.restype = i32
            lib.oracle_addmm_bf16_rows.argtypes = [vp, vp, vp, i32, i64, i64, i64, i64, i64,
                                                   vp, i32]
            lib.oracle_addmm_bf16_at.restype = i32
            lib.oracle_addmm_bf16_at.argtypes = [vp, vp, vp, i32, i64, i64, i64, vp, vp, i64,
                                                 vp, i32]
            lib.oracle_addmm_mxfp4_rows.restype = i32
            lib.oracle_addmm_mxfp4_rows.argtypes = [vp, vp, vp, vp, vp, i32, i64, i64, i64,
                                                    i64, i64, vp, i32]
            lib.oracle_addmm_mxfp4_at.restype = i32
            lib.oracle_addmm_mxfp4_at.argtypes = [vp, vp, vp, vp, vp, i32, i64, i64, i64, vp,
                                                  vp, i64, vp, i32]
            lib.oracle_schedule.restype = i64
            lib.oracle_schedule.argtypes = [i32, i64, i64, i64, vp, i64]
            lib.oracle_schedule_hybrid.restype = i64
            lib.oracle_schedule_hybrid.argtypes = [i32, i64, i64, i64, i64, vp, i64]
            lib.oracle_addmm_bf16_scheduled.restype = i32
            lib.oracle_addmm_bf16_scheduled.argtypes = [vp, vp, vp, i32, i64, i64, i64, i32,
                                                        i64, i64, i64, i64, vp]
            lib.oracle_gemm_bf16_t_rows.restype = i32
            lib.oracle_gemm_bf16_t_rows.argtypes = [vp, i32, vp, i32, vp, i32, i64, i64, i64, i64,
                                                    i64, vp, i32]
            lib.oracle_gemm_bf16_t_at.restype = i32
            lib.oracle_gemm_bf16_t_at.argtypes = [vp, i32, vp, i32, i64, i64, i64, vp, vp, i64, vp,
                                                  i32]
            lib.oracle_addmm_backward_bf16.restype = i32
            lib.oracle_addmm_backward_bf16.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, vp, i32]
            lib.oracle_e4m3_value.restype = d
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.oracle_addmm_fp8_rows.restype = i32
            lib.oracle_addmm_fp8_rows.argtypes = [vp, vp, vp, i32, i64, i64, i64, i64, i64, vp, i32]
            lib.oracle_addmm_fp8_at.restype = i32
            lib.oracle_addmm_fp8_at.argtypes = [vp, vp, vp, i32, i64, i64, i64, vp, vp, i64, vp,
                                                i32]
            lib.oracle_hardware_threads.restype = i32
            lib.oracle_hardware_threads.argtypes = []
            _handle = lib
    return _handle


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _bias(bias):
    """Return (array, dtype code) for a bias given as float32 or bf16 bits (uint16)."""
    if bias is None:
        return None, F32
    bias = np.ascontiguousarray(bias)
    if bias.dtype == np.float32:
        return bias, F32
    if bias.dtype == np.uint16:
        return bias, BF16
    raise TypeError("bias must be float32 or bf16 bits (uint16)")


# ---- scalar encodings -------------------------------------------------------------------

def bf16_value(bits: int) -> float:
    return _lib().oracle_bf16_value(int(bits))


def e2m1_value(code: int) -> float:
    return _lib().oracle_e2m1_value(int(code))


def e8m0_value(e: int) -> float:
    return _lib().oracle_e8m0_value(int(e))


def e4m3_value(code: int) -> float:
    return _lib().oracle_e4m3_value(int(code))


def round_bf16(x: float) -> int:
    return int(_lib().oracle_round_bf16(float(x)))


def round_output(x: np.ndarray, out_dtype: int) -> np.ndarray:
    """Round binary64 values to fp32 (out_dtype 0) or bf16 bits (out_dtype 1)."""
    x = _c(x, np.float64)
    y = np.empty(x.shape, dtype=np.float32 if out_dtype == F32 else np.uint16)
    _lib().oracle_round_output(_ptr(x), _ptr(y), x.size, out_dtype)
    return y


# ---- GEMMs ---------------------------------------------------------------------------------

def addmm_bf16(A, B, bias=None, rows=None, threads=0):
    """binary64 C (before output rounding) for bf16 A (M,K) and B (K,N) given as uint16 bits.
    ``rows=(m0, m1)`` restricts the computation to a block of rows."""
    A, B = _c(A, np.uint16), _c(B, np.uint16)
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    bias, bdt = _bias(bias)
    m0, m1 = rows if rows is not None else (0, M)
    out = np.empty((m1 - m0, N), dtype=np.float64)
    rc = _lib().oracle_addmm_bf16_rows(_ptr(A), _ptr(B), _ptr(bias), bdt, M, N, K, m0, m1,
                                       _ptr(out), threads)
    if rc:
        raise ValueError(f"oracle_addmm_bf16_rows failed ({rc})")
    return out


def addmm_bf16_at(A, B, bias, ms, ns, threads=0):
    A, B = _c(A, np.uint16), _c(B, np.uint16)
    M, K = A.shape
    N = B.shape[1]
    bias, bdt = _bias(bias)
    ms, ns = _c(ms, np.int64), _c(ns, np.int64)
    out = np.empty(ms.shape, dtype=np.float64)
    rc = _lib().oracle_addmm_bf16_at(_ptr(A), _ptr(B), _ptr(bias), bdt, M, N, K, _ptr(ms),
                                     _ptr(ns), ms.size, _ptr(out), threads)
    if rc:
        raise ValueError(f"oracle_addmm_bf16_at failed ({rc})")
    return out


def addmm_mxfp4(A, A_scale, B, B_scale, bias=None, rows=None, threads=0):
    """binary64 C for MXFP4 A (M, K/2 bytes) with A_scale (M, K/32) and B (N, K/2 bytes)
    with B_scale (N, K/32)."""
    A, B = _c(A, np.uint8), _c(B, np.uint8)
    A_scale, B_scale = _c(A_scale, np.uint8), _c(B_scale, np.uint8)
    M, K = A.shape[0], A.shape[1] * 2
    N = B.shape[0]
    assert B.shape[1] * 2 == K and A_scale.shape == (M, K // 32) and B_scale.shape == (N, K // 32)
    bias, bdt = _bias(bias)
    m0, m1 = rows if rows is not None else (0, M)
    out = np.empty((m1 - m0, N), dtype=np.float64)
    rc = _lib().oracle_addmm_mxfp4_rows(_ptr(A), _ptr(A_scale), _ptr(B), _ptr(B_scale),
                                        _ptr(bias), bdt, M, N, K, m0, m1, _ptr(out), threads)
    if rc:
        raise ValueError(f"oracle_addmm_mxfp4_rows failed ({rc})")
    return out


def addmm_mxfp4_at(A, A_scale, B, B_scale, bias, ms, ns, threads=0):
    A, B = _c(A, np.uint8), _c(B, np.uint8)
    A_scale, B_scale = _c(A_scale, np.uint8), _c(B_scale, np.uint8)
    M, K = A.shape[0], A.shape[1] * 2
    N = B.shape[0]
    bias, bdt = _bias(bias)
    ms, ns = _c(ms, np.int64), _c(ns, np.int64)
    out = np.empty(ms.shape, dtype=np.float64)
    rc = _lib().oracle_addmm_mxfp4_at(_ptr(A), _ptr(A_scale), _ptr(B), _ptr(B_scale),
                                      _ptr(bias), bdt, M, N, K, _ptr(ms), _ptr(ns), ms.size,
                                      _ptr(out), threads)
    if rc:
        raise ValueError(f"oracle_addmm_mxfp4_at failed ({rc})")
    return out


def addmm_fp8(A, B, bias=None, rows=None, threads=0):
    """binary64 C for E4M3 A (M,K) and B (K,N) given as uint8 codes."""
    A, B = _c(A, np.uint8), _c(B, np.uint8)
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    bias, bdt = _bias(bias)
    m0, m1 = rows if rows is not None else (0, M)
    out = np.empty((m1 - m0, N), dtype=np.float64)
    rc = _lib().oracle_addmm_fp8_rows(_ptr(A), _ptr(B), _ptr(bias), bdt, M, N, K, m0, m1,
                                      _ptr(out), threads)
    if rc:
        raise ValueError(f"oracle_addmm_fp8_rows failed ({rc})")
    return out


def addmm_fp8_at(A, B, bias, ms, ns, threads=0):
    """addmm_fp8 at the positions (ms[i], ns[i])."""
    A, B = _c(A, np.uint8), _c(B, np.uint8)
    M, K = A.shape
    N = B.shape[1]
    bias, bdt = _bias(bias)
    ms, ns = _c(ms, np.int64), _c(ns, np.int64)
    out = np.empty(ms.shape, dtype=np.float64)
    rc = _lib().oracle_addmm_fp8_at(_ptr(A), _ptr(B), _ptr(bias), bdt, M, N, K, _ptr(ms),
                                    _ptr(ns), ms.size, _ptr(out), threads)
    if rc:
        raise ValueError(f"oracle_addmm_fp8_at failed ({rc})")
    return out


def gemm_bf16_t(A, trans_a, B, trans_b, bias=None, rows=None, threads=0):
    """binary64 op(A) @ op(B) (+ bias): A stored (M,K), or (K,M) when trans_a; B stored (K,N),
    or (N,K) when trans_b; bf16 bits as uint16."""
    A, B = _c(A, np.uint16), _c(B, np.uint16)
    M, K = (A.shape[1], A.shape[0]) if trans_a else A.shape
    N, K2 = (B.shape[0], B.shape[1]) if trans_b else (B.shape[1], B.shape[0])
    assert K == K2
    bias, bdt = _bias(bias)
    m0, m1 = rows if rows is not None else (0, M)
    out = np.empty((m1 - m0, N), dtype=np.float64)
    rc = _lib().oracle_gemm_bf16_t_rows(_ptr(A), int(bool(trans_a)), _ptr(B), int(bool(trans_b)),
                                        _ptr(bias), bdt, M, N, K, m0, m1, _ptr(out), threads)
    if rc:
        raise ValueError(f"oracle_gemm_bf16_t_rows failed ({rc})")
    return out


def gemm_bf16_t_at(A, trans_a, B, trans_b, ms, ns, threads=0):
    A, B = _c(A, np.uint16), _c(B, np.uint16)
    M, K = (A.shape[1], A.shape[0]) if trans_a else A.shape
    N = B.shape[0] if trans_b else B.shape[1]
    ms, ns = _c(ms, np.int64), _c(ns, np.int64)
    out = np.empty(ms.shape, dtype=np.float64)
    rc = _lib().oracle_gemm_bf16_t_at(_ptr(A), int(bool(trans_a)), _ptr(B), int(bool(trans_b)),
                                      M, N, K, _ptr(ms), _ptr(ns), ms.size, _ptr(out), threads)
    if rc:
        raise ValueError(f"oracle_gemm_bf16_t_at failed ({rc})")
    return out


def addmm_backward_bf16(dC, A, B, threads=0):
    """(dA, dB, dbias) in binary64 for C = A @ B + bias, given dC; bf16 bits as uint16."""
    dC, A, B = _c(dC, np.uint16), _c(A, np.uint16), _c(B, np.uint16)
    M, K = A.shape
    N = B.shape[1]
    assert dC.shape == (M, N) and B.shape == (K, N)
    dA = np.empty((M, K), dtype=np.float64)
    dB = np.empty((K, N), dtype=np.float64)
    db = np.empty(N, dtype=np.float64)
    rc = _lib().oracle_addmm_backward_bf16(_ptr(dC), _ptr(A), _ptr(B), M, N, K, _ptr(dA),
                                           _ptr(dB), _ptr(db), threads)
    if rc:
        raise ValueError(f"oracle_addmm_backward_bf16 failed ({rc})")
    return dA, dB, db


def schedule(mode, tiles, iters, grid, hybrid_waves=0):
    """List of (cta, tile, k_begin, k_end, role) segments, each CTA's in execution order.
    hybrid_waves: full waves added to the hybrid's Stream-K region (the two-tile form)."""
    lib = _lib()
    n = lib.oracle_schedule_hybrid(mode, tiles, iters, grid, hybrid_waves, None, 0)
    if n < 0:
        raise ValueError("bad schedule arguments")
    rows = np.zeros((max(n, 1), 5), dtype=np.int64)
    lib.oracle_schedule_hybrid(mode, tiles, iters, grid, hybrid_waves, _ptr(rows), n)
    return rows[:n]


def addmm_bf16_scheduled(A, B, bias, mode, BM, BN, BK, grid):
    """binary64 C summed tile by tile in the order a schedule would: owner segment, then
    contributions by increasing CTA, then the bias once."""
    A, B = _c(A, np.uint16), _c(B, np.uint16)
    M, K = A.shape
    N = B.shape[1]
    bias, bdt = _bias(bias)
    out = np.empty((M, N), dtype=np.float64)
    rc = _lib().oracle_addmm_bf16_scheduled(_ptr(A), _ptr(B), _ptr(bias), bdt, M, N, K, mode,
                                            BM, BN, BK, grid, _ptr(out))
    if rc:
        raise ValueError(f"oracle_addmm_bf16_scheduled failed ({rc})")
    return out


def hardware_threads() -> int:
    return int(_lib().oracle_hardware_threads())
