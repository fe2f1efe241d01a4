"""GB300-native persistent / SM-constrained / Stream-K addmm GEMM (bf16 and MXFP4).

A thin ctypes binding over the C ABI in ``include/sk_gemm.h`` (library ``_lib/libskgemm.so``,
built by ``_build.build()``).  The functions named like the C entry points take raw device
pointers (ints) and sizes; the ``gemm_bf16`` / ``gemm_mxfp4`` helpers take torch tensors and
only marshal them: every step of the computation runs in the CUDA library.  Nothing here falls
back to another implementation: if the library is missing, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

MODES = {"dp": 0, "persistent": 1, "streamk": 2, "hybrid": 3, "auto": 4}
SK_F32, SK_BF16 = 0, 1
STATUS = {0: "SK_OK", 1: "SK_ERR_INVALID_ARG", 2: "SK_ERR_UNSUPPORTED", 3: "SK_ERR_OOM",
          4: "SK_ERR_CUDA", 5: "SK_ERR_TIMEOUT", 6: "SK_ERR_NOT_CORESIDENT"}
SK_OK, SK_ERR_INVALID_ARG, SK_ERR_UNSUPPORTED, SK_ERR_OOM = 0, 1, 2, 3
SK_ERR_CUDA, SK_ERR_TIMEOUT, SK_ERR_NOT_CORESIDENT = 4, 5, 6

_lock = threading.Lock()
_handle = None


class SkError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class Options(ctypes.Structure):
    """sk_options_t."""
    _fields_ = [("tile_n", ctypes.c_int32), ("raster_group", ctypes.c_int32),
                ("spin_timeout_ns", ctypes.c_int64), ("inject_faults", ctypes.c_int32),
                ("drop_release_cta", ctypes.c_int32), ("tile_m", ctypes.c_int32),
                ("hybrid_sk_waves", ctypes.c_int32), ("resident_limit", ctypes.c_int32),
                ("sm_record_len", ctypes.c_int32), ("sm_record", ctypes.c_void_p),
                ("tile_k", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class Plan(ctypes.Structure):
    """sk_plan_t."""
    _fields_ = [("format", ctypes.c_int32), ("mode", ctypes.c_int32),
                ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32), ("tile_k", ctypes.c_int32),
                ("tiles_m", ctypes.c_int32), ("tiles_n", ctypes.c_int32),
                ("tiles", ctypes.c_int64), ("iters", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("raster_group", ctypes.c_int32), ("ctas_per_tile", ctypes.c_int32),
                ("whole_tiles", ctypes.c_int64), ("sk_tiles", ctypes.c_int64),
                ("sk_base", ctypes.c_int64), ("sk_extra", ctypes.c_int64)]


class DeviceCaps(ctypes.Structure):
    """sk_device_caps_t."""
    _fields_ = [("sm_count", ctypes.c_int32), ("cc_major", ctypes.c_int32),
                ("cc_minor", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32 * 3),
                ("max_pair_clusters", ctypes.c_int32 * 2), ("setup_error", ctypes.c_int32 * 5),
                ("fp8_ctas_per_sm", ctypes.c_int32 * 2), ("fp8_max_pair_clusters", ctypes.c_int32),
                ("fp8_setup_error", ctypes.c_int32 * 3)]


def library_path() -> str:
    return _build.LIB_PATH


def lib():
    """The loaded C library.  Raises if it has not been built."""
    global _handle
    with _lock:
        if _handle is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library not built ({path}); run __graft_entry__.build()")
            h = ctypes.CDLL(path)
            vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            h.sk_gemm_bf16.restype = i32
            h.sk_gemm_bf16.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i32, i32, vp]
            h.sk_gemm_bf16_ex.restype = i32
            h.sk_gemm_bf16_ex.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i32, i32,
                                          ctypes.POINTER(Options), vp]
            h.sk_gemm_mxfp4.restype = i32
            h.sk_gemm_mxfp4.argtypes = [vp, vp, vp, vp, vp, vp, i32, i64, i64, i64, i32, i32, vp]
            h.sk_gemm_mxfp4_ex.restype = i32
            h.sk_gemm_mxfp4_ex.argtypes = [vp, vp, vp, vp, vp, vp, i32, i64, i64, i64, i32, i32,
                                           ctypes.POINTER(Options), vp]
            h.sk_gemm_fp8.restype = i32
            h.sk_gemm_fp8.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i32, i32, vp]
            h.sk_gemm_fp8_ex.restype = i32
            h.sk_gemm_fp8_ex.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i32, i32,
                                         ctypes.POINTER(Options), vp]
            for name in ("sk_gemm_bf16_host", "sk_gemm_fp8_host"):
                getattr(h, name).restype = i32
                getattr(h, name).argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i32, i32,
                                             ctypes.POINTER(Options), vp]
            h.sk_gemm_mxfp4_host.restype = i32
            h.sk_gemm_mxfp4_host.argtypes = [vp, vp, vp, vp, vp, vp, i32, i64, i64, i64, i32, i32,
                                             ctypes.POINTER(Options), vp]
            h.sk_gemm_bf16_t.restype = i32
            h.sk_gemm_bf16_t.argtypes = [vp, i32, vp, i32, vp, vp, i32, i64, i64, i64, i32, i32,
                                         ctypes.POINTER(Options), vp]
            h.sk_addmm_backward_bf16.restype = i32
            h.sk_addmm_backward_bf16.argtypes = [vp, vp, vp, vp, vp, vp, i32, i64, i64, i64, i32,
                                                 i32, vp]
            h.sk_gemm_bf16_static.restype = i32
            h.sk_gemm_bf16_static.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i32, i32, vp]
            h.sk_gemm_bf16_static_status.restype = i32
            h.sk_gemm_bf16_static_status.argtypes = [vp]
            h.sk_stream_status.restype = i32
            h.sk_stream_status.argtypes = [vp]
            h.sk_workspace_reserve.restype = i32
            h.sk_workspace_reserve.argtypes = [i32, vp, i32, i64, i64, i64]
            h.sk_workspace_release.restype = i32
            h.sk_workspace_release.argtypes = [i32, vp]
            h.sk_workspace_bytes.restype = i64
            h.sk_workspace_bytes.argtypes = [i32, vp]
            h.sk_workspace_release_all.restype = None
            h.sk_workspace_release_all.argtypes = []
            h.sk_status_string.restype = ctypes.c_char_p
            h.sk_status_string.argtypes = [i32]
            h.sk_plan.restype = i32
            h.sk_plan.argtypes = [i32, i64, i64, i64, i32, i32, i32, ctypes.POINTER(Options),
                                  ctypes.POINTER(Plan)]
            h.sk_autotune.restype = i32
            h.sk_autotune.argtypes = [i32, vp, vp, vp, vp, vp, vp, i32, i64, i64, i64, i32, i32,
                                      ctypes.POINTER(Plan), ctypes.POINTER(ctypes.c_float), vp]
            h.sk_device_caps.restype = i32
            h.sk_device_caps.argtypes = [i32, ctypes.POINTER(DeviceCaps)]
            h.sk_plan_segments.restype = i64
            h.sk_plan_segments.argtypes = [ctypes.POINTER(Plan), vp, i64]
            _handle = h
    return _handle


def _opts(options):
    if options is None:
        return None
    if isinstance(options, Options):
        return ctypes.byref(options)
    o = Options()
    o.drop_release_cta = -1
    for k, v in dict(options).items():
        setattr(o, k, v)
    return ctypes.byref(o)


# ---- the C entry points, by name (raw pointers and sizes) -------------------------------

def sk_gemm_bf16(A, B, bias, C, out_dtype, M, N, K, num_sms, mode, stream):
    return lib().sk_gemm_bf16(A, B, bias, C, out_dtype, M, N, K, num_sms, mode, stream)


def sk_gemm_bf16_ex(A, B, bias, C, out_dtype, M, N, K, num_sms, mode, options, stream):
    return lib().sk_gemm_bf16_ex(A, B, bias, C, out_dtype, M, N, K, num_sms, mode,
                                 _opts(options), stream)


def sk_gemm_mxfp4(A, A_scale, B, B_scale, bias, C, out_dtype, M, N, K, num_sms, mode, stream):
    return lib().sk_gemm_mxfp4(A, A_scale, B, B_scale, bias, C, out_dtype, M, N, K, num_sms,
                               mode, stream)


def sk_gemm_mxfp4_ex(A, A_scale, B, B_scale, bias, C, out_dtype, M, N, K, num_sms, mode,
                     options, stream):
    return lib().sk_gemm_mxfp4_ex(A, A_scale, B, B_scale, bias, C, out_dtype, M, N, K, num_sms,
                                  mode, _opts(options), stream)


def sk_gemm_fp8(A, B, bias, C, out_dtype, M, N, K, num_sms, mode, stream):
    return lib().sk_gemm_fp8(A, B, bias, C, out_dtype, M, N, K, num_sms, mode, stream)


def sk_gemm_fp8_ex(A, B, bias, C, out_dtype, M, N, K, num_sms, mode, options, stream):
    return lib().sk_gemm_fp8_ex(A, B, bias, C, out_dtype, M, N, K, num_sms, mode,
                                _opts(options), stream)


def sk_gemm_bf16_host(A, B, bias, C, out_dtype, M, N, K, num_sms, mode, options, stream):
    return lib().sk_gemm_bf16_host(A, B, bias, C, out_dtype, M, N, K, num_sms, mode,
                                   _opts(options), stream)


def sk_gemm_fp8_host(A, B, bias, C, out_dtype, M, N, K, num_sms, mode, options, stream):
    return lib().sk_gemm_fp8_host(A, B, bias, C, out_dtype, M, N, K, num_sms, mode,
                                  _opts(options), stream)


def sk_gemm_mxfp4_host(A, A_scale, B, B_scale, bias, C, out_dtype, M, N, K, num_sms, mode,
                       options, stream):
    return lib().sk_gemm_mxfp4_host(A, A_scale, B, B_scale, bias, C, out_dtype, M, N, K, num_sms,
                                    mode, _opts(options), stream)


def sk_gemm_bf16_t(A, trans_a, B, trans_b, bias, C, out_dtype, M, N, K, num_sms, mode, options,
                   stream):
    return lib().sk_gemm_bf16_t(A, trans_a, B, trans_b, bias, C, out_dtype, M, N, K, num_sms,
                                mode, _opts(options), stream)


def sk_addmm_backward_bf16(dC, A, B, dA, dB, dbias, grad_dtype, M, N, K, num_sms, mode, stream):
    return lib().sk_addmm_backward_bf16(dC, A, B, dA, dB, dbias, grad_dtype, M, N, K, num_sms,
                                        mode, stream)


def sk_gemm_bf16_static(A, B, bias, C, out_dtype, M, N, K, num_sms, mode, stream):
    """The bf16 addmm that allocates nothing (scratch in a fixed array inside the library),
    for callers that may not allocate device memory; calls must not overlap on the GPU."""
    return lib().sk_gemm_bf16_static(A, B, bias, C, out_dtype, M, N, K, num_sms, mode, stream)


def sk_gemm_bf16_static_status(stream):
    """Waits for `stream` and returns the error the last sk_gemm_bf16_static call recorded."""
    return lib().sk_gemm_bf16_static_status(stream)


def sk_stream_status(stream):
    return lib().sk_stream_status(stream)


def sk_workspace_reserve(device, stream, max_grid, max_mx_m=0, max_mx_n=0, max_mx_k=0):
    return lib().sk_workspace_reserve(device, stream, max_grid, max_mx_m, max_mx_n, max_mx_k)


def sk_workspace_release(device, stream):
    return lib().sk_workspace_release(device, stream)


def sk_workspace_bytes(device, stream):
    return lib().sk_workspace_bytes(device, stream)


def sk_workspace_release_all():
    lib().sk_workspace_release_all()


def sk_status_string(status):
    return lib().sk_status_string(status).decode()


def sk_device_caps(device=0):
    """dict of the device's SM count, compute capability and per-variant capacities."""
    c = DeviceCaps()
    st = lib().sk_device_caps(device, ctypes.byref(c))
    if st != SK_OK:
        raise SkError(st, "sk_device_caps")
    return {"sm_count": c.sm_count, "cc": (c.cc_major, c.cc_minor),
            "ctas_per_sm": list(c.ctas_per_sm), "max_pair_clusters": list(c.max_pair_clusters),
            "setup_error": list(c.setup_error), "fp8_ctas_per_sm": list(c.fp8_ctas_per_sm),
            "fp8_max_pair_clusters": c.fp8_max_pair_clusters,
            "fp8_setup_error": list(c.fp8_setup_error)}


def sk_plan(fmt, M, N, K, num_sms, mode, sm_count, options=None):
    p = Plan()
    st = lib().sk_plan(fmt, M, N, K, num_sms, _mode(mode), sm_count, _opts(options),
                       ctypes.byref(p))
    if st != SK_OK:
        raise SkError(st, "sk_plan")
    return p


def sk_plan_segments(plan):
    """(n, 7) int64 numpy array: cta, linear tile, k_begin, k_end, role, tile row, tile col."""
    import numpy as np
    n = lib().sk_plan_segments(ctypes.byref(plan), None, 0)
    if n < 0:
        raise SkError(SK_ERR_INVALID_ARG, "sk_plan_segments")
    rows = np.zeros((max(n, 1), 7), dtype=np.int64)
    lib().sk_plan_segments(ctypes.byref(plan), rows.ctypes.data_as(ctypes.c_void_p), n)
    return rows[:n]


# ---- torch helpers (marshalling only) ---------------------------------------------------

def _mode(mode):
    return MODES[mode] if isinstance(mode, str) else int(mode)


def _check(st, where):
    if st != SK_OK:
        raise SkError(st, where)


def _stream_ptr(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def gemm_bf16(a, b, bias=None, out=None, out_dtype=None, num_sms=0, mode="streamk",
              options=None, stream=None):
    """C = a @ b (+ bias) for bf16 CUDA tensors a (M,K), b (K,N); returns C (bf16 or fp32)."""
    import torch
    M, K = a.shape
    N = b.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or torch.bfloat16, device=a.device)
    for t in (a, b, out) + ((bias,) if bias is not None else ()):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")
    if a.dtype != torch.bfloat16 or b.dtype != torch.bfloat16:
        raise TypeError("a and b must be bf16")
    od = SK_BF16 if out.dtype == torch.bfloat16 else SK_F32
    if bias is not None and bias.dtype != out.dtype:
        raise TypeError("bias must have the output dtype")
    st = sk_gemm_bf16_ex(a.data_ptr(), b.data_ptr(), bias.data_ptr() if bias is not None else None,
                         out.data_ptr(), od, M, N, K, num_sms, _mode(mode), options,
                         _stream_ptr(stream))
    _check(st, "sk_gemm_bf16")
    return out


def gemm_mxfp4(a, a_scale, b, b_scale, bias=None, out=None, out_dtype=None, num_sms=0,
               mode="streamk", options=None, stream=None):
    """C = dec(a) @ dec(b)^T (+ bias) for MXFP4 uint8 CUDA tensors a (M,K/2), b (N,K/2) with
    E8M0 scales a_scale (M,K/32), b_scale (N,K/32)."""
    import torch
    M, K = a.shape[0], a.shape[1] * 2
    N = b.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or torch.bfloat16, device=a.device)
    for t in (a, a_scale, b, b_scale, out) + ((bias,) if bias is not None else ()):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")
    od = SK_BF16 if out.dtype == torch.bfloat16 else SK_F32
    if bias is not None and bias.dtype != out.dtype:
        raise TypeError("bias must have the output dtype")
    st = sk_gemm_mxfp4_ex(a.data_ptr(), a_scale.data_ptr(), b.data_ptr(), b_scale.data_ptr(),
                          bias.data_ptr() if bias is not None else None, out.data_ptr(), od,
                          M, N, K, num_sms, _mode(mode), options, _stream_ptr(stream))
    _check(st, "sk_gemm_mxfp4")
    return out


def gemm_fp8(a, b, bias=None, out=None, out_dtype=None, num_sms=0, mode="streamk",
             options=None, stream=None):
    """C = a @ b (+ bias) for E4M3 CUDA tensors a (M,K), b (K,N), given as float8_e4m3fn or as
    uint8 codes; returns C (bf16 or fp32)."""
    import torch
    M, K = a.shape
    N = b.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or torch.bfloat16, device=a.device)
    for t in (a, b, out) + ((bias,) if bias is not None else ()):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")
    ok = (torch.uint8, torch.float8_e4m3fn)
    if a.dtype not in ok or b.dtype not in ok:
        raise TypeError("a and b must be float8_e4m3fn (or uint8 codes)")
    od = SK_BF16 if out.dtype == torch.bfloat16 else SK_F32
    if bias is not None and bias.dtype != out.dtype:
        raise TypeError("bias must have the output dtype")
    st = sk_gemm_fp8_ex(a.data_ptr(), b.data_ptr(), bias.data_ptr() if bias is not None else None,
                        out.data_ptr(), od, M, N, K, num_sms, _mode(mode), options,
                        _stream_ptr(stream))
    _check(st, "sk_gemm_fp8")
    return out


def gemm_host(fmt, a, b, bias=None, out=None, out_dtype=None, a_scale=None, b_scale=None,
              num_sms=0, mode="streamk", options=None, stream=None):
    """The addmm on host (CPU) tensors, ideally pinned: fmt "bf16" (a (M,K), b (K,N) bf16),
    "fp8" (a (M,K), b (K,N) float8_e4m3fn or uint8 codes) or "mxfp4" (a (M,K/2), b (N,K/2)
    uint8 codes with E8M0 scales).  Copies in, computes and copies out on the given (or current)
    CUDA stream; synchronises that stream before returning C."""
    import torch
    tensors = [a, b] + [t for t in (bias, out, a_scale, b_scale) if t is not None]
    for t in tensors:
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous host tensors")
    if fmt == "mxfp4":
        M, K, N = a.shape[0], a.shape[1] * 2, b.shape[0]
    else:
        (M, K), N = a.shape, b.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or torch.bfloat16, pin_memory=True)
    od = SK_BF16 if out.dtype == torch.bfloat16 else SK_F32
    if bias is not None and bias.dtype != out.dtype:
        raise TypeError("bias must have the output dtype")
    bp = bias.data_ptr() if bias is not None else None
    s = torch.cuda.current_stream() if stream is None else stream
    if fmt == "bf16":
        st = sk_gemm_bf16_host(a.data_ptr(), b.data_ptr(), bp, out.data_ptr(), od, M, N, K,
                               num_sms, _mode(mode), options, s.cuda_stream)
    elif fmt == "fp8":
        st = sk_gemm_fp8_host(a.data_ptr(), b.data_ptr(), bp, out.data_ptr(), od, M, N, K,
                              num_sms, _mode(mode), options, s.cuda_stream)
    elif fmt == "mxfp4":
        st = sk_gemm_mxfp4_host(a.data_ptr(), a_scale.data_ptr(), b.data_ptr(),
                                b_scale.data_ptr(), bp, out.data_ptr(), od, M, N, K, num_sms,
                                _mode(mode), options, s.cuda_stream)
    else:
        raise ValueError(fmt)
    _check(st, f"sk_gemm_{fmt}_host")
    s.synchronize()
    return out


def gemm_bf16_t(a, b, trans_a=False, trans_b=False, bias=None, out=None, out_dtype=None,
                num_sms=0, mode="streamk", options=None, stream=None):
    """op(a) @ op(b) (+ bias): a is (M,K), or (K,M) stored when trans_a; b is (K,N), or (N,K)
    stored when trans_b.  bf16 CUDA tensors."""
    import torch
    M, K = (a.shape[1], a.shape[0]) if trans_a else a.shape
    N = b.shape[0] if trans_b else b.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or torch.bfloat16, device=a.device)
    for t in (a, b, out) + ((bias,) if bias is not None else ()):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")
    od = SK_BF16 if out.dtype == torch.bfloat16 else SK_F32
    st = sk_gemm_bf16_t(a.data_ptr(), int(bool(trans_a)), b.data_ptr(), int(bool(trans_b)),
                        bias.data_ptr() if bias is not None else None, out.data_ptr(), od, M, N,
                        K, num_sms, _mode(mode), options, _stream_ptr(stream))
    _check(st, "sk_gemm_bf16_t")
    return out


def addmm_backward(dc, a, b, need=("a", "b", "bias"), grad_dtype=None, num_sms=0,
                   mode="streamk", stream=None):
    """(da, db, dbias) of c = a @ b + bias for bf16 CUDA tensors; entries not in `need` are
    None."""
    import torch
    M, K = a.shape
    N = b.shape[1]
    dt = grad_dtype or torch.bfloat16
    da = torch.empty((M, K), dtype=dt, device=dc.device) if "a" in need else None
    db = torch.empty((K, N), dtype=dt, device=dc.device) if "b" in need else None
    dbias = torch.empty((N,), dtype=dt, device=dc.device) if "bias" in need else None
    ptr = lambda t: t.data_ptr() if t is not None else None
    st = sk_addmm_backward_bf16(dc.data_ptr(), a.data_ptr(), b.data_ptr(), ptr(da), ptr(db),
                                ptr(dbias), SK_BF16 if dt == torch.bfloat16 else SK_F32, M, N, K,
                                num_sms, _mode(mode), _stream_ptr(stream))
    _check(st, "sk_addmm_backward_bf16")
    return da, db, dbias


def autotune(fmt, a, b, bias=None, out=None, out_dtype=None, a_scale=None, b_scale=None,
             num_sms=0, reps=5, stream=None):
    """Measure every schedule x tile candidate for this problem on the GPU and keep the fastest
    for later mode="auto" calls.  CUDA tensors as for gemm_bf16 / gemm_fp8 / gemm_mxfp4.
    Returns (plan, ms per call)."""
    import torch
    if fmt == "mxfp4":
        M, K, N = a.shape[0], a.shape[1] * 2, b.shape[0]
    else:
        (M, K), N = a.shape, b.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or torch.bfloat16, device=a.device)
    od = SK_BF16 if out.dtype == torch.bfloat16 else SK_F32
    ptr = lambda t: t.data_ptr() if t is not None else None
    plan, ms = Plan(), ctypes.c_float()
    st = lib().sk_autotune({"bf16": 0, "mxfp4": 1, "fp8": 2}[fmt], a.data_ptr(), ptr(a_scale),
                           b.data_ptr(), ptr(b_scale), ptr(bias), out.data_ptr(), od, M, N, K,
                           num_sms, reps, ctypes.byref(plan), ctypes.byref(ms),
                           _stream_ptr(stream))
    _check(st, "sk_autotune")
    return plan, ms.value


def stream_status(stream=None):
    """Synchronise the stream and raise if a kernel recorded an error (e.g. a timeout)."""
    _check(sk_stream_status(_stream_ptr(stream)), "sk_stream_status")
