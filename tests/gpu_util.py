"""Helpers shared by the GPU parity tests: move seeded numpy inputs to the device, run the
library through its binding, and compare with the oracle at the stated tolerances."""
import numpy as np
import torch

import oracle
import sm_constrained_persistent_gb300 as sk

# Tolerances (addmm parity bar): bf16 output |C - ref| <= 1e-2 + 1e-2 |ref|;
# fp32 output |C - ref| <= 1e-3 (1 + |ref|); exact-integer inputs: bit-exact.
BF16_ATOL, BF16_RTOL = 1e-2, 1e-2
F32_TOL = 1e-3


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev_u8(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def dev_bias(b):
    if b is None:
        return None
    if b.dtype == np.float32:
        return torch.from_numpy(b).cuda()
    return dev_bf16(b)


def out_torch_dtype(p_or_name):
    return torch.bfloat16 if p_or_name == "bf16" else torch.float32


def host_values(c):
    """Device result -> float64 numpy (exact)."""
    return c.float().cpu().numpy().astype(np.float64)


def host_bits(c):
    if c.dtype == torch.bfloat16:
        return c.cpu().view(torch.int16).numpy().view(np.uint16)
    return c.cpu().numpy().view(np.uint32)


def run_bf16(p, out="bf16", mode="streamk", num_sms=0, options=None, stream=None):
    a, b = dev_bf16(p["A"]), dev_bf16(p["B"])
    bias = dev_bias(p["bias"])
    c = sk.gemm_bf16(a, b, bias, out_dtype=out_torch_dtype(out), num_sms=num_sms, mode=mode,
                     options=options, stream=stream)
    sk.stream_status(stream)
    return c


def run_mxfp4(p, out="bf16", mode="streamk", num_sms=0, options=None, stream=None):
    c = sk.gemm_mxfp4(dev_u8(p["A"]), dev_u8(p["A_scale"]), dev_u8(p["B"]), dev_u8(p["B_scale"]),
                      dev_bias(p["bias"]), out_dtype=out_torch_dtype(out), num_sms=num_sms,
                      mode=mode, options=options, stream=stream)
    sk.stream_status(stream)
    return c


def reference(ref64, out):
    """Oracle result rounded to the output dtype, as float64 values."""
    r = oracle.round_output(ref64, oracle.BF16 if out == "bf16" else oracle.F32)
    if out == "bf16":
        return (r.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return r.astype(np.float64)


def assert_close(got, ref, out, what=""):
    """Element-wise check at the parity tolerance; reports the worst element."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    if out == "bf16":
        bound = BF16_ATOL + BF16_RTOL * np.abs(ref)
    else:
        bound = F32_TOL * (1.0 + np.abs(ref))
    err = np.abs(got - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), got.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {idx}: "
                             f"got {got[idx]!r} ref {ref[idx]!r}")


def sample_positions(M, N, n_random=2048, n_rows=4, n_cols=4, seed=0):
    """Random elements plus whole rows and columns (first, last and random ones)."""
    rng = np.random.default_rng(seed)
    ms = [rng.integers(0, M, n_random)]
    ns = [rng.integers(0, N, n_random)]
    rows = sorted(set([0, M - 1] + list(rng.integers(0, M, n_rows))))
    cols = sorted(set([0, N - 1] + list(rng.integers(0, N, n_cols))))
    for r in rows:
        ms.append(np.full(N, r))
        ns.append(np.arange(N))
    for c in cols:
        ms.append(np.arange(M))
        ns.append(np.full(M, c))
    return np.concatenate(ms).astype(np.int64), np.concatenate(ns).astype(np.int64)
