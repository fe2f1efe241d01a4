"""Failure paths of the C ABI, exercised without a GPU fault, and the per-stream workspace
release.

  * A Stream-K or hybrid grid the device could not hold at once is refused before anything is
    launched (SK_ERR_NOT_CORESIDENT); the device's room is stood in for by the options'
    resident_limit test control.
  * A workspace (Stream-K slots, MXFP4 scale scratch, host-buffer staging) that cannot grow
    because device memory is full reports SK_ERR_OOM, and the next call, once memory is free,
    runs and matches the oracle.  The pages note a crash around these scratch buffers (tritonBLAS
    PR #74 "Stream-k mxfp4 kernel", review comment on the scratch buffers); here the
    allocation failure is a status code.
  * sk_workspace_release frees one stream's workspace; a later call on that stream builds a
    new one."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
import sm_constrained_persistent_gb300 as sk
from sm_constrained_persistent_gb300 import inputs

pytestmark = pytest.mark.gpu


def _stream_ptr(s=None):
    return (s or torch.cuda.current_stream()).cuda_stream


# ---- co-residency refusal ------------------------------------------------------------------

@pytest.mark.parametrize("mode", ["streamk", "hybrid"])
@pytest.mark.parametrize("tile,num_sms,limit", [("one_cta", 16, 8), ("pair", 16, 4)])
def test_grid_above_the_resident_limit_is_refused_before_launch(cuda_device, mode, tile, num_sms,
                                                                 limit):
    # 81 tiles of 128 x 128 (25 pair tiles): a Stream-K region under both schedules
    M, N, K = 1152, 1152, 1024
    p = inputs.bf16_problem(M, N, K, seed=77, operand_scale="sqrt_k", bias="f32_normal")
    a, b, bias = gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"]), gu.dev_bias(p["bias"])
    opts = {"tile_m": 128, "tile_n": 128} if tile == "one_cta" else {"tile_m": 256}
    plan = sk.sk_plan(0, M, N, K, num_sms, mode, torch.cuda.get_device_properties(0).multi_processor_count,
                      opts)
    assert plan.sk_tiles > 0 and plan.grid > limit
    c = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    st = sk.sk_gemm_bf16_ex(a.data_ptr(), b.data_ptr(), bias.data_ptr(), c.data_ptr(), sk.SK_F32,
                            M, N, K, num_sms, sk.MODES[mode], dict(opts, resident_limit=limit),
                            _stream_ptr())
    assert st == sk.SK_ERR_NOT_CORESIDENT
    torch.cuda.synchronize()
    assert torch.isnan(c).all(), "a refused call wrote C"
    # a grid that fits under the limit, and the same call without the limit, both run
    ref = gu.reference(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), "f32")
    for ns, o in [(limit * (1 if tile == "one_cta" else 2), dict(opts, resident_limit=limit)),
                  (num_sms, opts)]:
        c = sk.gemm_bf16(a, b, bias, out_dtype=torch.float32, num_sms=ns, mode=mode, options=o)
        sk.stream_status()
        gu.assert_close(gu.host_values(c), ref, "f32", f"{mode}/{tile}/{ns}")


def test_persistent_and_dp_grids_need_no_coresidency(cuda_device):
    M, N, K = 1024, 1024, 512
    p = inputs.bf16_problem(M, N, K, seed=78, integer=True, bias="f32_int")
    a, b, bias = gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"]), gu.dev_bias(p["bias"])
    want = oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), oracle.F32)
    for mode in ("persistent", "dp"):
        c = sk.gemm_bf16(a, b, bias, out_dtype=torch.float32, num_sms=16, mode=mode,
                         options={"tile_m": 128, "tile_n": 128, "resident_limit": 1})
        sk.stream_status()
        assert np.array_equal(c.cpu().numpy(), want), mode


# ---- allocation failure --------------------------------------------------------------------

def _stream_without_workspace():
    """A stream the library holds no workspace for (torch hands out streams from a pool, so a
    new torch stream may be one an earlier test used)."""
    s = torch.cuda.Stream()
    assert sk.sk_workspace_release(0, s.cuda_stream) == sk.SK_OK
    torch.cuda.synchronize()
    assert sk.sk_workspace_bytes(0, s.cuda_stream) == 0
    return s


def _fill_device_memory(leave_bytes):
    """A tensor that takes all free device memory but about `leave_bytes`.  Every workspace the
    library holds is released first: workspaces grow through the stream-ordered allocator, whose
    pool keeps free space inside memory that stays mapped, and a later allocation could be served
    from there however full the device is."""
    sk.sk_workspace_release_all()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    n = free - leave_bytes
    for _ in range(64):
        try:
            return torch.empty(n, dtype=torch.uint8, device="cuda")
        except torch.OutOfMemoryError:
            n -= 32 << 20
    pytest.skip("could not fill device memory")


def test_device_workspace_that_cannot_grow_reports_oom_and_recovers(cuda_device):
    M, N, K = 2048, 2048, 4096
    p = inputs.mxfp4_problem(M, N, K, seed=91, exp_range=2)
    args = [gu.dev_u8(p[k]) for k in ("A", "A_scale", "B", "B_scale")]
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    # load the kernels and set them up first (on another stream), so the call below needs
    # device memory only for its own workspace
    sk.gemm_mxfp4(*args, None, out=c, mode="streamk")
    sk.stream_status()
    fresh = _stream_without_workspace()   # the call must grow ~19 MiB of Stream-K slots
    hog = _fill_device_memory(4 << 20)
    try:
        assert torch.cuda.mem_get_info()[0] < (16 << 20)
        c.fill_(float("nan"))
        torch.cuda.synchronize()
        st = sk.sk_gemm_mxfp4_ex(*(t.data_ptr() for t in args), None, c.data_ptr(), sk.SK_F32,
                                 M, N, K, 0, sk.MODES["streamk"], None, fresh.cuda_stream)
        assert st == sk.SK_ERR_OOM, sk.STATUS.get(st, st)
    finally:
        del hog
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    sk.gemm_mxfp4(*args, None, out=c, mode="streamk", stream=fresh)
    assert sk.sk_stream_status(fresh.cuda_stream) == sk.SK_OK
    torch.cuda.synchronize()
    ref = gu.reference(oracle.addmm_mxfp4(p["A"], p["A_scale"], p["B"], p["B_scale"], None), "f32")
    gu.assert_close(gu.host_values(c), ref, "f32", "MXFP4 Stream-K after OOM")
    assert sk.sk_workspace_release(0, fresh.cuda_stream) == sk.SK_OK


def test_host_buffer_staging_that_cannot_grow_reports_oom_and_recovers(cuda_device):
    M, N, K = 2048, 2048, 2048
    p = inputs.bf16_problem(M, N, K, seed=92, operand_scale="sqrt_k", bias="bf16_uniform")
    a = torch.from_numpy(p["A"].view(np.int16)).view(torch.bfloat16).pin_memory()
    b = torch.from_numpy(p["B"].view(np.int16)).view(torch.bfloat16).pin_memory()
    bias = torch.from_numpy(p["bias"].view(np.int16)).view(torch.bfloat16).pin_memory()
    out = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    sk.gemm_host("bf16", a, b, bias, out=out, mode="streamk")   # kernels loaded and set up
    fresh = _stream_without_workspace()
    hog = _fill_device_memory(4 << 20)
    try:
        st = sk.sk_gemm_bf16_host(a.data_ptr(), b.data_ptr(), bias.data_ptr(), out.data_ptr(),
                                   sk.SK_BF16, M, N, K, 0, sk.MODES["streamk"], None,
                                   fresh.cuda_stream)
        assert st == sk.SK_ERR_OOM, sk.STATUS.get(st, st)
        fresh.synchronize()
    finally:
        del hog
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    out.zero_()
    sk.gemm_host("bf16", a, b, bias, out=out, mode="streamk", stream=fresh)
    assert sk.sk_stream_status(fresh.cuda_stream) == sk.SK_OK
    ref = gu.reference(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), "bf16")
    gu.assert_close(out.float().numpy().astype(np.float64), ref, "bf16", "host call after OOM")
    assert sk.sk_workspace_release(0, fresh.cuda_stream) == sk.SK_OK


# ---- per-stream workspace release ----------------------------------------------------------

def test_workspace_release_frees_one_stream_and_a_later_call_rebuilds_it(cuda_device):
    M, N, K = 2048, 2048, 2048
    p = inputs.bf16_problem(M, N, K, seed=93, integer=True, bias="f32_int")
    a, b, bias = gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"]), gu.dev_bias(p["bias"])
    want = oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), oracle.F32)
    s = _stream_without_workspace()
    host = [torch.from_numpy(p[k].view(np.int16)).view(torch.bfloat16).pin_memory()
            for k in ("A", "B")]
    hout = torch.empty((M, N), dtype=torch.float32).pin_memory()
    c = sk.gemm_bf16(a, b, bias, out_dtype=torch.float32, mode="streamk", stream=s)
    sk.gemm_host("bf16", host[0], host[1], torch.from_numpy(p["bias"]).pin_memory(), out=hout,
                 mode="streamk", stream=s)
    assert sk.sk_stream_status(s.cuda_stream) == sk.SK_OK
    held = sk.sk_workspace_bytes(0, s.cuda_stream)
    # Stream-K slots of the SM pairs (~19 MiB) and the host staging (A, B, C: 8 + 8 + 16 MiB)
    assert held >= 40 << 20, f"only {held >> 20} MiB held"
    assert sk.sk_workspace_release(0, s.cuda_stream) == sk.SK_OK
    assert sk.sk_workspace_bytes(0, s.cuda_stream) == 0
    torch.cuda.synchronize()
    # The frees reach the device: the stream-ordered pool then hands out the same memory again
    # (the pool may keep the pages mapped, so free memory as the device reports it need not
    # grow by all of it).
    assert sk.sk_workspace_release(0, s.cuda_stream) == sk.SK_OK   # nothing left: not an error
    c.zero_()
    sk.gemm_bf16(a, b, bias, out=c, mode="streamk", stream=s)
    assert sk.sk_stream_status(s.cuda_stream) == sk.SK_OK
    assert np.array_equal(c.cpu().numpy(), want)
    hout.zero_()
    sk.gemm_host("bf16", host[0], host[1], torch.from_numpy(p["bias"]).pin_memory(), out=hout,
                 mode="streamk", stream=s)
    assert np.array_equal(hout.numpy(), want)
    assert sk.sk_workspace_bytes(0, s.cuda_stream) >= held
    assert sk.sk_workspace_release(0, s.cuda_stream) == sk.SK_OK
    assert sk.sk_workspace_bytes(0, s.cuda_stream) == 0


def test_workspace_release_checks_the_device_and_leaves_no_cuda_error(cuda_device):
    assert sk.sk_workspace_release(torch.cuda.device_count() + 7, None) == sk.SK_ERR_INVALID_ARG
    # the refused device change must not surface as the next CUDA call's error
    x = torch.zeros(16, device="cuda")
    x.add_(1.0)
    torch.cuda.synchronize()
    assert float(x.sum()) == 16.0


def test_workspace_release_is_refused_while_capturing(cuda_device):
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    st = None
    with torch.cuda.graph(g, stream=s):
        st = sk.sk_workspace_release(0, s.cuda_stream)
    assert st == sk.SK_ERR_UNSUPPORTED
