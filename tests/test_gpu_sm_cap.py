"""An SM-constrained call runs on at most num_sms SMs.

The cap is the point of the SM-constrained persistent GEMM (flashinfer PR #982
"SM-constraint-GEMM by triton persistent kernel": its checklist verifies the SMs a capped call
occupies with an nsys profile, and its nsys block shows a request of 133 SMs launched as 132
CTAs).  Here every CTA writes the index of its SM (%smid) into the options' SM-usage record;
the distinct SMs of a persistent, Stream-K or hybrid call must number no more than num_sms
(an SM pair counts both its SMs), one CTA per SM, alone and while a copy kernel runs on
another stream.  Each call's result is also checked against the oracle."""
import functools

import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
import sm_constrained_persistent_gb300 as sk
from sm_constrained_persistent_gb300 import inputs

pytestmark = pytest.mark.gpu

M, N, K = 2304, 2304, 512   # 324 tiles of 128 x 128 and 81 pair tiles: more than any grid here
TILES = {"one_cta": {"tile_m": 128, "tile_n": 128}, "pair": {"tile_m": 256}}


@functools.lru_cache(maxsize=1)
def _problem():
    p = inputs.bf16_problem(M, N, K, seed=4242, operand_scale="sqrt_k", bias="f32_normal")
    ref = gu.reference(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), "f32")
    return p, ref


def _sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _capped_call(mode, num_sms, tile, stream=None):
    """Runs the call with an SM-usage record; returns (C, SMs recorded, CTAs launched)."""
    p, _ = _problem()
    opts = dict(TILES[tile])
    plan = sk.sk_plan(0, M, N, K, num_sms, mode, _sm_count(), opts)
    ctas = plan.grid * plan.ctas_per_tile
    record = torch.full((ctas + 8,), -1, dtype=torch.int32, device="cuda")   # 8 spare entries
    opts.update(sm_record=record.data_ptr(), sm_record_len=ctas)
    a, b, bias = gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"]), gu.dev_bias(p["bias"])
    c = sk.gemm_bf16(a, b, bias, out_dtype=torch.float32, num_sms=num_sms, mode=mode,
                     options=opts, stream=stream)
    return c, record, ctas


def _check_record(record, ctas, num_sms, what):
    r = record.cpu().numpy()
    assert (r[:ctas] >= 0).all(), f"{what}: a CTA did not record its SM"
    assert (r[ctas:] == -1).all(), f"{what}: a store beyond the launched CTAs"
    used = np.unique(r[:ctas])
    assert (used < _sm_count()).all()
    assert len(used) == ctas, f"{what}: {ctas} CTAs on {len(used)} SMs (one CTA per SM expected)"
    assert len(used) <= num_sms, f"{what}: {len(used)} SMs used for num_sms = {num_sms}"
    return len(used)


@pytest.mark.parametrize("tile", list(TILES))
@pytest.mark.parametrize("mode", ["persistent", "streamk", "hybrid"])
@pytest.mark.parametrize("num_sms", [1, 16, 64, 76, 151])
def test_capped_call_runs_on_at_most_num_sms_sms(cuda_device, tile, mode, num_sms):
    if tile == "pair" and num_sms < 2:
        pytest.skip("a pair tile needs two SMs")
    c, record, ctas = _capped_call(mode, num_sms, tile)
    sk.stream_status()
    used = _check_record(record, ctas, num_sms, f"{mode}/{tile}/{num_sms}")
    if tile == "pair":
        assert used == 2 * min(num_sms // 2, ctas // 2)
    _, ref = _problem()
    gu.assert_close(gu.host_values(c), ref, "f32", f"{mode}/{tile}/{num_sms}")


def test_request_above_the_sm_count_is_capped_to_it(cuda_device):
    """As in the pages' nsys block (133 requested on a 132-SM part, 132 CTAs launched)."""
    S = _sm_count()
    c, record, ctas = _capped_call("persistent", S + 1, "one_cta")
    sk.stream_status()
    assert ctas == S
    assert _check_record(record, ctas, S, "persistent/S+1") == S


@pytest.mark.parametrize("mode", ["persistent", "streamk"])
@pytest.mark.parametrize("tile", list(TILES))
def test_cap_holds_beside_a_copy_kernel(cuda_device, mode, tile):
    """The GEMM capped at 64 SMs on one stream while 256 MiB copies run on another."""
    src = torch.ones((256 << 20) // 4, dtype=torch.float32, device="cuda")
    dst = torch.empty_like(src)
    s_copy, s_gemm = torch.cuda.Stream(), torch.cuda.Stream()
    _problem()
    torch.cuda.synchronize()
    with torch.cuda.stream(s_copy):
        for _ in range(20):
            dst.copy_(src)
    c, record, ctas = _capped_call(mode, 64, tile, stream=s_gemm)
    torch.cuda.synchronize()
    assert sk.sk_stream_status(s_gemm.cuda_stream) == sk.SK_OK
    _check_record(record, ctas, 64, f"co-run {mode}/{tile}")
    _, ref = _problem()
    gu.assert_close(gu.host_values(c), ref, "f32", f"co-run {mode}/{tile}")


def test_record_shorter_than_the_launch_is_refused(cuda_device):
    p, _ = _problem()
    plan = sk.sk_plan(0, M, N, K, 16, "streamk", _sm_count(), TILES["one_cta"])
    record = torch.full((64,), -1, dtype=torch.int32, device="cuda")
    c = torch.empty((M, N), dtype=torch.float32, device="cuda")
    a, b = gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"])
    opts = dict(TILES["one_cta"], sm_record=record.data_ptr(), sm_record_len=plan.grid - 1)
    st = sk.sk_gemm_bf16_ex(a.data_ptr(), b.data_ptr(), None, c.data_ptr(), sk.SK_F32, M, N, K, 16,
                            sk.MODES["streamk"], opts, torch.cuda.current_stream().cuda_stream)
    assert st == sk.SK_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (record.cpu().numpy() == -1).all()
