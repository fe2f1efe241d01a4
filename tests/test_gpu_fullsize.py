"""Full-output parity at the benchmark's full sizes: every element of C, for every workload the
benchmark names, against the oracle computed once per workload on all host threads.

Workloads (the seeded synthetic inputs of the benchmark): the bf16, MXFP4 and fp8 8192^3 addmm
(bf16 bias, bf16 output), the wave-quantised 1920 x 1920 x 16384 GEMM (with its stated
128 x 128 tiles and with the library's own tiles), the SM-constrained persistent sweep over
num_sms in {1, 16, 32, 64, 128, all} on 4096^3 and on the skinny 64 x 14336 x 4096, and the
few-tile, long-K 1024 x 1024 x 16384 GEMM whose split tiles several SM pairs finish together.  Each case
compares all M x N outputs at the parity tolerance (bf16 output: |C - ref| <= 1e-2 + 1e-2 |ref|)
and reports its worst element relative to the bound in the test summary."""
import functools

import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
import sm_constrained_persistent_gb300 as sk
from sm_constrained_persistent_gb300 import inputs

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=1)
def _workload(name):
    """Inputs on the device and the oracle's full result (rounded to bf16), one workload at a
    time (the cache holds one: the 8192^3 references are 512 MiB each)."""
    p = inputs.workload(name)
    if p["format"] == "bf16":
        ref64 = oracle.addmm_bf16(p["A"], p["B"], p["bias"])
        dev = {"A": gu.dev_bf16(p["A"]), "B": gu.dev_bf16(p["B"])}
    elif p["format"] == "fp8":
        ref64 = oracle.addmm_fp8(p["A"], p["B"], p["bias"])
        dev = {"A": gu.dev_u8(p["A"]), "B": gu.dev_u8(p["B"])}
    else:
        ref64 = oracle.addmm_mxfp4(p["A"], p["A_scale"], p["B"], p["B_scale"], p["bias"])
        dev = {k: gu.dev_u8(p[k]) for k in ("A", "A_scale", "B", "B_scale")}
    dev["bias"] = gu.dev_bias(p["bias"])
    ref = gu.reference(ref64, p["out_dtype"])
    del ref64
    return p, dev, ref


def _run(p, dev, mode, num_sms=0, options=None):
    kw = dict(out_dtype=gu.out_torch_dtype(p["out_dtype"]), num_sms=num_sms, mode=mode,
              options=options)
    if p["format"] == "bf16":
        c = sk.gemm_bf16(dev["A"], dev["B"], dev["bias"], **kw)
    elif p["format"] == "fp8":
        c = sk.gemm_fp8(dev["A"], dev["B"], dev["bias"], **kw)
    else:
        c = sk.gemm_mxfp4(dev["A"], dev["A_scale"], dev["B"], dev["B_scale"], dev["bias"], **kw)
    sk.stream_status()
    return c


def _check_all(name, what, mode, parity_report, num_sms=0, options=None):
    p, dev, ref = _workload(name)
    c = _run(p, dev, mode, num_sms, options)
    got = gu.host_values(c)
    del c
    bound = gu.BF16_ATOL + gu.BF16_RTOL * np.abs(ref)
    ratio = np.abs(got - ref) / bound
    worst = np.unravel_index(int(np.argmax(ratio)), ratio.shape)
    parity_report.append(f"{what}: all {ref.size} elements, worst |C-ref|/bound "
                         f"{ratio[worst]:.3f} at {tuple(int(i) for i in worst)}")
    gu.assert_close(got, ref, p["out_dtype"], what)


# the three 8192^3 addmm workloads (kept adjacent so each oracle result is computed once)
@pytest.mark.parametrize("name,mode", [(n, m) for n in ("addmm_bf16_8192", "addmm_mxfp4_8192",
                                                        "addmm_fp8_8192")
                                       for m in ("streamk", "dp", "persistent", "hybrid")])
def test_addmm_8192_every_element(cuda_device, parity_report, name, mode):
    _check_all(name, f"{name}/{mode}", mode, parity_report)


@pytest.mark.parametrize("tiles", ["tile128", "auto"])
@pytest.mark.parametrize("mode", ["streamk", "dp", "persistent", "hybrid"])
def test_wave_quantised_1920_every_element(cuda_device, parity_report, tiles, mode):
    opts = {"tile_m": 128, "tile_n": 128} if tiles == "tile128" else None
    _check_all("gemm_bf16_1920x1920x16384", f"1920x1920x16384/{tiles}/{mode}", mode,
               parity_report, options=opts)


@pytest.mark.parametrize("num_sms", [1, 16, 32, 64, 128, 0])
@pytest.mark.parametrize("name", ["gemm_bf16_4096", "gemm_bf16_skinny_64x14336x4096"])
def test_num_sms_sweep_every_element(cuda_device, parity_report, name, num_sms):
    _check_all(name, f"{name}/persistent/num_sms={num_sms or 'all'}", "persistent", parity_report,
               num_sms=num_sms)


@pytest.mark.parametrize("name", ["gemm_bf16_4096", "gemm_bf16_skinny_64x14336x4096"])
def test_sweep_shapes_streamk_every_element(cuda_device, parity_report, name):
    _check_all(name, f"{name}/streamk", "streamk", parity_report)


@pytest.mark.parametrize("mode", ["streamk", "hybrid", "dp"])
def test_few_tiles_long_k_1024_every_element(cuda_device, parity_report, mode):
    # 16 pair tiles on 76 pairs: ~5 pairs per tile, four of which finish it with its owner
    _check_all("gemm_bf16_1024x1024x16384", f"1024x1024x16384/{mode}", mode, parity_report)
