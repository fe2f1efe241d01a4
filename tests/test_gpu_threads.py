"""Concurrent callers: Python threads (ctypes releases the GIL inside each C call) drive the
library on their own streams at once -- device calls, host-buffer calls and the automatic
mode -- while the library creates and grows per-stream workspaces.  Every result must equal
the oracle's bit for bit (exact-integer inputs)."""
import threading

import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
import sm_constrained_persistent_gb300 as sk
from sm_constrained_persistent_gb300 import inputs

pytestmark = pytest.mark.gpu


def test_threads_on_separate_streams_get_exact_results(cuda_device):
    shapes = [(512, 384, 1024), (1000, 264, 640), (256, 1024, 2048), (768, 768, 512)]
    probs = [inputs.bf16_problem(M, N, K, seed=i, integer=True, bias="f32_int")
             for i, (M, N, K) in enumerate(shapes)]
    wants = [oracle.round_output(oracle.addmm_bf16(p["A"], p["B"], p["bias"]), oracle.F32)
             .view(np.uint32) for p in probs]
    errors = []

    def worker(t):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            p, want = probs[t % len(probs)], wants[t % len(probs)]
            a, b, bias = gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"]), gu.dev_bias(p["bias"])
            for i in range(12):
                mode = ["dp", "persistent", "streamk", "hybrid", "auto"][(t + i) % 5]
                with torch.cuda.stream(s):
                    if i % 4 == 3:   # the host-buffer path now and then
                        c = sk.gemm_host("bf16", a.cpu(), b.cpu(), bias.cpu(),
                                         out_dtype=torch.float32, mode=mode, stream=s)
                    else:
                        c = sk.gemm_bf16(a, b, bias, out_dtype=torch.float32, mode=mode,
                                         num_sms=[0, 7, 64][i % 3], stream=s)
                        sk.stream_status(s)
                got = gu.host_bits(c)
                if not np.array_equal(got, want):
                    errors.append((t, i, mode))
        except Exception as e:      # reported below, on the main thread
            errors.append((t, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(6)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
