"""The entry point that allocates nothing (sk_gemm_bf16_static), for callers that may not
allocate device memory when they run the GEMM: its output must match the regular entry
point's on two calls in a row (the second call reuses the fixed scratch array the first one
left behind).  This file is collected last so that a failure here stops a -x run only after
every other test has run."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import sm_constrained_persistent_gb300 as sk
from sm_constrained_persistent_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode", ["streamk", "hybrid", "persistent", "dp"])
def test_static_scratch_entry_matches_allocating_entry_twice(cuda_device, mode):
    M, N, K = 1000, 1032, 2056
    p = inputs.bf16_problem(M, N, K, seed=2024, operand_scale="sqrt_k", bias="bf16_uniform")
    a, b, bias = gu.dev_bf16(p["A"]), gu.dev_bf16(p["B"]), gu.dev_bias(p["bias"])
    stream = torch.cuda.current_stream().cuda_stream
    want = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = sk.sk_gemm_bf16(a.data_ptr(), b.data_ptr(), bias.data_ptr(), want.data_ptr(), sk.SK_BF16,
                         M, N, K, 0, sk.MODES[mode], stream)
    assert st == sk.SK_OK
    assert sk.sk_stream_status(stream) == sk.SK_OK
    ref = gu.host_values(want)
    for call in range(2):
        got = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = sk.sk_gemm_bf16_static(a.data_ptr(), b.data_ptr(), bias.data_ptr(), got.data_ptr(),
                                    sk.SK_BF16, M, N, K, 0, sk.MODES[mode], stream)
        assert st == sk.SK_OK, sk.STATUS.get(st, st)
        torch.cuda.synchronize()
        gu.assert_close(gu.host_values(got), ref, "bf16", f"{mode} call {call}")


def test_static_scratch_entry_checks_arguments_like_the_regular_one(cuda_device):
    assert sk.sk_gemm_bf16_static(None, 16, None, 16, 1, 64, 64, 64, 0, 2, None) == sk.SK_ERR_INVALID_ARG
    assert sk.sk_gemm_bf16_static(16, 16, None, 16, 1, 64, 60, 64, 0, 2, None) == sk.SK_ERR_INVALID_ARG
