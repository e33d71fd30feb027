"""Failure detection on the GPU without a fault: a bounded wait on a barrier
that nothing arrives at must end with MOE_ERR_TIMEOUT in the error word, and
the context must stay usable afterwards."""
import time

import pytest
import torch

import mixture_experts_ffn_softmax_gb300 as pkg

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    pkg.selftest_wait_timeout(err, limit_us=20000)
    assert pkg.read_error(err.data_ptr()) == 5          # MOE_ERR_TIMEOUT
    assert time.time() - t0 < 10
    # the context still works: a small forward runs and reports no error
    M, H, I, E, k = 8, 64, 64, 2, 1
    x = torch.ones(M, H, device="cuda").bfloat16()
    w13 = torch.zeros(E, H, 2 * I, device="cuda").bfloat16()
    w2 = torch.zeros(E, I, H, device="cuda").bfloat16()
    ws = pkg.alloc_workspace(pkg.workspace_size(M, H, I, E, k))
    y = pkg.moe_forward(x, torch.ones(M, k, device="cuda"),
                        torch.zeros(M, k, dtype=torch.int32, device="cuda"), w13, w2,
                        workspace=ws)
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 0
    assert (y.float() == 0).all()


@pytest.mark.parametrize("gather", ["separate", "fused"])
def test_profiler_counts_launches(gather):
    M, H, I, E, k = 32, 64, 64, 2, 1
    x = torch.ones(M, H, device="cuda").bfloat16()
    w13 = torch.zeros(E, H, 2 * I, device="cuda").bfloat16()
    w2 = torch.zeros(E, I, H, device="cuda").bfloat16()
    pkg.set_gather_mode(gather)
    pkg.set_small_path(False)   # the general path's launches
    try:
        n0 = pkg.launch_count()
        pkg.profiler_start()
        pkg.moe_forward(x, torch.ones(M, k, device="cuda"),
                        torch.zeros(M, k, dtype=torch.int32, device="cuda"), w13, w2)
        prof = pkg.profiler_stop()
    finally:
        pkg.set_gather_mode("auto")
        pkg.set_small_path(True)
    assert pkg.launch_count() - n0 == sum(v[0] for v in prof.values())
    names = ["align_small", "gemm1_swiglu", "gemm2_sorted", "reduce_sorted"]
    if gather == "separate":
        names.append("gather_rows")
    else:
        assert "gather_rows" not in prof
    for name in names:
        assert prof[name][0] == 1 and prof[name][1] > 0
