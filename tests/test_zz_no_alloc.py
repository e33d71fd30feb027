"""moe_align_static_scratch: the align entry point for callers that cannot
allocate device memory (an operator inside another framework with no handle
to its allocator, or a latency-critical loop where cudaMalloc is not
allowed).  Its scratch is a static device array owned by the library.

Checks, through the C ABI, that calls in a row give exactly what the
regular moe_align (caller-provided scratch) gives: the outputs are integer
index data, so the comparison is bit-exact.  Every case is large enough to
take the four-kernel align path (more than 4096 routed items with more than
16 experts), the only path that uses the static array; the second and third
calls are smaller than the first and use other expert counts, so the table
is laid out differently in the array each time, and stale contents left by
an earlier call would show up as a mismatch.  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import mixture_experts_ffn_softmax_gb300 as pkg

pytestmark = pytest.mark.gpu

MAX_INTS = 1 << 18   # MOE_ALIGN_STATIC_SCRATCH_INTS


def _outputs(M, k, E, bm, dev):
    cap = pkg.align_capacity(M, k, E, bm)
    return {
        "sorted": torch.full((cap,), -7, dtype=torch.int32, device=dev),
        "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
        "counts": torch.full((E,), -7, dtype=torch.int32, device=dev),
        "blocks": torch.full((max(cap // bm, 1),), -7, dtype=torch.int32, device=dev),
        "err": torch.zeros(1, dtype=torch.int32, device=dev),
    }


def _call_static(ids, M, k, E, bm, o):
    st = pkg.lib().moe_align_static_scratch(
        ids.data_ptr(), M, k, E, bm, o["sorted"].data_ptr(), o["offsets"].data_ptr(),
        o["counts"].data_ptr(), o["blocks"].data_ptr(), o["err"].data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == 0, pkg.lib().moe_last_error_detail()


def _call_regular(ids, M, k, E, bm, o):
    n = pkg.lib().moe_align_scratch_size(M, k, E)
    scratch = torch.empty(max(n, 4), dtype=torch.uint8, device=ids.device)
    st = pkg.lib().moe_align(
        ids.data_ptr(), M, k, E, bm, o["sorted"].data_ptr(), o["offsets"].data_ptr(),
        o["counts"].data_ptr(), o["blocks"].data_ptr(), scratch.data_ptr(), scratch.numel(),
        o["err"].data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, pkg.lib().moe_last_error_detail()


def _ids(M, k, E, seed):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
    ids[: M // 3, 0] = 1                                   # some skew
    return torch.from_numpy(ids).cuda()


def test_static_scratch_align_matches_regular_align_twice():
    dev = torch.device("cuda")
    for M, k, E, bm, seed in ((8192, 8, 256, 128, 0), (1000, 6, 64, 16, 1),
                              (3000, 8, 100, 64, 2)):
        assert -(-(M * k) // 256) * E <= MAX_INTS
        assert M * k > 4096 and E > 16        # the four-kernel path, which uses the array
        ids = _ids(M, k, E, seed)
        a, b = _outputs(M, k, E, bm, dev), _outputs(M, k, E, bm, dev)
        _call_static(ids, M, k, E, bm, a)
        _call_regular(ids, M, k, E, bm, b)
        torch.cuda.synchronize()
        n = int(b["offsets"][E].item())
        assert torch.equal(a["offsets"], b["offsets"])
        assert torch.equal(a["counts"], b["counts"])
        assert torch.equal(a["sorted"][:n], b["sorted"][:n])
        assert torch.equal(a["blocks"], b["blocks"])
        assert int(a["err"].item()) == 0 and int(b["err"].item()) == 0
        assert int(a["counts"].sum().item()) == M * k


def test_static_scratch_align_rejects_oversize():
    # ceil(M*k/256) * E above the static array's capacity -> clear error, no launch
    M, k, E = 1 << 16, 8, 256
    p = ctypes.c_void_p(4096)
    st = pkg.lib().moe_align_static_scratch(p, M, k, E, 128, p, p, p, p, None, None)
    assert st == 3   # MOE_ERR_WORKSPACE_TOO_SMALL
    assert b"static scratch" in pkg.lib().moe_last_error_detail()
