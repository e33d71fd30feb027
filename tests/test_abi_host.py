"""CPU tests of the C ABI: the library loads, exports every symbol the
header declares, and host-side validation returns the documented status
codes before any GPU access."""
import ctypes
import os
import re

import pytest

import mixture_experts_ffn_softmax_gb300 as pkg
from mixture_experts_ffn_softmax_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbmoe.h")

OK, INVALID, WS_SMALL, NO_DEVICE = 0, 1, 3, 7


def declared_symbols():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"GBMOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", txt)))


def test_library_exports_every_declared_symbol():
    lib = pkg.lib()
    names = declared_symbols()
    assert len(names) >= 18
    for n in names:
        assert hasattr(lib, n), f"libgbmoe.so does not export {n}"
        assert n in _lib.SIGNATURES, f"binding lacks a signature for {n}"
    assert lib.moe_abi_version() == 1


def test_status_strings():
    lib = pkg.lib()
    for code, name in pkg.STATUS.items():
        assert lib.moe_status_string(code).decode() == name


def _route(lib, M=4, E=8, k=2, method=0, renorm=1, kg=1, G=1, mode=0, scale=1.0, ptr=1):
    p = ctypes.c_void_p(ptr)
    return lib.moe_route(p, M, E, k, method, renorm, kg, G, mode, scale, p, p, None)


def test_route_validation():
    lib = pkg.lib()
    assert _route(lib, M=-1) == INVALID
    assert _route(lib, E=0) == INVALID
    assert _route(lib, E=1025) == INVALID
    assert _route(lib, k=0) == INVALID
    assert _route(lib, k=9) == INVALID                     # top_k > E
    assert _route(lib, E=128, k=65) == INVALID             # top_k > 64
    assert _route(lib, method=2) == INVALID
    assert _route(lib, E=8, G=3) == INVALID                # E % group_count
    assert _route(lib, E=8, G=4, kg=5) == INVALID          # k_group > group_count
    assert _route(lib, E=8, G=4, kg=0) == INVALID
    assert _route(lib, E=8, G=8, kg=2, mode=1) == INVALID  # mode 1 needs >= 2 per group
    assert _route(lib, E=8, G=4, kg=1, k=3) == INVALID     # top_k > experts in kept groups
    assert _route(lib, mode=2) == INVALID
    assert _route(lib, scale=float("nan")) == INVALID
    assert _route(lib, ptr=0) == INVALID                   # null pointers
    assert _route(lib, M=0) == OK                          # empty: no-op
    assert _route(lib, k=9) == INVALID
    assert b"top_k" in lib.moe_last_error_detail()


def test_route_needs_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _route(pkg.lib()) == NO_DEVICE


def test_workspace_size_validation():
    lib = pkg.lib()
    n = ctypes.c_size_t(0)
    assert lib.moe_workspace_size(16, 4096, 14336, 8, 2, 0, ctypes.byref(n)) == OK
    assert n.value > 0
    assert lib.moe_workspace_size(16, 100, 64, 8, 2, 0, ctypes.byref(n)) == INVALID
    assert lib.moe_workspace_size(16, 64, 60, 8, 2, 0, ctypes.byref(n)) == INVALID
    assert lib.moe_workspace_size(16, 64, 64, 0, 2, 0, ctypes.byref(n)) == INVALID
    assert lib.moe_workspace_size(16, 64, 64, 8, 65, 0, ctypes.byref(n)) == INVALID
    assert lib.moe_workspace_size(16, 64, 64, 8, 2, 1, ctypes.byref(n)) == OK   # atomic reduce
    assert lib.moe_workspace_size(16, 64, 64, 8, 2, 2, ctypes.byref(n)) == OK   # separate
    assert lib.moe_workspace_size(16, 64, 64, 8, 2, 7, ctypes.byref(n)) == INVALID
    assert lib.moe_workspace_size(-1, 64, 64, 8, 2, 0, ctypes.byref(n)) == INVALID


def test_workspace_is_bounded_by_the_token_chunk():
    a = pkg.workspace_size(pkg.CHUNK_TOKENS, 1024, 512, 16, 4)
    b = pkg.workspace_size(10 * pkg.CHUNK_TOKENS, 1024, 512, 16, 4)
    assert a == b
    assert pkg.workspace_size(100, 1024, 512, 16, 4) < a


def test_workspace_layout_regions_are_ordered_and_aligned():
    lay = pkg.workspace_layout(333, 512, 640, 8, 2)
    keys = ["error_word", "expert_num_tokens", "expert_offsets", "block_expert_ids",
            "sorted_token_ids", "align_scratch", "inv", "a_perm", "z", "item_out"]
    offs = [lay[k] for k in keys]
    assert offs == sorted(offs) and offs[0] == 0
    assert all(o % 1024 == 0 for o in offs)
    cap = lay["cap"]
    assert cap % 128 == 0 and cap >= 333 * 2
    assert lay["item_out"] - lay["z"] >= cap * 640 * 2
    assert lay["a_perm"] - lay["inv"] >= 333 * 2 * 4
    assert lay["z"] - lay["a_perm"] >= cap * 512 * 2
    assert pkg.workspace_size(333, 512, 640, 8, 2) >= lay["item_out"] + cap * 512 * 4


def test_forward_validation():
    lib = pkg.lib()
    p = ctypes.c_void_p(4096)
    n = ctypes.c_size_t(0)
    lib.moe_workspace_size(8, 64, 64, 4, 2, 0, ctypes.byref(n))
    need = n.value

    def fwd(M=8, H=64, I=64, E=4, k=2, ws=need, mode=0, out=p, wsp=ctypes.c_void_p(1 << 20)):
        return lib.moe_forward(p, p, p, M, H, I, E, k, p, p, None, None, wsp, ws, mode, out,
                               None)
    assert fwd(M=0) == OK
    assert fwd(H=60) == INVALID
    assert fwd(ws=need - 1) == WS_SMALL
    assert fwd(mode=3) == INVALID
    assert fwd(out=None) == INVALID
    assert fwd(wsp=ctypes.c_void_p((1 << 20) + 16)) == INVALID   # workspace alignment
    bad = ctypes.c_void_p(4096 + 8)                                # misaligned tensor
    assert lib.moe_forward(bad, p, p, 8, 64, 64, 4, 2, p, p, None, None,
                           ctypes.c_void_p(1 << 20), need, 0, p, None) == INVALID


def test_forward_host_validation():
    """The host-memory step checks routing and forward arguments before it
    enqueues anything (no GPU here: valid arguments reach the device check)."""
    lib = pkg.lib()
    p = ctypes.c_void_p(4096)
    n = ctypes.c_size_t(0)
    lib.moe_workspace_size(8, 64, 64, 4, 2, 0, ctypes.byref(n))
    need = n.value
    io = _lib.HostIo(4096, 4096, 4096, 4096, 4096, 4096, 4096, 4096)

    def step(M=8, H=64, I=64, E=4, k=2, ws=need, io_=io, method=0, groups=1):
        rp = _lib.RouteParams(k, method, 1, 1, groups, 0, 1.0)
        return lib.moe_forward_host(ctypes.byref(io_) if io_ is not None else None, M, H, I, E,
                                    ctypes.byref(rp), p, p, None, None, ctypes.c_void_p(1 << 20),
                                    ws, 0, None)
    assert step(M=0) == OK
    assert step(io_=None) == INVALID
    assert step(k=5) == INVALID          # top_k > E
    assert step(method=2) == INVALID
    assert step(groups=3) == INVALID     # E % group_count
    assert step(H=60) == INVALID
    assert step(ws=need - 1) == WS_SMALL
    assert step() == NO_DEVICE


def test_batched_validation():
    lib = pkg.lib()
    n = ctypes.c_size_t(0)
    assert lib.moe_batched_workspace_size(32, 512, 4096, 2048, ctypes.byref(n)) == OK
    assert lib.moe_batched_workspace_size(32, 0, 4096, 2048, ctypes.byref(n)) == INVALID
    assert lib.moe_batched_workspace_size(32, 512, 4095, 2048, ctypes.byref(n)) == INVALID
    assert lib.moe_batched_workspace_size(1024, 1 << 21, 64, 64, ctypes.byref(n)) == INVALID


def test_align_capacity_and_validation():
    lib = pkg.lib()
    assert lib.moe_align_capacity(64, 2, 8, 128) == 128 + 8 * 127 + (128 - (128 + 8 * 127) % 128) % 128
    assert lib.moe_align_capacity(1, 1, 256, 128) == 128          # one busy expert at most
    assert lib.moe_align_capacity(0, 2, 8, 16) == 0
    p = ctypes.c_void_p(4096)
    assert lib.moe_align(p, 4, 2, 8, 0, p, p, p, p, p, 1 << 20, None, None) == INVALID
    assert lib.moe_align(p, 4, 2, 8, 2048, p, p, p, p, p, 1 << 20, None, None) == INVALID
    assert lib.moe_align(p, 4, 2, 8, 16, p, p, p, p, p, 0, None, None) == WS_SMALL


def test_gemm_tile_mode_validation():
    lib = pkg.lib()
    assert lib.moe_set_gemm_tiles(3) == INVALID
    assert lib.moe_set_gemm_tiles(-1) == INVALID
    for m in (2, 1, 0):
        assert lib.moe_set_gemm_tiles(m) == OK


def test_pdl_switch_validation():
    lib = pkg.lib()
    assert lib.moe_set_pdl(2) == INVALID
    assert lib.moe_set_pdl(-1) == INVALID
    for m in (0, 1):
        assert lib.moe_set_pdl(m) == OK


def test_item_rows_switch_validation():
    lib = pkg.lib()
    assert lib.moe_set_item_rows(3) == INVALID
    assert lib.moe_set_item_rows(-1) == INVALID
    for m in (2, 1, 0):
        assert lib.moe_set_item_rows(m) == OK
    with pytest.raises(ValueError):
        pkg.set_item_rows("bf16")


def test_small_path_switch_validation():
    lib = pkg.lib()
    assert lib.moe_set_small_path(2) == INVALID
    assert lib.moe_set_small_path(-1) == INVALID
    for m in (0, 1):
        assert lib.moe_set_small_path(m) == OK


def test_host_out_direct_switch_validation():
    lib = pkg.lib()
    assert lib.moe_set_host_out_direct(2) == INVALID
    assert lib.moe_set_host_out_direct(-1) == INVALID
    for m in (0, 1):
        assert lib.moe_set_host_out_direct(m) == OK


def test_wq_decode_switch_validation():
    lib = pkg.lib()
    assert lib.moe_set_wq_decode(2) == INVALID
    assert lib.moe_set_wq_decode(-1) == INVALID
    for m in (0, 1):
        assert lib.moe_set_wq_decode(m) == OK


def test_gather_mode_validation():
    lib = pkg.lib()
    assert lib.moe_set_gather_mode(3) == INVALID
    assert lib.moe_set_gather_mode(-1) == INVALID
    for m in (2, 1, 0):
        assert lib.moe_set_gather_mode(m) == OK
    with pytest.raises(KeyError):
        pkg.set_gather_mode("tma")


def test_binding_fails_loudly_without_library(tmp_path):
    _lib._lib_saved = _lib._lib
    try:
        _lib._lib = None
        with pytest.raises(ImportError):
            _lib.load(str(tmp_path / "libgbmoe.so"))
    finally:
        _lib._lib = _lib._lib_saved
