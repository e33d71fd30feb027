"""GB300-native fused Mixture-of-Experts FFN forward.

Python binding of libgbmoe.so with the C ABI's names.  These functions only
marshal arguments: every step of the path (routing, align, permute, the two
grouped GEMMs, weight-and-reduce) runs in the library's CUDA kernels.
PyTorch supplies device memory and the current stream.

    w, ids = moe_route(logits, top_k, "softmax", renormalize=True)
    y = moe_forward(hidden, w, ids, w13, w2)            # [M, H] bf16
    y = fused_moe(hidden, logits, w13, w2, top_k, ...)  # route + forward
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib

MOE_OK = 0
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
          3: "MOE_ERR_WORKSPACE_TOO_SMALL", 4: "MOE_ERR_BAD_EXPERT_ID", 5: "MOE_ERR_TIMEOUT",
          6: "MOE_ERR_CUDA", 7: "MOE_ERR_NO_DEVICE"}
ROUTING = {"softmax": 0, "sigmoid": 1}
REDUCE = {"auto": 0, "epilogue_atomic": 1, "separate": 2}
BLOCK_M = 128
CHUNK_TOKENS = 16384


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}"
                         + (f" ({detail})" if detail else ""))


def lib():
    return _lib.load()


def _check(st: int, where: str):
    if st != MOE_OK:
        d = lib().moe_last_error_detail()
        raise MoEError(st, where, d.decode() if d else "")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


_raw_current_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_current_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream(stream=None):
    """The cudaStream_t handle of `stream`, else of the current stream.  The
    current one is read as a raw handle once CUDA is initialised (building a
    torch Stream object costs microseconds per call, as much as a launch)."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_current_stream is not None and _current_device is not None and \
            torch.cuda.is_initialized():
        return _raw_current_stream(_current_device())
    return torch.cuda.current_stream().cuda_stream


def workspace_size(M: int, H: int, I: int, E: int, top_k: int, reduce: str = "auto") -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size(M, H, I, E, top_k, REDUCE[reduce], ctypes.byref(n)),
           "moe_workspace_size")
    return n.value


def batched_workspace_size(E: int, T: int, H: int, I: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_batched_workspace_size(E, T, H, I, ctypes.byref(n)),
           "moe_batched_workspace_size")
    return n.value


def alloc_workspace(nbytes: int, device=None) -> torch.Tensor:
    # torch's caching allocator returns 512-byte aligned blocks.
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device or "cuda")


def moe_route(router_logits: torch.Tensor, top_k: int, routing_method: str = "softmax",
              renormalize: bool = False, k_group: int = 1, group_count: int = 1,
              group_select_mode: int = 0, routed_scaling_factor: float = 1.0,
              topk_weights: Optional[torch.Tensor] = None,
              topk_ids: Optional[torch.Tensor] = None, stream=None):
    """router_logits fp32 or bf16 [M, E] -> (topk_weights fp32 [M, k],
    topk_ids int32 [M, k])."""
    assert router_logits.dtype in (torch.float32, torch.bfloat16) and router_logits.dim() == 2
    M, E = router_logits.shape
    dev = router_logits.device
    if topk_weights is None:
        topk_weights = torch.empty(M, top_k, dtype=torch.float32, device=dev)
    if topk_ids is None:
        topk_ids = torch.empty(M, top_k, dtype=torch.int32, device=dev)
    fn = lib().moe_route if router_logits.dtype == torch.float32 else lib().moe_route_bf16
    _check(fn(_ptr(router_logits), M, E, top_k, ROUTING[routing_method],
              int(bool(renormalize)), k_group, group_count, group_select_mode,
              float(routed_scaling_factor), _ptr(topk_weights), _ptr(topk_ids),
              _stream(stream)), "moe_route")
    return topk_weights, topk_ids


def moe_router_logits(hidden: torch.Tensor, w_gate: torch.Tensor,
                      b_gate: Optional[torch.Tensor] = None,
                      logits: Optional[torch.Tensor] = None, stream=None):
    """s = hidden @ w_gate + b_gate on the tensor cores: hidden bf16 [M, H],
    w_gate bf16 [H, E], b_gate bf16 [E] -> fp32 [M, E]."""
    M, H = hidden.shape
    E = w_gate.shape[1]
    assert hidden.dtype == torch.bfloat16 and w_gate.dtype == torch.bfloat16
    if logits is None:
        logits = torch.empty(M, E, dtype=torch.float32, device=hidden.device)
    _check(lib().moe_router_logits(_ptr(hidden), _ptr(w_gate), _ptr(b_gate), M, H, E,
                                   _ptr(logits), _stream(stream)), "moe_router_logits")
    return logits


def align_capacity(M: int, top_k: int, E: int, block_m: int = BLOCK_M) -> int:
    return lib().moe_align_capacity(M, top_k, E, block_m)


def moe_align(topk_ids: torch.Tensor, E: int, block_m: int = BLOCK_M,
              error_word: Optional[torch.Tensor] = None, stream=None):
    """topk_ids int32 [M, k] -> dict(sorted_token_ids, expert_offsets,
    expert_num_tokens, block_expert_ids); sorted_token_ids is trimmed to
    capacity (valid up to expert_offsets[E])."""
    assert topk_ids.dtype == torch.int32 and topk_ids.dim() == 2
    M, k = topk_ids.shape
    dev = topk_ids.device
    cap = align_capacity(M, k, E, block_m)
    sorted_ids = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    blocks = torch.empty(max(cap // block_m, 1), dtype=torch.int32, device=dev)
    scratch_n = lib().moe_align_scratch_size(M, k, E)
    scratch = torch.empty(max(scratch_n, 4), dtype=torch.uint8, device=dev)
    _check(lib().moe_align(_ptr(topk_ids), M, k, E, block_m, _ptr(sorted_ids), _ptr(offsets),
                           _ptr(counts), _ptr(blocks), _ptr(scratch), scratch.numel(),
                           _ptr(error_word), _stream(stream)), "moe_align")
    return {"sorted_token_ids": sorted_ids[:cap], "expert_offsets": offsets,
            "expert_num_tokens": counts, "block_expert_ids": blocks[:cap // block_m]}


def moe_forward(hidden: torch.Tensor, topk_weights: torch.Tensor, topk_ids: torch.Tensor,
                w13: torch.Tensor, w2: torch.Tensor, w13_bias: Optional[torch.Tensor] = None,
                w2_bias: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                out: Optional[torch.Tensor] = None, reduce: str = "auto", stream=None,
                apply_router_weight_on_input: bool = False,
                expert_map: Optional[torch.Tensor] = None):
    """y [M, H] bf16 = sum_j topk_weights[:, j] * SwiGLU-expert_{topk_ids[:, j]}(hidden).

    apply_router_weight_on_input: the weight multiplies the second layer's
    input instead of its output.  expert_map: int32 [num_global_experts]
    mapping global ids in topk_ids to local experts (the E of w13) or -1
    (held elsewhere; those items contribute nothing)."""
    M, H = hidden.shape
    E, H2, I2 = w13.shape
    I = I2 // 2
    k = topk_ids.shape[1]
    assert hidden.dtype == torch.bfloat16 and w13.dtype == torch.bfloat16
    assert w2.dtype == torch.bfloat16 and tuple(w2.shape) == (E, I, H) and H2 == H
    assert topk_ids.dtype == torch.int32 and topk_weights.dtype == torch.float32
    if workspace is None:
        workspace = alloc_workspace(workspace_size(M, H, I, E, k, reduce), hidden.device)
    if out is None:
        out = torch.empty_like(hidden)
    if not apply_router_weight_on_input and expert_map is None:
        _check(lib().moe_forward(_ptr(hidden), _ptr(topk_weights), _ptr(topk_ids), M, H, I, E,
                                 k, _ptr(w13), _ptr(w2), _ptr(w13_bias), _ptr(w2_bias),
                                 _ptr(workspace), workspace.numel(), REDUCE[reduce], _ptr(out),
                                 _stream(stream)), "moe_forward")
        return out
    if expert_map is not None:
        assert expert_map.dtype == torch.int32 and expert_map.dim() == 1
    opts = _lib.ForwardOpts(REDUCE[reduce], int(bool(apply_router_weight_on_input)),
                            _ptr(expert_map), 0 if expert_map is None else expert_map.numel())
    _check(lib().moe_forward_opts(_ptr(hidden), _ptr(topk_weights), _ptr(topk_ids), M, H, I, E,
                                  k, _ptr(w13), _ptr(w2), _ptr(w13_bias), _ptr(w2_bias),
                                  _ptr(workspace), workspace.numel(), ctypes.byref(opts),
                                  _ptr(out), _stream(stream)), "moe_forward_opts")
    return out


def workspace_size_fp8(M: int, H: int, I: int, E: int, top_k: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size_fp8(M, H, I, E, top_k, ctypes.byref(n)),
           "moe_workspace_size_fp8")
    return n.value


def moe_forward_fp8(hidden: torch.Tensor, topk_weights: torch.Tensor, topk_ids: torch.Tensor,
                    w13_q: torch.Tensor, w2_q: torch.Tensor, w13_scale: torch.Tensor,
                    w2_scale: torch.Tensor, w13_bias: Optional[torch.Tensor] = None,
                    w2_bias: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None,
                    out: Optional[torch.Tensor] = None, stream=None):
    """FP8 W8A8 layer: w13_q [E, H, 2I] / w2_q [E, I, H] E4M3 (torch.float8_e4m3fn
    or uint8 bytes), scales fp32 per expert [E], per output channel
    ([E, 2I] / [E, H]) or per 128 x 128 block ([E, H/128, 2I/128] /
    [E, I/128, H/128]); activations are quantised on the GPU per row, or per
    (row, group of 128) with block scales."""
    M, H = hidden.shape
    E, _, I2 = w13_q.shape
    I = I2 // 2
    k = topk_ids.shape[1]
    scale_mode = w13_scale.dim() - 1          # 0 per expert, 1 per channel, 2 per block
    assert w13_scale.dtype == torch.float32 and w2_scale.dtype == torch.float32
    if workspace is None:
        workspace = alloc_workspace(workspace_size_fp8(M, H, I, E, k), hidden.device)
    if out is None:
        out = torch.empty_like(hidden)
    wts = _lib.Fp8Weights(_ptr(w13_q), _ptr(w2_q), _ptr(w13_scale), _ptr(w2_scale), scale_mode)
    _check(lib().moe_forward_fp8(_ptr(hidden), _ptr(topk_weights), _ptr(topk_ids), M, H, I, E, k,
                                 ctypes.byref(wts), _ptr(w13_bias), _ptr(w2_bias),
                                 _ptr(workspace), workspace.numel(), _ptr(out), _stream(stream)),
           "moe_forward_fp8")
    return out


def moe_quant_rows_fp8(x: torch.Tensor, q8: Optional[torch.Tensor] = None,
                       scale: Optional[torch.Tensor] = None, stream=None):
    """Per-row E4M3 quantisation of x [M, H] bf16 -> (codes [M, H]
    torch.float8_e4m3fn, scale [M] fp32): x ~ codes * scale[:, None]."""
    M, H = x.shape
    if q8 is None:
        q8 = torch.empty(M, H, dtype=torch.float8_e4m3fn, device=x.device)
    if scale is None:
        scale = torch.empty(M, dtype=torch.float32, device=x.device)
    _check(lib().moe_quant_rows_fp8(_ptr(x), M, H, _ptr(q8), _ptr(scale), _stream(stream)),
           "moe_quant_rows_fp8")
    return q8, scale


WQ_FORMATS = {"int4": 0, "int8": 1, "mxfp4": 2, "mxfp6_e3m2": 3, "mxfp6_e2m3": 4}


def _wq_shape(fmt: str, codes: torch.Tensor):
    E, K, n = codes.shape
    return E, K, (2 * n if fmt in ("int4", "mxfp4") else n)


def moe_dequant_weights(fmt: str, codes: torch.Tensor, scale: torch.Tensor,
                        zero: Optional[torch.Tensor] = None, group_size: int = 128,
                        out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Weight-only quantised weights -> bf16 [E, K, N] (fmt "int4", "int8",
    "mxfp4", "mxfp6_e3m2" or "mxfp6_e2m3"; layouts as moe_forward_wq)."""
    E, K, N = _wq_shape(fmt, codes)
    if out is None:
        out = torch.empty(E, K, N, dtype=torch.bfloat16, device=codes.device)
    _check(lib().moe_dequant_weights(WQ_FORMATS[fmt], _ptr(codes), _ptr(scale), _ptr(zero), E, K,
                                     N, group_size, _ptr(out), _stream(stream)),
           "moe_dequant_weights")
    return out


def moe_forward_wq(hidden: torch.Tensor, topk_weights: torch.Tensor, topk_ids: torch.Tensor,
                   fmt: str, w13_q: torch.Tensor, w2_q: torch.Tensor, w13_scale: torch.Tensor,
                   w2_scale: torch.Tensor, w13_zero: Optional[torch.Tensor] = None,
                   w2_zero: Optional[torch.Tensor] = None, group_size: int = 128,
                   w13_bias: Optional[torch.Tensor] = None,
                   w2_bias: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None,
                   out: Optional[torch.Tensor] = None, stream=None):
    """Layer with weight-only quantised experts.  int4 / MX FP4 codes uint8
    [E, K, N/2] (column 2j in the low nibble), int8 codes int8 [E, K, N],
    MX FP6 codes uint8 [E, K, N] (6-bit code in the low bits); scales bf16
    [E, K/G, N] (int) or uint8 UE8M0 [E, K/32, N] (MX); zero points uint8 /
    int8 [E, K/G, N] or None.  w13: K = H, N = 2I; w2: K = I, N = H."""
    M, H = hidden.shape
    E, _, N13 = _wq_shape(fmt, w13_q)
    I = N13 // 2
    k = topk_ids.shape[1]
    if workspace is None:
        workspace = alloc_workspace(workspace_size(M, H, I, E, k, "separate"), hidden.device)
    if out is None:
        out = torch.empty_like(hidden)
    wts = _lib.WqWeights(WQ_FORMATS[fmt], group_size, _ptr(w13_q), _ptr(w2_q), _ptr(w13_scale),
                         _ptr(w2_scale), _ptr(w13_zero), _ptr(w2_zero))
    _check(lib().moe_forward_wq(_ptr(hidden), _ptr(topk_weights), _ptr(topk_ids), M, H, I, E, k,
                                ctypes.byref(wts), _ptr(w13_bias), _ptr(w2_bias), _ptr(workspace),
                                workspace.numel(), _ptr(out), _stream(stream)), "moe_forward_wq")
    return out


class HostStaging:
    """Device buffers of moe_forward_host for M tokens: hidden [M, H] bf16,
    router logits [M, E] fp32, top-k weights [M, k] fp32 and ids [M, k]
    int32, out [M, H] bf16, and the forward's workspace."""

    def __init__(self, M: int, H: int, I: int, E: int, top_k: int, device="cuda",
                 reduce: str = "auto"):
        self.hidden = torch.empty(M, H, dtype=torch.bfloat16, device=device)
        self.logits = torch.empty(M, E, dtype=torch.float32, device=device)
        self.topk_weights = torch.empty(M, top_k, dtype=torch.float32, device=device)
        self.topk_ids = torch.empty(M, top_k, dtype=torch.int32, device=device)
        self.out = torch.empty(M, H, dtype=torch.bfloat16, device=device)
        self.workspace = alloc_workspace(workspace_size(M, H, I, E, top_k, reduce), device)


def moe_forward_host(hidden: torch.Tensor, router_logits: torch.Tensor, w13: torch.Tensor,
                     w2: torch.Tensor, top_k: int, routing_method: str = "softmax",
                     renormalize: bool = False, k_group: int = 1, group_count: int = 1,
                     group_select_mode: int = 0, routed_scaling_factor: float = 1.0,
                     w13_bias: Optional[torch.Tensor] = None,
                     w2_bias: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                     staging: Optional[HostStaging] = None, reduce: str = "auto", stream=None):
    """One layer step from host memory: hidden bf16 [M, H] and router_logits
    fp32 [M, E] on the host (pinned for full copy speed) -> out bf16 [M, H]
    on the host, routed as moe_route and computed as moe_forward, the copies
    inside the call.  Asynchronous on `stream`: out is complete once the
    stream has passed the call."""
    M, H = hidden.shape
    E, _, I2 = w13.shape
    assert hidden.device.type == "cpu" and router_logits.device.type == "cpu"
    assert hidden.dtype == torch.bfloat16 and router_logits.dtype == torch.float32
    assert hidden.is_contiguous() and router_logits.is_contiguous()
    if staging is None:
        staging = HostStaging(M, H, I2 // 2, E, top_k, w13.device, reduce)
    if out is None:
        out = torch.empty(M, H, dtype=torch.bfloat16, pin_memory=True)
    io = _lib.HostIo(_ptr(hidden), _ptr(router_logits), _ptr(out), _ptr(staging.hidden),
                     _ptr(staging.logits), _ptr(staging.topk_weights), _ptr(staging.topk_ids),
                     _ptr(staging.out))
    rp = _lib.RouteParams(top_k, ROUTING[routing_method], int(bool(renormalize)), k_group,
                          group_count, group_select_mode, float(routed_scaling_factor))
    _check(lib().moe_forward_host(ctypes.byref(io), M, H, I2 // 2, E, ctypes.byref(rp),
                                  _ptr(w13), _ptr(w2), _ptr(w13_bias), _ptr(w2_bias),
                                  _ptr(staging.workspace), staging.workspace.numel(),
                                  REDUCE[reduce], _stream(stream)), "moe_forward_host")
    return out


def moe_forward_batched(x: torch.Tensor, expert_num_tokens: torch.Tensor, w13: torch.Tensor,
                        w2: torch.Tensor, w13_bias: Optional[torch.Tensor] = None,
                        w2_bias: Optional[torch.Tensor] = None,
                        row_weight: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None,
                        out: Optional[torch.Tensor] = None, stream=None):
    """Batched layout: x [E, T, H] bf16 with expert_num_tokens [E] int32 ->
    out [E, T, H] bf16 (rows past the count are not written)."""
    E, T, H = x.shape
    I = w13.shape[2] // 2
    assert expert_num_tokens.dtype == torch.int32
    if workspace is None:
        workspace = alloc_workspace(batched_workspace_size(E, T, H, I), x.device)
    if out is None:
        out = torch.empty_like(x)
    _check(lib().moe_forward_batched(_ptr(x), _ptr(expert_num_tokens), E, T, H, I, _ptr(w13),
                                     _ptr(w2), _ptr(w13_bias), _ptr(w2_bias), _ptr(row_weight),
                                     _ptr(workspace), workspace.numel(), _ptr(out),
                                     _stream(stream)), "moe_forward_batched")
    return out


def fused_moe(hidden: torch.Tensor, router_logits: torch.Tensor, w13: torch.Tensor,
              w2: torch.Tensor, top_k: int, w13_bias=None, w2_bias=None, k_group: int = 1,
              group_count: int = 1, group_select_mode: int = 0, routing_method: str = "softmax",
              renormalize: bool = False, routed_scaling_factor: float = 1.0, workspace=None,
              out=None, stream=None):
    """The whole layer: route, then forward (the MindIE-SD `fused_moe` shape)."""
    w, ids = moe_route(router_logits, top_k, routing_method, renormalize, k_group, group_count,
                       group_select_mode, routed_scaling_factor, stream=stream)
    return moe_forward(hidden, w, ids, w13, w2, w13_bias, w2_bias, workspace, out, stream=stream)


def moe_layer(hidden: torch.Tensor, w_gate: torch.Tensor, w13: torch.Tensor, w2: torch.Tensor,
              top_k: int, b_gate=None, w13_bias=None, w2_bias=None, k_group: int = 1,
              group_count: int = 1, group_select_mode: int = 0,
              routing_method: str = "softmax", renormalize: bool = False,
              routed_scaling_factor: float = 1.0, workspace=None, out=None, stream=None):
    """The layer from the hidden states: router logits (x W_g + b_g), routing,
    then the expert forward."""
    logits = moe_router_logits(hidden, w_gate, b_gate, stream=stream)
    return fused_moe(hidden, logits, w13, w2, top_k, w13_bias, w2_bias, k_group, group_count,
                     group_select_mode, routing_method, renormalize, routed_scaling_factor,
                     workspace, out, stream)


def workspace_error_word(workspace: torch.Tensor) -> int:
    return lib().moe_workspace_error_word(_ptr(workspace))


def read_error(error_word_ptr: int, reset: bool = True, stream=None) -> int:
    """Synchronises the stream and returns the device error status (0 = ok)."""
    return lib().moe_read_error(error_word_ptr, int(reset), _stream(stream))


def workspace_layout(M: int, H: int, I: int, E: int, top_k: int) -> dict:
    """Byte offsets of the forward workspace's regions (for inspecting
    intermediate stages)."""
    arr = (ctypes.c_size_t * 11)()
    _check(lib().moe_workspace_layout(M, H, I, E, top_k, arr), "moe_workspace_layout")
    names = ["error_word", "expert_num_tokens", "expert_offsets", "block_expert_ids",
             "sorted_token_ids", "align_scratch", "inv", "a_perm", "z", "item_out", "cap"]
    return dict(zip(names, list(arr)))


def selftest_wait_timeout(error_word: torch.Tensor, limit_us: int = 20000, stream=None):
    _check(lib().moe_selftest_wait_timeout(_ptr(error_word), limit_us, _stream(stream)),
           "moe_selftest_wait_timeout")


def set_gemm_tiles(mode: str = "auto"):
    """Grouped-GEMM tile shape: "auto", "single" (one CTA per 128x256 tile)
    or "pairs" (CTA pairs sharing a 256x256 tcgen05 cta_group::2 tile)."""
    _check(lib().moe_set_gemm_tiles({"auto": 0, "single": 1, "pairs": 2}[mode]),
           "moe_set_gemm_tiles")


def launch_count() -> int:
    return lib().moe_launch_count()


def set_gather_mode(mode: str = "auto"):
    """Where GEMM1 takes its rows from: "auto", "separate" (a gather kernel
    writes the expert-sorted rows first) or "fused" (GEMM1 copies them from
    the token rows itself).  Results are identical."""
    _check(lib().moe_set_gather_mode({"auto": 0, "separate": 1, "fused": 2}[mode]),
           "moe_set_gather_mode")


def set_pdl(enabled: bool = True):
    """Programmatic dependent launch between the library's consecutive
    kernels (on by default): each kernel waits on the device for the one
    before it, and kernels with small grids let the next one be scheduled
    while they run.  Results are identical either way."""
    _check(lib().moe_set_pdl(1 if enabled else 0), "moe_set_pdl")


def set_item_rows(fmt: str = "auto"):
    """Item rows of the separate weight-and-reduce: "auto" (default: fp16
    when top_k >= 4), "fp32", or "fp16" (fp16 values with a power-of-two
    exponent per row and 32-column chunk).  Results agree to fp16 rounding
    of each weighted item row."""
    modes = {"auto": 0, "fp32": 1, "fp16": 2}
    if fmt not in modes:
        raise ValueError(f"item row format {fmt!r}")
    _check(lib().moe_set_item_rows(modes[fmt]), "moe_set_item_rows")


def set_wq_decode(enabled: bool = True):
    """Weight-only layers of at most 32 tokens through the decode GEMMs
    (weights expanded in registers, the expert's few rows as the MMA's N; on
    by default) or always through the grouped tensor-core GEMMs.  Results
    agree up to fp32 summation order."""
    _check(lib().moe_set_wq_decode(1 if enabled else 0), "moe_set_wq_decode")


def set_host_out_direct(enabled: bool = True):
    """moe_forward_host with a pinned `out`: the last token chunk's reduce
    writes its rows straight into it over the host link (on by default), or
    every chunk goes through the device staging buffer and a copy.  Results
    are identical."""
    _check(lib().moe_set_host_out_direct(1 if enabled else 0), "moe_set_host_out_direct")


def set_small_path(enabled: bool = True):
    """Small calls (at most 256 routed items, small expert weights, the
    automatic reduce) in two kernels with the plan, gather and reduce folded
    into the GEMMs (on by default), or always the general path.  Results
    agree up to fp32 summation order."""
    _check(lib().moe_set_small_path(1 if enabled else 0), "moe_set_small_path")


def profiler_start():
    _check(lib().moe_profiler_start(), "moe_profiler_start")


def profiler_stop():
    """Returns {kernel name: (launches, total_ms)} for launches since start."""
    cap = 64
    arr = (_lib.KernelTime * cap)()
    n = ctypes.c_int32(0)
    _check(lib().moe_profiler_stop(arr, cap, ctypes.byref(n)), "moe_profiler_stop")
    return {arr[i].name.decode(): (arr[i].launches, arr[i].total_ms) for i in range(n.value)}


__all__ = ["moe_route", "moe_router_logits", "moe_layer", "moe_align", "moe_forward",
           "moe_forward_host", "HostStaging", "set_gather_mode", "set_pdl", "set_wq_decode",
           "set_item_rows", "set_host_out_direct", "set_small_path",
           "moe_forward_batched", "moe_forward_fp8", "workspace_size_fp8", "moe_quant_rows_fp8",
           "moe_dequant_weights", "moe_forward_wq", "WQ_FORMATS",
           "fused_moe",
           "workspace_size", "batched_workspace_size", "alloc_workspace", "align_capacity",
           "workspace_error_word", "read_error", "launch_count", "workspace_layout",
           "selftest_wait_timeout", "set_gemm_tiles", "profiler_start",
           "profiler_stop", "MoEError", "STATUS", "lib"]
