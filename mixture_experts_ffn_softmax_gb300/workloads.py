"""Seeded synthetic inputs for the fused MoE forward.

This module only draws random numbers with the shapes, distributions and
structure of the workloads named below; it holds none of the method's
arithmetic (no routing, no sorting, no expert FFN).  Both the CUDA path and
the CPU oracle receive the very same tensors from here.

Workloads (shapes from the MindIE-SD `fused_moe` page, "函数签名" / weight
layout: w13 [E, H, 2I], w2 [E, I, H], biases [E, 2I] and [E, H]):

* tiny            M=64,    H=256,  I=512,   E=8,   k=2, softmax + renormalize
* mixtral_prefill M=4096,  H=4096, I=14336, E=8,   k=2, softmax + renormalize
* mixtral_decode  M=16,    same layer
* deepseek_m64 / deepseek_m8192
                  E=256, k=8, H=7168, I=2048, sigmoid, group_count=8,
                  k_group=4, group_select_mode=1, routed_scaling_factor=2.5
* qwen_skew       E=128, k=8, H=2048, I=768, M=16384, softmax without
                  renormalize, with w13_bias / w2_bias ~ N(0, 0.01) and a
                  per-expert popularity bias added to the logits (Zipf law
                  over a seeded expert ranking: bias_e = -1.2 ln(rank_e + 1))
* qwen_skew_lit   the same, bias_e = raw Zipf(1.2) integer draws (stress case)
* batched         E=32, T=512, H=4096, I=2048, expert_num_tokens ~ U{0..512},
                  rows past the count filled with NaN, per-row weight = one
                  component of a Dirichlet(1) 4-vector

Every draw is seeded: stream seed+1 hidden, +2 logits, +3 w13, +4 w2,
+5 biases, +6 extras (counts, bias ranking, row weights).  N(0, s) means a
standard deviation of s.  Values are drawn in fp32 and rounded to bf16 where
the tensor is bf16.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class MoESpec:
    name: str
    M: int
    H: int
    I: int
    E: int
    top_k: int
    routing_method: str = "softmax"      # "softmax" | "sigmoid"
    renormalize: bool = False
    k_group: int = 1
    group_count: int = 1
    group_select_mode: int = 0
    routed_scaling_factor: float = 1.0
    bias: bool = False                   # w13_bias / w2_bias present
    logit_bias: Optional[str] = None     # None | "zipf_rank" | "zipf_raw"
    weight_std: float = 0.02
    bias_std: float = 0.01

    def scaled(self, name: str, **kw) -> "MoESpec":
        return dataclasses.replace(self, name=name, **kw)

    @property
    def R(self) -> int:
        return self.M * self.top_k

    def flops(self) -> float:
        """6 * R * H * I: two GEMMs, the first 2I wide."""
        return 6.0 * self.R * self.H * self.I


@dataclasses.dataclass(frozen=True)
class BatchedSpec:
    name: str
    E: int
    T: int
    H: int
    I: int
    top_k: int = 4
    bias: bool = False
    weight_std: float = 0.02
    bias_std: float = 0.01


SPECS = {
    "tiny": MoESpec("tiny", M=64, H=256, I=512, E=8, top_k=2,
                    routing_method="softmax", renormalize=True),
    "mixtral_prefill": MoESpec("mixtral_prefill", M=4096, H=4096, I=14336, E=8, top_k=2,
                               routing_method="softmax", renormalize=True),
    "mixtral_decode": MoESpec("mixtral_decode", M=16, H=4096, I=14336, E=8, top_k=2,
                              routing_method="softmax", renormalize=True),
    "deepseek_m64": MoESpec("deepseek_m64", M=64, H=7168, I=2048, E=256, top_k=8,
                            routing_method="sigmoid", k_group=4, group_count=8,
                            group_select_mode=1, routed_scaling_factor=2.5),
    "deepseek_m8192": MoESpec("deepseek_m8192", M=8192, H=7168, I=2048, E=256, top_k=8,
                              routing_method="sigmoid", k_group=4, group_count=8,
                              group_select_mode=1, routed_scaling_factor=2.5),
    "qwen_skew": MoESpec("qwen_skew", M=16384, H=2048, I=768, E=128, top_k=8,
                         routing_method="softmax", renormalize=False, bias=True,
                         logit_bias="zipf_rank"),
    "qwen_skew_lit": MoESpec("qwen_skew_lit", M=16384, H=2048, I=768, E=128, top_k=8,
                             routing_method="softmax", renormalize=False, bias=True,
                             logit_bias="zipf_raw"),
}

BATCHED_SPECS = {
    "batched": BatchedSpec("batched", E=32, T=512, H=4096, I=2048, top_k=4),
}

# Reduced copies that keep each workload's routing structure (E, k, groups,
# method, biases) but shrink H, I and M so the oracle finishes in seconds,
# while still spanning several GEMM tiles and a ragged tail in every dim.
SMALL_SPECS = {
    "tiny": SPECS["tiny"],
    "mixtral_small": SPECS["mixtral_prefill"].scaled("mixtral_small", M=333, H=512, I=640),
    "mixtral_decode_small": SPECS["mixtral_decode"].scaled("mixtral_decode_small", M=16, H=512, I=640),
    "deepseek_small": SPECS["deepseek_m8192"].scaled("deepseek_small", M=97, H=384, I=256),
    "qwen_small": SPECS["qwen_skew"].scaled("qwen_small", M=517, H=256, I=192),
    "qwen_lit_small": SPECS["qwen_skew_lit"].scaled("qwen_lit_small", M=211, H=256, I=192),
    "ragged_small": MoESpec("ragged_small", M=129, H=328, I=200, E=6, top_k=3,
                            routing_method="softmax", renormalize=True, bias=True),
}

# Copies sized for detailed profiler captures (a few GB on the device): the
# DeepSeek-V3 expert shape and rows per expert (256) with 32 experts.
PROFILE_SPECS = {
    "deepseek_e32": MoESpec("deepseek_e32", M=1024, H=7168, I=2048, E=32, top_k=8,
                            routing_method="sigmoid", k_group=4, group_count=8,
                            group_select_mode=1, routed_scaling_factor=2.5),
}

SMALL_BATCHED_SPECS = {
    "batched_small": BatchedSpec("batched_small", E=6, T=160, H=256, I=320, top_k=4),
    "batched_bias_small": BatchedSpec("batched_bias_small", E=5, T=140, H=200, I=136,
                                      top_k=2, bias=True),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std, g, device, dtype, chunk_elems=1 << 28):
    """N(0, std) drawn in fp32 and rounded to `dtype`, in slices along dim 0 so
    that full-size weights never need a full fp32 copy."""
    out = torch.empty(shape, dtype=dtype, device=device)
    if out.numel() == 0:
        return out
    rows = shape[0]
    per_row = max(1, out.numel() // rows)
    step = max(1, chunk_elems // per_row)
    for r0 in range(0, rows, step):
        r1 = min(rows, r0 + step)
        t = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=g, device=device,
                        dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        out[r0:r1].copy_(t)
    return out


def logit_bias(spec: MoESpec, seed: int = 0) -> Optional[np.ndarray]:
    """Per-expert additive logit bias that skews the routing (fp32, [E])."""
    if spec.logit_bias is None:
        return None
    rng = np.random.default_rng(seed + 6)
    if spec.logit_bias == "zipf_rank":
        rank = rng.permutation(spec.E)
        return (-1.2 * np.log(rank + 1.0)).astype(np.float32)
    if spec.logit_bias == "zipf_raw":
        return rng.zipf(1.2, spec.E).astype(np.float32)
    raise ValueError(spec.logit_bias)


def make_moe_inputs(spec: MoESpec, device="cpu", seed: int = 0, weights: bool = True):
    """Returns a dict of tensors on `device`:
    hidden [M,H] bf16, router_logits [M,E] fp32, w13 [E,H,2I] bf16,
    w2 [E,I,H] bf16, w13_bias [E,2I] bf16 or None, w2_bias [E,H] bf16 or None.
    """
    device = torch.device(device)
    M, H, I, E = spec.M, spec.H, spec.I, spec.E
    d = {}
    d["hidden"] = _normal((M, H), 1.0, _gen(seed + 1, device), device, torch.bfloat16)
    logits = _normal((M, E), 1.0, _gen(seed + 2, device), device, torch.float32)
    lb = logit_bias(spec, seed)
    if lb is not None:
        logits += torch.from_numpy(lb).to(device)
    d["router_logits"] = logits
    if weights:
        d["w13"] = _normal((E, H, 2 * I), spec.weight_std, _gen(seed + 3, device), device,
                           torch.bfloat16)
        d["w2"] = _normal((E, I, H), spec.weight_std, _gen(seed + 4, device), device,
                          torch.bfloat16)
        if spec.bias:
            g = _gen(seed + 5, device)
            d["w13_bias"] = _normal((E, 2 * I), spec.bias_std, g, device, torch.bfloat16)
            d["w2_bias"] = _normal((E, H), spec.bias_std, g, device, torch.bfloat16)
        else:
            d["w13_bias"] = None
            d["w2_bias"] = None
    return d


def make_fp8_weights(spec: MoESpec, device="cpu", seed: int = 0, per_channel: bool = True,
                     block: bool = False):
    """FP8 (E4M3) expert weights for the W8A8 layer: codes drawn as N(0, 1)
    values cast to float8_e4m3fn, and scales ~ U(0.015, 0.025) per output
    channel ([E, 2I] and [E, H]), per expert ([E]), or (block) per 128 x 128
    block ([E, H/128, 2I/128] and [E, I/128, H/128]) -- effective weights of
    standard deviation ~0.02, like the bf16 workloads."""
    device = torch.device(device)
    E, H, I = spec.E, spec.H, spec.I
    g = _gen(seed + 13, device)
    w13 = _normal((E, H, 2 * I), 1.0, g, device, torch.float8_e4m3fn)
    w2 = _normal((E, I, H), 1.0, g, device, torch.float8_e4m3fn)
    gs = _gen(seed + 14, device)
    if block:
        shape13, shape2 = (E, H // 128, 2 * I // 128), (E, I // 128, H // 128)
    elif per_channel:
        shape13, shape2 = (E, 2 * I), (E, H)
    else:
        shape13, shape2 = (E,), (E,)
    s13 = torch.rand(shape13, generator=gs, device=device) * 0.01 + 0.015
    s2 = torch.rand(shape2, generator=gs, device=device) * 0.01 + 0.015
    return {"w13_q": w13, "w2_q": w2, "w13_scale": s13, "w2_scale": s2}


def _codes(shape, lo, hi, g, device, dtype):
    """Uniform integer codes in [lo, hi], drawn in slices along dim 0."""
    out = torch.empty(shape, dtype=dtype, device=device)
    step = max(1, (1 << 28) // max(1, out[0].numel()))
    for r0 in range(0, shape[0], step):
        sl = out[r0:r0 + step]
        sl.copy_(torch.randint(lo, hi + 1, sl.shape, generator=g, device=device,
                               dtype=torch.int32).to(dtype))
    return out


def _pack_nibbles(codes: torch.Tensor) -> torch.Tensor:
    """int codes 0..15 [..., N] -> uint8 [..., N/2]: column 2j in the low nibble."""
    c = codes.to(torch.uint8)
    return c[..., 0::2] | (c[..., 1::2] << 4)


def make_wq_weights(spec: MoESpec, fmt: str = "int4", group_size: int = 128, device="cpu",
                    seed: int = 0, zero: bool = True):
    """Weight-only quantised expert weights for the layer:
    int4: codes ~ U{0..15}, zero points ~ U{6..9} (or none: 8), bf16 scales
          ~ U(0.0035, 0.0052) per (group, column) -- effective std ~0.02;
    int8: codes ~ U{-128..127}, zero points ~ U{-4..4} (or none), scales
          ~ U(2.2e-4, 3.2e-4);
    mxfp4: E2M1 codes ~ U{0..15}, UE8M0 scales ~ U{118..120} per block of 32;
    mxfp6_e3m2 / mxfp6_e2m3: codes ~ U{0..63} one per byte, UE8M0 scales
    ~ U{117..119} / U{119..121}.
    Returns codes, scales and zero points for w13 [E, H, 2I] and w2 [E, I, H]."""
    device = torch.device(device)
    E, H, I = spec.E, spec.H, spec.I
    g = _gen(seed + 21, device)
    mx = fmt.startswith("mxfp")
    out = {"fmt": fmt, "group_size": 32 if mx else group_size}
    G = out["group_size"]
    for name, K, N in (("w13", H, 2 * I), ("w2", I, H)):
        if fmt == "int8":
            out[name + "_q"] = _codes((E, K, N), -128, 127, g, device, torch.int8)
        elif fmt.startswith("mxfp6"):
            out[name + "_q"] = _codes((E, K, N), 0, 63, g, device, torch.uint8)
        else:
            q = _codes((E, K, N), 0, 15, g, device, torch.uint8)
            out[name + "_q"] = _pack_nibbles(q)
            del q
        if mx:
            lo, hi = {"mxfp4": (118, 120), "mxfp6_e3m2": (117, 119), "mxfp6_e2m3": (119, 121)}[fmt]
            out[name + "_scale"] = _codes((E, K // 32, N), lo, hi, g, device, torch.uint8)
            out[name + "_zero"] = None
            continue
        lo, hi = (0.0035, 0.0052) if fmt == "int4" else (2.2e-4, 3.2e-4)
        out[name + "_scale"] = (torch.rand(E, K // G, N, generator=g, device=device) * (hi - lo)
                                + lo).bfloat16()
        if zero:
            zlo, zhi, zdt = (6, 9, torch.uint8) if fmt == "int4" else (-4, 4, torch.int8)
            out[name + "_zero"] = _codes((E, K // G, N), zlo, zhi, g, device, zdt)
        else:
            out[name + "_zero"] = None
    return out


def make_batched_inputs(spec: BatchedSpec, device="cpu", seed: int = 0):
    """Returns a dict: x [E,T,H] bf16 (rows >= count are NaN), expert_num_tokens
    [E] int32 ~ U{0..T}, w13, w2, biases, row_weight [E,T] fp32 (one component
    of a Dirichlet(1) top_k-vector per row; 0 past the count)."""
    device = torch.device(device)
    E, T, H, I = spec.E, spec.T, spec.H, spec.I
    rng = np.random.default_rng(seed + 6)
    counts = rng.integers(0, T + 1, size=E).astype(np.int32)
    # Dirichlet(1) over top_k components, one component kept per row.
    dir_w = rng.dirichlet(np.ones(spec.top_k), size=(E, T)).astype(np.float32)
    comp = rng.integers(0, spec.top_k, size=(E, T))
    roww = np.take_along_axis(dir_w, comp[..., None], axis=2)[..., 0]
    valid = np.arange(T)[None, :] < counts[:, None]
    roww = np.where(valid, roww, 0.0).astype(np.float32)

    d = {}
    x = _normal((E, T, H), 1.0, _gen(seed + 1, device), device, torch.bfloat16)
    inval = torch.from_numpy(~valid).to(device)
    x[inval] = float("nan")
    d["x"] = x
    d["expert_num_tokens"] = torch.from_numpy(counts).to(device)
    d["row_weight"] = torch.from_numpy(roww).to(device)
    d["w13"] = _normal((E, H, 2 * I), spec.weight_std, _gen(seed + 3, device), device,
                       torch.bfloat16)
    d["w2"] = _normal((E, I, H), spec.weight_std, _gen(seed + 4, device), device,
                      torch.bfloat16)
    if spec.bias:
        g = _gen(seed + 5, device)
        d["w13_bias"] = _normal((E, 2 * I), spec.bias_std, g, device, torch.bfloat16)
        d["w2_bias"] = _normal((E, H), spec.bias_std, g, device, torch.bfloat16)
    else:
        d["w13_bias"] = None
        d["w2_bias"] = None
    return d


def to_f64(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    """Exact widening of a bf16 / fp32 tensor to a float64 numpy array."""
    if t is None:
        return None
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = ["MoESpec", "BatchedSpec", "SPECS", "BATCHED_SPECS", "SMALL_SPECS", "PROFILE_SPECS",
           "SMALL_BATCHED_SPECS", "make_moe_inputs", "make_batched_inputs", "make_fp8_weights",
           "logit_bias", "to_f64", "ceil_div"]
