"""CPU oracle for the fused MoE forward -- TEST INFRASTRUCTURE ONLY.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's ``cpu_baseline`` /
``--impl reference`` legs may import this module.  The product path
(``mixture_experts_ffn_softmax_gb300``) never calls it and shares no code
with it: the only thing both sides have in common is the seeded input
generator module, which holds none of the method's arithmetic.

Everything here is plain numpy in float64 (inputs are widened exactly from
bf16 / fp32), written straight from the definitions on the pages, with no
blocking, fusion or reordering beyond what those definitions state.  Library
primitives used as steps: ``np.exp``, ``@`` (matmul), ``np.argsort`` with a
stable sort.

Sources (page title, section):

* "FlagGems fused_moe.py analysis" (FlagDoc flaggems/fused_moe.md), section
  1.1 "MoE layer math": router scores s_t, p_t = softmax(s_t), S_t = TopK(p_t, k),
  f_e(x) = W2_e^T SiLU(W1_e^T x + b1_e) + b2_e, y_t = sum_{e in S_t} alpha_{t,e} f_e(x_t).
* same page, section 1.2 "fused_moe math": routed items r = (token, slot) with
  t(r), e(r), a(r); h_r = W1^T x_t(r) + b1, z_r = phi(h_r),
  o_r = W2^T z_r + b2, y_t = sum_{r: t(r)=t} a(r) o_r.
* same page, "moe_align_block_size": flatten (token, slot) items, sort them
  by expert, pad each expert's count up to BLOCK_SIZE_M; outputs
  sorted_token_ids, expert_ids per M-block, num_tokens_post_padded.
* same page, "apply_moe_activation" / SiLU-and-mul: the activation of the
  2I-wide first projection is SiLU(gate) * up.
* "MindIE-SD Fused MoE" page, parameter table and "路由选择" (routing)
  section: softmax / sigmoid scores, renormalize (softmax only; sigmoid
  weights are always normalised), grouped routing (group_count groups,
  group score = max (mode 0) or top-2 sum (mode 1), keep k_group groups,
  then top-k inside them), routed_scaling_factor applied in the expert
  selection stage; w13 [E, H, 2I] fused gate/up, w2 [E, I, H].
* same page, "自定义 routing function" example: softmax -> topk -> divide
  by the sum of the selected weights when renormalize is set.
* "vLLM FusedMoEModularKernel" page, Introduction: the Batched activation
  format (num_experts, max_tokens, K) with expert_num_tokens, where not
  every row is valid.

Readings where the pages are silent:

* w13 columns [0, I) are the gate half and [I, 2I) the up half.
* b13 is added to both halves before SiLU-and-mul; b2 is added per routed
  item before the routing weight multiplies it.
* Top-k is the exact-arithmetic TopK of p.  softmax (per row) and sigmoid
  are strictly increasing in the logit, so that order is the order of the
  logits themselves; ties (equal logits) go to the lower expert id, and the
  selected ids are listed by descending score.
* Group scores are taken on the post-activation scores p; mode 0 (max) is
  again ordered by the group's largest logit, mode 1 (sum of the two
  largest p) is a sum of transcendentals evaluated in fp64 here; the
  decision margin between the last kept and the first dropped group is
  returned so callers can accept either choice on numerical near-ties.
  Ties between groups go to the lower group id.
* Weights: softmax + renormalize -> p_sel / sum(p_sel); softmax without
  renormalize -> p_sel; sigmoid -> p_sel / sum(p_sel) always; then times
  routed_scaling_factor (renormalise first, then scale).
* Align: sentinel value R (= number of routed items) in padding slots;
  items of one expert in ascending item order; an empty expert gets zero
  slots and zero blocks.
* Batched layout: out[e, i] = row_weight[e, i] * f_e(x[e, i]) for
  i < expert_num_tokens[e] (row_weight = 1 if absent); other rows are not
  defined.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "e4m3_round", "quantize_rows_e4m3", "bf16_round", "forward_fp8",
    "quantize_groups_e4m3", "forward_fp8_block",
    "unpack_nibbles", "mx_decode", "ue8m0_scale", "dequant_int", "dequant_mx",
    "forward_wq",
    "router_logits", "scores", "group_mask", "topk_select", "route_weights", "route",
    "route_with_groups", "align", "silu", "expert_ffn", "forward",
    "token_output", "forward_batched", "moe_layer",
]


# --------------------------------------------------------------------------
# Router (FlagDoc fused_moe.py 分析, section 1.1: s_t = W_g^T x_t + b_g)
# --------------------------------------------------------------------------

def router_logits(x, w_gate, b_gate=None):
    """s = x W_g + b_g with W_g stored [H, E] (d x E on the page) and b_g [E]."""
    s = np.asarray(x, dtype=np.float64) @ np.asarray(w_gate, dtype=np.float64)
    if b_gate is not None:
        s = s + np.asarray(b_gate, dtype=np.float64)
    return s


# --------------------------------------------------------------------------
# Routing (MindIE-SD Fused MoE: parameter table and routing section;
# FlagGems analysis section 1.1: p_t = softmax(s_t), S_t = TopK(p_t, k))
# --------------------------------------------------------------------------

def scores(logits: np.ndarray, method: str) -> np.ndarray:
    """p = softmax(l) over the expert axis, or p = sigmoid(l) elementwise."""
    l = np.asarray(logits, dtype=np.float64)
    if method == "softmax":
        shifted = l - l.max(axis=-1, keepdims=True)
        ex = np.exp(shifted)
        return ex / ex.sum(axis=-1, keepdims=True)
    if method == "sigmoid":
        with np.errstate(over="ignore"):
            return 1.0 / (1.0 + np.exp(-l))
    raise ValueError(f"unknown routing method {method!r}")


def group_mask(logits: np.ndarray, p: np.ndarray, k_group: int, group_count: int,
               group_select_mode: int):
    """Grouped pre-selection.  Experts are split into group_count equal,
    contiguous groups; each group is scored (mode 0: its largest p; mode 1:
    the sum of its two largest p); the k_group best groups are kept (ties to
    the lower group id).  Returns (allowed [M,E] bool, margin [M]) where
    margin is the score gap between the last kept and the first dropped
    group (inf when nothing is dropped)."""
    l = np.asarray(logits, dtype=np.float64)
    M, E = p.shape
    if group_count <= 1:
        return np.ones((M, E), dtype=bool), np.full(M, np.inf)
    gs = E // group_count
    lg = l.reshape(M, group_count, gs)
    pg = p.reshape(M, group_count, gs)
    if group_select_mode == 0:
        # max p of the group == p of the group's largest logit (monotone).
        key = lg.max(axis=2)
        gscore = pg.max(axis=2)
    elif group_select_mode == 1:
        top2 = np.sort(pg, axis=2)[:, :, -2:]
        gscore = top2[:, :, 0] + top2[:, :, 1]
        key = gscore
    else:
        raise ValueError("group_select_mode must be 0 or 1")
    order = np.argsort(-key, axis=1, kind="stable")       # ties -> lower group id
    kept = order[:, :k_group]
    gmask = np.zeros((M, group_count), dtype=bool)
    np.put_along_axis(gmask, kept, True, axis=1)
    if k_group < group_count and group_select_mode == 1:
        s = np.take_along_axis(gscore, order, axis=1)
        margin = s[:, k_group - 1] - s[:, k_group]
    else:
        # mode 0 is decided exactly on the logits: no numerical near-tie.
        margin = np.full(M, np.inf)
    allowed = np.repeat(gmask, gs, axis=1)
    return allowed, margin


def topk_select(logits: np.ndarray, allowed: np.ndarray, top_k: int) -> np.ndarray:
    """TopK of p restricted to allowed experts, by descending score with ties
    to the lower expert id.  Ordered by the logits (p is strictly increasing
    in the logit for both scoring functions)."""
    l = np.asarray(logits, dtype=np.float64)
    masked = np.where(allowed, l, -np.inf)
    order = np.argsort(-masked, axis=1, kind="stable")
    return order[:, :top_k]


def route_weights(p: np.ndarray, ids: np.ndarray, method: str, renormalize: bool,
                  routed_scaling_factor: float) -> np.ndarray:
    w = np.take_along_axis(p, ids, axis=1)
    if method == "sigmoid" or renormalize:
        w = w / w.sum(axis=1, keepdims=True)
    return w * float(routed_scaling_factor)


def route(logits, top_k: int, method: str = "softmax", renormalize: bool = False,
          k_group: int = 1, group_count: int = 1, group_select_mode: int = 0,
          routed_scaling_factor: float = 1.0):
    """Returns (topk_weights [M,k] f64, topk_ids [M,k] int32, group_margin [M])."""
    l = np.asarray(logits, dtype=np.float64)
    p = scores(l, method)
    allowed, margin = group_mask(l, p, k_group, group_count, group_select_mode)
    ids = topk_select(l, allowed, top_k)
    w = route_weights(p, ids, method, renormalize, routed_scaling_factor)
    return w, ids.astype(np.int32), margin


def route_with_groups(logits_row, groups, top_k: int, method: str, renormalize: bool,
                      group_count: int, routed_scaling_factor: float):
    """Routing of ONE token with the kept groups given explicitly.  Used to
    list every valid answer for a token whose group decision is a numerical
    near-tie (several results are correct there)."""
    l = np.asarray(logits_row, dtype=np.float64)[None, :]
    p = scores(l, method)
    E = l.shape[1]
    gs = E // group_count
    allowed = np.zeros((1, E), dtype=bool)
    for g in groups:
        allowed[0, g * gs:(g + 1) * gs] = True
    ids = topk_select(l, allowed, top_k)
    w = route_weights(p, ids, method, renormalize, routed_scaling_factor)
    return w[0], ids[0].astype(np.int32)


# --------------------------------------------------------------------------
# Align / permute (FlagGems analysis, "moe_align_block_size")
# --------------------------------------------------------------------------

def align(topk_ids, E: int, block_m: int):
    """Returns dict with expert_num_tokens [E], expert_offsets [E+1] (padded,
    exclusive scan), sorted_token_ids [offsets[E]] (item index r = t*k + j,
    sentinel R in padding), block_expert_ids [offsets[E] / block_m]."""
    ids = np.asarray(topk_ids).reshape(-1).astype(np.int64)
    R = ids.size
    if R and (ids.min() < 0 or ids.max() >= E):
        raise ValueError("expert id out of range")
    counts = np.array([(ids == e).sum() for e in range(E)], dtype=np.int64)
    padded = np.array([-(-int(c) // block_m) * block_m for c in counts], dtype=np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(padded)
    sorted_ids = np.full(int(offsets[E]), R, dtype=np.int64)
    blocks = []
    for e in range(E):
        members = np.flatnonzero(ids == e)              # ascending item order
        sorted_ids[offsets[e]:offsets[e] + members.size] = members
        blocks += [e] * int(padded[e] // block_m)
    return {
        "expert_num_tokens": counts.astype(np.int32),
        "expert_offsets": offsets.astype(np.int32),
        "sorted_token_ids": sorted_ids.astype(np.int32),
        "block_expert_ids": np.array(blocks, dtype=np.int32),
        "num_tokens_post_padded": int(offsets[E]),
    }


# --------------------------------------------------------------------------
# Expert FFN and combine (FlagGems analysis sections 1.1 and 1.2)
# --------------------------------------------------------------------------

def silu(u):
    """SiLU(u) = u * sigmoid(u) = u / (1 + exp(-u))."""
    u = np.asarray(u, dtype=np.float64)
    with np.errstate(over="ignore"):
        return u / (1.0 + np.exp(-u))


def expert_ffn(x_rows, w13_e, w2_e, b13_e=None, b2_e=None, z_scale=None):
    """f_e for a stack of rows: h = x W13_e + b13_e (2I wide), z = SiLU(h[:, :I])
    * h[:, I:], o = z W2_e + b2_e.  Weights are stored [H, 2I] and [I, H].
    z_scale (one scalar per row), if given, multiplies z before W2."""
    x_rows = np.asarray(x_rows, dtype=np.float64)
    I = w2_e.shape[0]
    h = x_rows @ w13_e
    if b13_e is not None:
        h = h + b13_e
    z = silu(h[:, :I]) * h[:, I:]
    if z_scale is not None:
        z = z * np.asarray(z_scale, dtype=np.float64)[:, None]
    o = z @ w2_e
    if b2_e is not None:
        o = o + b2_e
    return o


def forward(x, topk_weights, topk_ids, w13, w2, w13_bias=None, w2_bias=None,
            apply_router_weight_on_input=False, expert_map=None):
    """y_t = sum_j a(t, j) * f_{ids[t, j]}(x_t), evaluated expert by expert over
    the routed items (t, j) that name that expert.

    apply_router_weight_on_input (FlagDoc section 1.2, the switch of the same
    name): a(r) multiplies the input z_r of the second linear layer instead
    of its output, o_r = W2^T (a z_r) + b2 and y_t = sum_r o_r.  By linearity
    this equals the default when b2 = 0.

    expert_map ("expert_map" of the FlagDoc kernel, expert parallelism):
    global expert id -> index of that expert in the given (local) weights, or
    -1 for an expert held elsewhere; items routed there contribute nothing."""
    x = np.asarray(x, dtype=np.float64)
    a = np.asarray(topk_weights, dtype=np.float64)
    ids = np.asarray(topk_ids)
    if expert_map is not None:
        ids = np.asarray(expert_map)[ids]
    M, H = x.shape
    E = w13.shape[0]
    y = np.zeros((M, H), dtype=np.float64)
    for e in range(E):
        t, j = np.nonzero(ids == e)
        if t.size == 0:
            continue
        b13 = None if w13_bias is None else w13_bias[e]
        b2 = None if w2_bias is None else w2_bias[e]
        if apply_router_weight_on_input:
            np.add.at(y, t, expert_ffn(x[t], w13[e], w2[e], b13, b2, z_scale=a[t, j]))
        else:
            np.add.at(y, t, a[t, j][:, None] * expert_ffn(x[t], w13[e], w2[e], b13, b2))
    return y


def token_output(x_t, weights_t, ids_t, w13, w2, w13_bias=None, w2_bias=None):
    """y for one token, from its own routed items only (for sampled checks at
    sizes where the whole forward is too slow).  Weight tensors may be given
    as a mapping expert id -> array for just the experts this token uses."""
    x_t = np.asarray(x_t, dtype=np.float64)[None, :]
    y = None
    for a, e in zip(weights_t, ids_t):
        e = int(e)
        o = expert_ffn(x_t, w13[e], w2[e],
                       None if w13_bias is None else w13_bias[e],
                       None if w2_bias is None else w2_bias[e])[0]
        y = float(a) * o if y is None else y + float(a) * o
    return y


def forward_batched(x_b, expert_num_tokens, w13, w2, w13_bias=None, w2_bias=None,
                    row_weight=None):
    """Batched layout: out[e, i] = row_weight[e, i] * f_e(x_b[e, i]) for the
    valid rows i < expert_num_tokens[e].  Returns a list of E arrays, one
    [count_e, H] array per expert (invalid rows have no defined output)."""
    E = x_b.shape[0]
    outs = []
    for e in range(E):
        c = int(expert_num_tokens[e])
        rows = np.asarray(x_b[e, :c], dtype=np.float64)
        o = expert_ffn(rows, w13[e], w2[e],
                       None if w13_bias is None else w13_bias[e],
                       None if w2_bias is None else w2_bias[e])
        if row_weight is not None:
            o = o * np.asarray(row_weight[e, :c], dtype=np.float64)[:, None]
        outs.append(o)
    return outs


def moe_layer(x, logits, w13, w2, top_k, method="softmax", renormalize=False,
              k_group=1, group_count=1, group_select_mode=0, routed_scaling_factor=1.0,
              w13_bias=None, w2_bias=None):
    """Route, then forward: the whole layer from router logits to y."""
    w, ids, margin = route(logits, top_k, method, renormalize, k_group, group_count,
                           group_select_mode, routed_scaling_factor)
    return forward(x, w, ids, w13, w2, w13_bias, w2_bias), w, ids, margin


# --------------------------------------------------------------------------
# FP8 W8A8 (FlagDoc fused_moe.py 分析, "FP8 W8A8" and "数据类型与量化辅助":
# activations quantised to FP8 before each GEMM; the kernel multiplies the
# FP8 dot product by the activation scale and the weight scale)
# --------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_round(v):
    """Round float32 values to the nearest FP8 E4M3 value (1 sign, 4 exponent
    bits with bias 7, 3 mantissa bits, no infinities, largest finite 448),
    ties to even, saturating to +-448.  Returns the rounded values as fp64.
    Normal binades [2^e, 2^(e+1)) for e in [-6, 8] have spacing 2^(e-3);
    below 2^-6 the subnormal spacing is 2^-9."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.clip(e, -6, 8)
    step = np.exp2(e - 3)
    q = np.round(a / step) * step        # numpy rounds half to even
    q = np.minimum(q, E4M3_MAX)
    return np.sign(v) * q


def quantize_rows_e4m3(x):
    """Dynamic per-row (per-token) FP8 quantisation: scale = max|row| / 448
    (1 for an all-zero row), q = e4m3(x / scale); the division and the scale
    are taken in fp32 (the decision that picks each code is made in the
    precision of the kernel).  Returns (q as fp64 values, scale as fp64)."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.abs(x32).max(axis=1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    q = e4m3_round(x32 / scale[:, None])
    return q, scale.astype(np.float64)


def quantize_groups_e4m3(x, group=128):
    """Per-(row, group of `group` consecutive columns) FP8 quantisation: each
    group is quantised as its own row by quantize_rows_e4m3.  Returns (q as
    fp64 values [M, K], scale [M, K / group] as fp64)."""
    x32 = np.asarray(x, dtype=np.float32)
    M, K = x32.shape
    G = K // group
    q, s = quantize_rows_e4m3(x32.reshape(M * G, group))
    return q.reshape(M, K), s.reshape(M, G)


def forward_fp8_block(x, topk_weights, topk_ids, w13_q, w2_q, w13_scale, w2_scale,
                      w13_bias=None, w2_bias=None, block=128):
    """The FP8 W8A8 layer with block-wise scales ("fused_moe.py 分析", "FP8 W8A8",
    block-wise: within each K block the dot product of the FP8 codes is
    multiplied by that block's activation scale and weight scale, and the
    blocks are summed).  Weight scales [E, K/128, N/128] (128 x 128 blocks);
    activations quantised per (row, group of 128 along K), z as held in bf16
    (see forward_fp8):
        h[r, n] = sum_b (q_x[r, b] . W13q[b, n]) * s_x[r, b] * s_w13[b, n // 128]."""
    x = np.asarray(x, dtype=np.float64)
    a = np.asarray(topk_weights, dtype=np.float64)
    ids = np.asarray(topk_ids)
    M, H = x.shape
    E = w13_q.shape[0]
    I = w2_q.shape[1]
    y = np.zeros((M, H), dtype=np.float64)
    qx, sx = quantize_groups_e4m3(x, block)

    def block_gemm(q, s, wq, ws):
        K, N = wq.shape
        out = np.zeros((q.shape[0], N), dtype=np.float64)
        for b in range(K // block):
            ks = slice(b * block, (b + 1) * block)
            part = q[:, ks] @ np.asarray(wq[ks], dtype=np.float64)       # exact in fp64
            col_scale = np.repeat(np.asarray(ws[b], dtype=np.float64), block)[:N]
            out += part * s[:, b][:, None] * col_scale
        return out

    for e in range(E):
        t, j = np.nonzero(ids == e)
        if t.size == 0:
            continue
        h = block_gemm(qx[t], sx[t], w13_q[e], w13_scale[e])
        if w13_bias is not None:
            h = h + w13_bias[e]
        z = silu(h[:, :I]) * h[:, I:]
        qz, sz = quantize_groups_e4m3(bf16_round(z), block)
        o = block_gemm(qz, sz, w2_q[e], w2_scale[e])
        if w2_bias is not None:
            o = o + w2_bias[e]
        np.add.at(y, t, a[t, j][:, None] * o)
    return y


def bf16_round(v):
    """Round to bfloat16 (nearest, ties to even) via float32, as fp64."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32))
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def forward_fp8(x, topk_weights, topk_ids, w13_q, w2_q, w13_scale, w2_scale,
                w13_bias=None, w2_bias=None):
    """The FP8 W8A8 layer.  Weights are FP8 values w_q with scales per expert
    ([E]) or per output channel ([E, 2I] / [E, H]); each routed row is
    quantised per row before GEMM1 (x) and before GEMM2 (z):
        h = (q_x W13q) * s_x * s_w13 + b13,  z = SiLU(h_gate) * h_up,
        o = (q_z W2q) * s_z * s_w2 + b2,     y_t = sum_j a(t, j) o.
    The second quantisation reads z as held between the GEMMs, in the
    compute dtype (bf16): on the FlagDoc page the activation output
    (intermediate_cache2) is stored in compute_type and that is what
    moe_kernel_quantize_input quantises for the w2 GEMM.  Dot products of the
    FP8 values are exact in fp64."""
    x = np.asarray(x, dtype=np.float64)
    a = np.asarray(topk_weights, dtype=np.float64)
    ids = np.asarray(topk_ids)
    M, H = x.shape
    E = w13_q.shape[0]
    I = w2_q.shape[1]
    y = np.zeros((M, H), dtype=np.float64)
    qx, sx = quantize_rows_e4m3(x)
    for e in range(E):
        t, j = np.nonzero(ids == e)
        if t.size == 0:
            continue
        s13 = np.asarray(w13_scale[e], dtype=np.float64)
        s2 = np.asarray(w2_scale[e], dtype=np.float64)
        h = (qx[t] @ np.asarray(w13_q[e], dtype=np.float64)) * sx[t][:, None] * s13
        if w13_bias is not None:
            h = h + w13_bias[e]
        z = silu(h[:, :I]) * h[:, I:]
        qz, sz = quantize_rows_e4m3(bf16_round(z))
        o = (qz @ np.asarray(w2_q[e], dtype=np.float64)) * sz[:, None] * s2
        if w2_bias is not None:
            o = o + w2_bias[e]
        np.add.at(y, t, a[t, j][:, None] * o)
    return y



# --------------------------------------------------------------------------
# Weight-only quantised experts.  FlagDoc fused_moe.py 分析, "WNA16 路径" and
# "5. 特殊量化格式处理": int8 / int4 weights with a group scale and a zero
# point, and OCP MX weights, are dequantised to the activation dtype
# (hidden_states.dtype, bf16 here) and the layer then runs as the ordinary
# one.  Layouts (the pages fix none; GPTQ/AWQ-style group quantisation
# along K in the [E, K, N] orientation of the bf16 weights):
#   int4 / fp4 codes  uint8 [E, K, N/2]: byte j of a row holds column 2j in
#                     its low nibble and column 2j+1 in its high nibble
#   int8 codes        int8 [E, K, N]
#   int scales        [E, K/G, N] (group of G rows of K per scale), zero
#                     points [E, K/G, N] in the code domain (int4: 0..15,
#                     int8: -128..127) or absent (int4: 8, int8: 0)
#   MX scales         uint8 UE8M0 [E, K/32, N]: 2^(s - 127), one per block
#                     of 32 elements along K (OCP MX: block size 32)
# --------------------------------------------------------------------------

def unpack_nibbles(packed):
    """uint8 [..., N/2] -> int64 [..., N]: column 2j = low nibble of byte j,
    column 2j+1 = its high nibble."""
    b = np.asarray(packed, dtype=np.uint8).astype(np.int64)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.int64)
    out[..., 0::2] = b & 0xF
    out[..., 1::2] = b >> 4
    return out


# OCP Microscaling formats (OCP MX v1.0): element formats with their bit
# fields (sign, exponent bits, mantissa bits, exponent bias); no inf/NaN.
MX_FORMATS = {"e2m1": (2, 1, 1), "e3m2": (3, 2, 3), "e2m3": (2, 3, 1)}


def mx_decode(codes, fmt):
    """Value of each MX element code: sign bit above an ebits exponent field
    and an mbits mantissa field; exponent field 0 is subnormal
    (m / 2^mbits * 2^(1 - bias)), otherwise 2^(e - bias) * (1 + m / 2^mbits)."""
    ebits, mbits, bias = MX_FORMATS[fmt]
    c = np.asarray(codes, dtype=np.int64)
    sign = np.where((c >> (ebits + mbits)) & 1, -1.0, 1.0)
    e = (c >> mbits) & ((1 << ebits) - 1)
    m = (c & ((1 << mbits) - 1)).astype(np.float64)
    mag = np.where(e == 0, m / (1 << mbits) * 2.0 ** (1 - bias),
                   2.0 ** (e.astype(np.float64) - bias) * (1.0 + m / (1 << mbits)))
    return sign * mag


def ue8m0_scale(s):
    """UE8M0 block scale: 2^(s - 127) (s = 255, NaN, is not used)."""
    return np.exp2(np.asarray(s, dtype=np.float64) - 127.0)


def dequant_int(q, scale, zero=None, bits=4):
    """Group dequantisation to the activation dtype:
        w[e, k, n] = bf16((q[e, k, n] - zero[e, k // G, n]) * scale[e, k // G, n])
    with G = K / scale.shape[1].  q: int4 codes packed as above (bits=4) or
    int8 codes (bits=8); zero absent = 8 (int4) or 0 (int8)."""
    codes = unpack_nibbles(q) if bits == 4 else np.asarray(q, dtype=np.int64)
    E, K, N = codes.shape
    sc = np.asarray(scale, dtype=np.float64)
    G = K // sc.shape[1]
    if zero is None:
        zp = np.full(sc.shape, 8 if bits == 4 else 0, dtype=np.int64)
    else:
        zp = np.asarray(zero, dtype=np.int64)
    kg = np.arange(K) // G
    return bf16_round((codes - zp[:, kg, :]).astype(np.float64) * sc[:, kg, :])


def dequant_mx(q, scale, fmt="e2m1"):
    """MX dequantisation to the activation dtype:
        w[e, k, n] = bf16(value(q[e, k, n]) * 2^(scale[e, k // 32, n] - 127)).
    q: E2M1 codes packed two per byte (fmt "e2m1"), or one 6-bit code per
    byte (fmt "e3m2" / "e2m3")."""
    codes = unpack_nibbles(q) if fmt == "e2m1" else np.asarray(q, dtype=np.int64)
    K = codes.shape[1]
    kb = np.arange(K) // 32
    s = ue8m0_scale(np.asarray(scale))
    return bf16_round(mx_decode(codes, fmt) * s[:, kb, :])


def forward_wq(x, topk_weights, topk_ids, w13_deq, w2_deq, w13_bias=None, w2_bias=None):
    """The weight-only quantised layer: the ordinary layer on the dequantised
    weights (dequant_int / dequant_mx of w13 and w2)."""
    return forward(x, topk_weights, topk_ids, w13_deq, w2_deq, w13_bias, w2_bias)
