"""Comparison helpers shared by the GPU parity tests (test code only)."""
import itertools

import numpy as np
import torch

import oracle
from mixture_experts_ffn_softmax_gb300 import workloads as wl

# Tolerances stated for the fused MoE forward: ids / permutation / counts /
# padding bit-exact; topk_weights within 1e-5 absolute; outputs (bf16 in,
# fp32 accumulate) within relative L2 <= 1e-2 and max abs <= 5e-2 * RMS.
WEIGHT_ATOL = 1e-5
OUT_REL_L2 = 1e-2
OUT_MAXABS_RMS = 5e-2
# Group mode 1 compares sums of transcendentals: the GPU takes that decision
# in fp32, the oracle in fp64.  Tokens whose two candidate group scores lie
# closer than this may go either way (both answers are checked for validity).
GROUP_TIE_TOL = 4e-6


def route_args(spec):
    return dict(top_k=spec.top_k, method=spec.routing_method, renormalize=spec.renormalize,
                k_group=spec.k_group, group_count=spec.group_count,
                group_select_mode=spec.group_select_mode,
                routed_scaling_factor=spec.routed_scaling_factor)


def _alternatives(l_row, a):
    """All valid (weights, ids) of one token whose kept-group decision is a
    near-tie: every k_group-subset that keeps all clearly-better groups."""
    G, kg = a["group_count"], a["k_group"]
    p = oracle.scores(l_row[None, :], a["method"])[0]
    E = l_row.size
    gs = E // G
    pg = np.sort(p.reshape(G, gs), axis=1)
    gscore = pg[:, -1] + pg[:, -2]
    order = np.argsort(-gscore, kind="stable")
    boundary = gscore[order[kg - 1]]
    sure = [g for g in range(G) if gscore[g] > boundary + GROUP_TIE_TOL]
    maybe = [g for g in range(G) if abs(gscore[g] - boundary) <= GROUP_TIE_TOL]
    alts = []
    for extra in itertools.combinations(maybe, kg - len(sure)):
        alts.append(oracle.route_with_groups(l_row, list(sure) + list(extra), a["top_k"],
                                             a["method"], a["renormalize"], G,
                                             a["routed_scaling_factor"]))
    return alts


def check_route(logits_np, gpu_w, gpu_ids, a):
    """Compares GPU routing with the oracle.  Returns the number of tokens
    accepted as numerical group near-ties."""
    w, ids, margin = oracle.route(logits_np, a["top_k"], a["method"], a["renormalize"],
                                  a["k_group"], a["group_count"], a["group_select_mode"],
                                  a["routed_scaling_factor"])
    gpu_ids = np.asarray(gpu_ids)
    gpu_w = np.asarray(gpu_w, dtype=np.float64)
    bad = np.flatnonzero((gpu_ids != ids).any(axis=1))
    ties = 0
    for t in bad:
        assert 0 < margin[t] < GROUP_TIE_TOL, (
            f"token {t}: ids {gpu_ids[t].tolist()} != oracle {ids[t].tolist()} "
            f"(group margin {margin[t]:.3g})")
        alts = _alternatives(np.asarray(logits_np[t], dtype=np.float64), a)
        match = [aw for aw, aid in alts if aid.tolist() == gpu_ids[t].tolist()]
        assert match, f"token {t}: GPU ids {gpu_ids[t].tolist()} are not a valid near-tie answer"
        w[t] = match[0]
        ties += 1
    err = np.abs(gpu_w - w).max() if w.size else 0.0
    assert err <= WEIGHT_ATOL, f"topk_weights max abs error {err:.3g} > {WEIGHT_ATOL}"
    return ties


def check_out(out, ref, what=""):
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(out).all(), f"{what}: non-finite output"
    nrm = np.linalg.norm(ref)
    rel = np.linalg.norm(out - ref) / max(nrm, 1e-30)
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    mx = np.abs(out - ref).max() if ref.size else 0.0
    assert rel <= OUT_REL_L2, f"{what}: relative L2 {rel:.3g} > {OUT_REL_L2}"
    assert mx <= OUT_MAXABS_RMS * rms, f"{what}: max abs {mx:.3g} > {OUT_MAXABS_RMS} * RMS {rms:.3g}"
    return rel, mx / max(rms, 1e-30)


def covering_tokens(ids, n_random, rng, block_m=128):
    """Token sample for full-size parity: for every expert that receives
    items, the tokens of its first item, of the first item of its last
    block_m-row block and of its last item (items of one expert sit in
    ascending item order r = t * top_k + j in the sorted layout, so these
    reach the first and the last row block of every expert's GEMM tiles),
    plus n_random tokens drawn at random.  Returns sorted token indices."""
    ids = np.asarray(ids)
    M, k = ids.shape
    flat = ids.reshape(-1)
    order = np.argsort(flat, kind="stable")
    bounds = np.searchsorted(flat[order], np.arange(flat.max() + 2))
    sel = set()
    for e in range(flat.max() + 1):
        items = order[bounds[e]:bounds[e + 1]]
        if items.size == 0:
            continue
        for pos in (0, (items.size - 1) // block_m * block_m, items.size - 1):
            sel.add(int(items[pos]) // k)
    sel.update(int(t) for t in rng.choice(M, size=min(M, n_random), replace=False))
    return np.array(sorted(sel))


class LazyF64:
    """Indexable view of a (possibly device, bf16) weight tensor that widens one
    expert at a time to float64 on the host, so full-size layers never need a
    full fp64 copy."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)
        self._cache = {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self._cache:
            if len(self._cache) > 4:
                self._cache.clear()
            self._cache[e] = wl.to_f64(self.t[e])
        return self._cache[e]


def f64(t):
    return None if t is None else wl.to_f64(t)


def sync():
    torch.cuda.synchronize()
