"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here calls the CUDA path.  Each test ties the oracle to something
other than itself: hand-derived closed forms (tests/golden), brute force
over all subsets on tiny inputs, library routines in special cases the
method reduces to, and invariants of the definition.  The mutation tests at
the end plant plausible mistakes in the oracle and check that some pin fails.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import moe_oracle as om

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- golden ---

def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def _golden_route_cases(golden_dir):
    return _load(golden_dir, "route_cases.json")["cases"]


def test_route_golden(golden_dir):
    for c in _golden_route_cases(golden_dir):
        logits = np.array([[math.log(q) for q in c["logits_ln"]]], dtype=np.float32)
        w, ids, _ = oracle.route(logits, c["top_k"], c["method"], c["renormalize"],
                                 c["k_group"], c["group_count"], c["group_select_mode"],
                                 c["scale"])
        assert ids[0].tolist() == c["ids"], c["name"]
        np.testing.assert_allclose(w[0], c["weights"], rtol=0, atol=2e-7, err_msg=c["name"])


def test_align_golden(golden_dir):
    for c in _load(golden_dir, "align_cases.json")["cases"]:
        a = oracle.align(np.array(c["topk_ids"], dtype=np.int32), c["E"], c["block_m"])
        for key in ("expert_num_tokens", "expert_offsets", "sorted_token_ids",
                    "block_expert_ids"):
            assert a[key].tolist() == c[key], (c["name"], key)


# ------------------------------------------------------------ brute force ---

def _brute_route(l_row, top_k, method, renormalize, k_group, G, mode, scale,
                 group_tol=0.0):
    """Enumerate every group subset and every expert subset.  The best set is
    the one with the largest score sum; among equal sums the lexicographically
    smallest sorted id list wins.  Sums are taken over the sorted values so
    equal multisets give bit-equal sums.  With group_tol > 0 every group subset
    whose total is within group_tol of the best is also answered (a list of
    (weights, ids) is returned): mode 1 has exact mathematical ties such as
    sigmoid(a) + sigmoid(-a) = 1 that floating point breaks either way."""
    E = len(l_row)
    if method == "softmax":
        ex = [math.exp(v - max(l_row)) for v in l_row]
        tot = math.fsum(ex)
        p = [v / tot for v in ex]
    else:
        p = [1.0 / (1.0 + math.exp(-v)) for v in l_row]
    gs = E // G
    if G > 1:
        gscore = []
        for g in range(G):
            members = list(range(g * gs, (g + 1) * gs))
            if mode == 0:
                gscore.append(max(p[e] for e in members))
            else:
                gscore.append(max(sum(sorted((p[a], p[b])))
                                  for a, b in itertools.combinations(members, 2)))
        best = None
        subs = list(itertools.combinations(range(G), k_group))
        for gsub in subs:
            key = (-sum(sorted(gscore[g] for g in gsub)), gsub)
            if best is None or key < best:
                best = key
        if group_tol > 0:
            return [_brute_route_in(p, [e for g in gsub for e in range(g * gs, (g + 1) * gs)],
                                    top_k, method, renormalize, scale)
                    for gsub in subs
                    if -sum(sorted(gscore[g] for g in gsub)) - best[0] <= group_tol]
        allowed = [e for g in best[1] for e in range(g * gs, (g + 1) * gs)]
    else:
        allowed = list(range(E))
    if group_tol > 0:
        return [_brute_route_in(p, allowed, top_k, method, renormalize, scale)]
    return _brute_route_in(p, allowed, top_k, method, renormalize, scale)


def _brute_route_in(p, allowed, top_k, method, renormalize, scale):
    best = None
    for sub in itertools.combinations(sorted(allowed), top_k):
        key = (-sum(sorted(p[e] for e in sub)), sub)
        if best is None or key < best:
            best = key
    chosen = sorted(best[1], key=lambda e: (-p[e], e))
    w = [p[e] for e in chosen]
    if method == "sigmoid" or renormalize:
        s = math.fsum(w)
        w = [v / s for v in w]
    return [scale * v for v in w], chosen


@pytest.mark.parametrize("seed", range(6))
def test_route_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    n_cases = 0
    for E, G in ((4, 1), (6, 1), (6, 2), (6, 3), (8, 2), (8, 4)):
        for method in ("softmax", "sigmoid"):
            for mode in ((0, 1) if G > 1 else (0,)):
                if mode == 1 and E // G < 2:
                    continue
                for k_group in range(1, G + 1):
                    kmax = min(3, k_group * (E // G))
                    for top_k in range(1, kmax + 1):
                        # small integer logits -> many exact ties
                        l = rng.integers(-2, 3, size=(4, E)).astype(np.float32)
                        for renorm in (False, True):
                            scale = 1.0 if renorm else 2.5
                            w, ids, _ = oracle.route(l, top_k, method, renorm, k_group, G,
                                                     mode, scale)
                            for t in range(l.shape[0]):
                                row = [float(v) for v in l[t]]
                                bw, bids = _brute_route(row, top_k, method, renorm, k_group,
                                                        G, mode, scale)
                                if ids[t].tolist() != bids and mode == 1:
                                    # only a group-score tie within rounding may differ
                                    alts = _brute_route(row, top_k, method, renorm, k_group,
                                                        G, mode, scale, group_tol=1e-12)
                                    match = [a for a in alts if a[1] == ids[t].tolist()]
                                    assert match, (E, G, method, mode, top_k, l[t])
                                    bw, bids = match[0]
                                assert ids[t].tolist() == bids, (E, G, method, mode, top_k, l[t])
                                np.testing.assert_allclose(w[t], bw, rtol=1e-12, atol=1e-14)
                                n_cases += 1
    assert n_cases > 200


def _brute_best_groups(l_row, method, k_group, G, mode):
    """The kept group subset by enumeration (largest summed group score, ties
    to the lexicographically smallest subset), scored as in _brute_route."""
    E = len(l_row)
    if method == "softmax":
        ex = [math.exp(v - max(l_row)) for v in l_row]
        tot = math.fsum(ex)
        p = [v / tot for v in ex]
    else:
        p = [1.0 / (1.0 + math.exp(-v)) for v in l_row]
    gs = E // G
    gscore = []
    for g in range(G):
        members = range(g * gs, (g + 1) * gs)
        if mode == 0:
            gscore.append(max(p[e] for e in members))
        else:
            gscore.append(max(p[a] + p[b] for a, b in itertools.combinations(members, 2)))
    best = min(itertools.combinations(range(G), k_group),
               key=lambda s: (-sum(sorted(gscore[g] for g in s)), s))
    return p, list(best)


@pytest.mark.parametrize("seed", range(3))
def test_route_with_groups_brute_force(seed):
    """MindIE-SD "Fused MoE", 路由选择 (grouped selection): once the kept
    groups are fixed, the result is the top-k over exactly those groups'
    experts.  For EVERY k_group-subset of groups, route_with_groups must equal
    enumeration of all top_k-subsets of that subset's experts (so a wrong
    group-to-expert index map or a mask over the wrong groups fails), and
    with the subset that enumeration of the group choice keeps it must equal
    route() itself."""
    rng = np.random.default_rng(300 + seed)
    n_cases = 0
    for E, G in ((6, 2), (6, 3), (8, 2), (8, 4), (12, 4)):
        gs = E // G
        for method in ("softmax", "sigmoid"):
            for k_group in range(1, G + 1):
                for top_k in range(1, min(3, k_group * gs) + 1):
                    # continuous logits, with a few exact ties planted
                    l = rng.standard_normal((3, E))
                    l[:, rng.integers(0, E)] = l[:, rng.integers(0, E)]
                    for renorm in (False, True):
                        scale = 1.0 if renorm else 2.5
                        for t in range(l.shape[0]):
                            row = [float(v) for v in l[t]]
                            p = _brute_best_groups(row, method, k_group, G, 0)[0]
                            for gsub in itertools.combinations(range(G), k_group):
                                experts = [e for g in gsub for e in range(g * gs, (g + 1) * gs)]
                                bw, bids = _brute_route_in(p, experts, top_k, method,
                                                           renorm, scale)
                                w, ids = oracle.route_with_groups(
                                    l[t], list(gsub), top_k, method, renorm, G, scale)
                                assert ids.tolist() == bids, (E, G, gsub, top_k, l[t])
                                np.testing.assert_allclose(w, bw, rtol=1e-12, atol=1e-14)
                                n_cases += 1
                            for mode in ((0, 1) if gs >= 2 else (0,)):
                                _, kept = _brute_best_groups(row, method, k_group, G, mode)
                                rw, rids, _ = oracle.route(l[t:t + 1], top_k, method, renorm,
                                                           k_group, G, mode, scale)
                                w, ids = oracle.route_with_groups(
                                    l[t], kept, top_k, method, renorm, G, scale)
                                assert ids.tolist() == rids[0].tolist(), (E, G, mode, kept)
                                np.testing.assert_allclose(w, rw[0], rtol=1e-12, atol=1e-14)
    assert n_cases > 500


def test_route_matches_printed_routing_function():
    """Without groups, softmax routing is the page's printed custom routing
    function: softmax over experts, torch.topk, then divide by the sum of the
    selected weights when renormalize is set.  Continuous logits -> no ties."""
    g = torch.Generator().manual_seed(7)
    for E, k in ((8, 2), (16, 4), (128, 8), (256, 8)):
        logits = torch.randn(64, E, generator=g, dtype=torch.float64)
        for renorm in (False, True):
            vals, idx = logits.softmax(dim=-1).topk(k, dim=-1)
            if renorm:
                vals = vals / vals.sum(dim=-1, keepdim=True)
            w, ids, _ = oracle.route(logits.numpy(), k, "softmax", renorm)
            assert (ids == idx.numpy()).all()
            np.testing.assert_allclose(w, vals.numpy(), rtol=1e-12, atol=1e-15)


def test_route_sigmoid_grouped_matches_library_path():
    """Grouped sigmoid routing assembled from library routines (torch.sigmoid,
    torch.topk over groups, masking, torch.topk over experts) on continuous
    logits, mode 1 = sum of torch.topk(2) inside each group."""
    g = torch.Generator().manual_seed(11)
    E, G, kg, k = 256, 8, 4, 8
    logits = torch.randn(128, E, generator=g, dtype=torch.float64)
    p = torch.sigmoid(logits)
    gscore = p.view(128, G, E // G).topk(2, dim=-1).values.sum(-1)
    gidx = gscore.topk(kg, dim=-1).indices
    gmask = torch.zeros(128, G, dtype=torch.bool).scatter_(1, gidx, True)
    pm = p.masked_fill(~gmask.repeat_interleave(E // G, dim=1), -1.0)
    vals, idx = pm.topk(k, dim=-1)
    vals = vals / vals.sum(-1, keepdim=True) * 2.5
    w, ids, _ = oracle.route(logits.numpy(), k, "sigmoid", False, kg, G, 1, 2.5)
    assert (ids == idx.numpy()).all()
    np.testing.assert_allclose(w, vals.numpy(), rtol=1e-12)


# ------------------------------------------------------------------ align ---

@pytest.mark.parametrize("seed", range(4))
def test_align_invariants(seed):
    rng = np.random.default_rng(seed)
    for M, k, E, bm in ((1, 1, 1, 1), (37, 2, 8, 16), (200, 8, 32, 128), (64, 3, 5, 7)):
        ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
        if seed % 2:
            ids[: M // 2] = ids[0]       # skew: many items on the same experts
        a = oracle.align(ids, E, bm)
        R = M * k
        flat = ids.reshape(-1)
        c = a["expert_num_tokens"]
        off = a["expert_offsets"]
        st = a["sorted_token_ids"]
        assert c.sum() == R
        for e in range(E):
            assert off[e + 1] - off[e] == -(-c[e] // bm) * bm
            seg = st[off[e]:off[e + 1]]
            real = seg[seg < R]
            assert real.tolist() == np.flatnonzero(flat == e).tolist()   # ascending, exact set
            assert (seg[c[e]:] == R).all() and (seg[:c[e]] < R).all()
        assert sorted(st[st < R].tolist()) == list(range(R))              # permutation
        assert len(a["block_expert_ids"]) == off[E] // bm
        for b, e in enumerate(a["block_expert_ids"]):
            assert off[e] <= b * bm < off[e + 1]
        # dispatch then combine is the identity (index_select / index_copy)
        x = rng.standard_normal((R, 3))
        disp = x[np.where(st < R, st, 0)]
        back = np.zeros_like(x)
        back[st[st < R]] = disp[st < R]
        assert np.array_equal(back, x)


def test_align_rejects_bad_ids():
    with pytest.raises(ValueError):
        oracle.align(np.array([[0, 4]]), 4, 2)
    with pytest.raises(ValueError):
        oracle.align(np.array([[-1, 0]]), 4, 2)


# -------------------------------------------------------------------- ffn ---

def _closed_form_case():
    """H=2, I=3, E=2 hand-built weights (see the expert formulas below)."""
    H, I, E = 2, 3, 2
    w13 = np.zeros((E, H, 2 * I))
    b13 = np.zeros((E, 2 * I))
    w2 = np.zeros((E, I, H))
    b2 = np.zeros((E, H))
    # expert 0: gate = [x0, x1, x0+x1] + [0, .5, 0]; up = [2 x0, -x1, 0] + [0, 0, 1]
    w13[0, :, :I] = [[1, 0, 1], [0, 1, 1]]
    w13[0, :, I:] = [[2, 0, 0], [0, -1, 0]]
    b13[0] = [0, 0.5, 0, 0, 0, 1]
    # y = [z0 + z2, z1 - z2] + [0.1, -0.2]
    w2[0] = [[1, 0], [0, 1], [1, -1]]
    b2[0] = [0.1, -0.2]
    # expert 1: gate = [-x0, 2 x1, 0]; up = [x1, x0, x0 + x1]; y = [z1 + 2 z2, z0]
    w13[1, :, :I] = [[-1, 0, 0], [0, 2, 0]]
    w13[1, :, I:] = [[0, 1, 1], [1, 0, 1]]
    w2[1] = [[0, 1], [1, 0], [2, 0]]
    return w13, b13, w2, b2


def _s(u):
    return u / (1.0 + math.exp(-u))


def _closed_form_expert(e, x0, x1):
    if e == 0:
        z0 = _s(x0) * (2 * x0)
        z1 = _s(x1 + 0.5) * (-x1)
        z2 = _s(x0 + x1) * 1.0
        return np.array([z0 + z2 + 0.1, z1 - z2 - 0.2])
    z0 = _s(-x0) * x1
    z1 = _s(2 * x1) * x0
    z2 = _s(0.0) * (x0 + x1)
    return np.array([z1 + 2 * z2, z0])


def test_ffn_closed_form():
    w13, b13, w2, b2 = _closed_form_case()
    x = np.array([[1.0, -2.0], [0.5, 3.0]])
    ids = np.array([[1, 0], [0, 1]])
    a = np.array([[0.7, 0.2], [0.25, 0.5]])      # deliberately not summing to 1
    y = oracle.forward(x, a, ids, w13, w2, b13, b2)
    expect = np.stack([
        0.7 * _closed_form_expert(1, 1.0, -2.0) + 0.2 * _closed_form_expert(0, 1.0, -2.0),
        0.25 * _closed_form_expert(0, 0.5, 3.0) + 0.5 * _closed_form_expert(1, 0.5, 3.0),
    ])
    np.testing.assert_allclose(y, expect, rtol=1e-14, atol=1e-14)
    for t in range(2):
        np.testing.assert_allclose(oracle.token_output(x[t], a[t], ids[t], w13, w2, b13, b2),
                                   expect[t], rtol=1e-14, atol=1e-14)


def _dense_swiglu_torch(x, w13, w2, b13, b2):
    """Dense SwiGLU FFN through torch.nn.functional (fp64 CPU)."""
    xt = torch.from_numpy(x)
    I = w2.shape[0]
    gate = torch.nn.functional.linear(xt, torch.from_numpy(w13[:, :I].T.copy()),
                                      torch.from_numpy(b13[:I]))
    up = torch.nn.functional.linear(xt, torch.from_numpy(w13[:, I:].T.copy()),
                                    torch.from_numpy(b13[I:]))
    z = torch.nn.functional.silu(gate) * up
    return torch.nn.functional.linear(z, torch.from_numpy(w2.T.copy()),
                                      torch.from_numpy(b2)).numpy()


def _rand_layer(rng, E, H, I, bias=True):
    w13 = rng.standard_normal((E, H, 2 * I)) * 0.2
    w2 = rng.standard_normal((E, I, H)) * 0.2
    b13 = rng.standard_normal((E, 2 * I)) * 0.1 if bias else np.zeros((E, 2 * I))
    b2 = rng.standard_normal((E, H)) * 0.1 if bias else np.zeros((E, H))
    return w13, w2, b13, b2


def test_single_expert_is_dense_swiglu():
    """E=1, k=1: softmax of one logit is 1 (renormalised), so the layer is the
    dense SwiGLU FFN."""
    rng = np.random.default_rng(3)
    w13, w2, b13, b2 = _rand_layer(rng, 1, 24, 40)
    x = rng.standard_normal((17, 24))
    logits = rng.standard_normal((17, 1))
    y, w, ids, _ = oracle.moe_layer(x, logits, w13, w2, 1, "softmax", True,
                                    w13_bias=b13, w2_bias=b2)
    assert (ids == 0).all() and np.allclose(w, 1.0)
    np.testing.assert_allclose(y, _dense_swiglu_torch(x, w13[0], w2[0], b13[0], b2[0]),
                               rtol=1e-12, atol=1e-12)


def test_uniform_topk_all_is_mean_of_experts():
    """All logits equal, top_k = E, softmax: weights 1/E, ids 0..E-1 by the tie
    rule, so y = mean over experts of the dense expert outputs."""
    rng = np.random.default_rng(4)
    E, H, I, M = 5, 16, 20, 9
    w13, w2, b13, b2 = _rand_layer(rng, E, H, I)
    x = rng.standard_normal((M, H))
    y, w, ids, _ = oracle.moe_layer(x, np.zeros((M, E)), w13, w2, E, "softmax", False,
                                    w13_bias=b13, w2_bias=b2)
    assert (ids == np.arange(E)).all()
    np.testing.assert_allclose(w, 1.0 / E, rtol=1e-15)
    mean = sum(_dense_swiglu_torch(x, w13[e], w2[e], b13[e], b2[e]) for e in range(E)) / E
    np.testing.assert_allclose(y, mean, rtol=1e-12, atol=1e-12)


def test_linearity_and_equivariance():
    rng = np.random.default_rng(5)
    E, H, I, M, k = 6, 12, 18, 11, 3
    w13, w2, b13, b2 = _rand_layer(rng, E, H, I)
    x = rng.standard_normal((M, H))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)])
    a = rng.random((M, k))
    y = oracle.forward(x, a, ids, w13, w2, b13, b2)
    # routing weights enter linearly (b2 is inside f_e, so it scales too)
    np.testing.assert_allclose(oracle.forward(x, 3 * a, ids, w13, w2, b13, b2), 3 * y,
                               rtol=1e-12, atol=1e-12)
    # with b2 = 0: w2 -> c w2 scales y by c; applying the weight before W2
    # (apply_router_weight_on_input) gives the same y
    y0 = oracle.forward(x, a, ids, w13, w2, b13, None)
    np.testing.assert_allclose(oracle.forward(x, a, ids, w13, 2.5 * w2, b13, None), 2.5 * y0,
                               rtol=1e-12, atol=1e-12)
    y_in = np.zeros_like(y0)
    for t in range(M):
        for j in range(k):
            e = ids[t, j]
            h = x[t] @ w13[e] + b13[e]
            z = a[t, j] * (h[:I] / (1 + np.exp(-h[:I])) * h[I:])
            y_in[t] += z @ w2[e]
    np.testing.assert_allclose(y_in, y0, rtol=1e-12, atol=1e-12)
    # token permutation equivariance
    perm = rng.permutation(M)
    np.testing.assert_allclose(oracle.forward(x[perm], a[perm], ids[perm], w13, w2, b13, b2),
                               y[perm], rtol=1e-12, atol=1e-12)
    # a repeated expert in two slots equals one slot with the summed weight
    ids2 = ids.copy()
    ids2[:, 1] = ids2[:, 0]
    a2 = a.copy()
    a1 = a.copy()
    a1[:, 0] += a1[:, 1]
    a1[:, 1] = 0.0
    np.testing.assert_allclose(oracle.forward(x, a2, ids2, w13, w2, b13, b2),
                               oracle.forward(x, a1, ids2, w13, w2, b13, b2),
                               rtol=1e-12, atol=1e-12)


def test_batched_matches_contiguous_items():
    """Scatter real tokens (each routed to k distinct experts) into the batched
    layout; row (e, i) must equal the contiguous path's weighted item output."""
    rng = np.random.default_rng(6)
    E, H, I, M, k, T = 5, 10, 14, 13, 2, 8
    w13, w2, b13, b2 = _rand_layer(rng, E, H, I)
    x = rng.standard_normal((M, H))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)])
    a = rng.random((M, k))
    xb = np.full((E, T, H), np.nan)
    rw = np.zeros((E, T))
    cnt = np.zeros(E, dtype=np.int32)
    where = {}
    for t in range(M):
        for j in range(k):
            e = ids[t, j]
            i = cnt[e]
            assert i < T
            xb[e, i] = x[t]
            rw[e, i] = a[t, j]
            where[(e, i)] = (t, j)
            cnt[e] += 1
    outs = oracle.forward_batched(xb, cnt, w13, w2, b13, b2, rw)
    y = np.zeros((M, H))
    for e in range(E):
        assert outs[e].shape == (cnt[e], H) and np.isfinite(outs[e]).all()
        for i in range(cnt[e]):
            t, j = where[(e, i)]
            one = np.zeros((1, k))
            one[0, j] = a[t, j]
            np.testing.assert_allclose(outs[e][i],
                                       oracle.forward(x[t:t + 1], one, ids[t:t + 1], w13, w2,
                                                      b13, b2)[0], rtol=1e-12, atol=1e-12)
            y[t] += outs[e][i]
    np.testing.assert_allclose(y, oracle.forward(x, a, ids, w13, w2, b13, b2),
                               rtol=1e-12, atol=1e-12)


def test_fp64_oracle_vs_fp32_evaluation():
    """The fp64 oracle and an fp32 evaluation of the same routed items agree to
    fp32 rounding on a tiny workload (guards against accidental precision loss
    in the oracle)."""
    from mixture_experts_ffn_softmax_gb300 import workloads as wl
    spec = wl.SPECS["tiny"]
    d = wl.make_moe_inputs(spec)
    f = {k: wl.to_f64(v) for k, v in d.items()}
    y, w, ids, _ = oracle.moe_layer(f["hidden"], f["router_logits"], f["w13"], f["w2"],
                                    spec.top_k, spec.routing_method, spec.renormalize)
    x32 = d["hidden"].float()
    y32 = torch.zeros_like(x32)
    for t in range(spec.M):
        for j in range(spec.top_k):
            e = int(ids[t, j])
            h = x32[t] @ d["w13"][e].float()
            z = torch.nn.functional.silu(h[:spec.I]) * h[spec.I:]
            y32[t] += float(w[t, j]) * (z @ d["w2"][e].float())
    rel = np.linalg.norm(y - y32.double().numpy()) / np.linalg.norm(y)
    assert rel < 1e-5


def test_router_logits_closed_form_and_linearity():
    """s = x W_g + b_g: with W_g picking coordinates the logits are the
    coordinates themselves plus the bias; the map is linear in x."""
    rng = np.random.default_rng(12)
    H, E, M = 6, 4, 5
    wg = np.zeros((H, E))
    wg[2, 0] = wg[0, 1] = wg[5, 2] = 1.0
    wg[1, 3], wg[4, 3] = 2.0, -1.0
    bg = np.array([0.5, 0.0, -0.25, 1.0])
    x = rng.standard_normal((M, H))
    s = oracle.router_logits(x, wg, bg)
    expect = np.stack([x[:, 2] + 0.5, x[:, 0], x[:, 5] - 0.25, 2 * x[:, 1] - x[:, 4] + 1.0], 1)
    np.testing.assert_allclose(s, expect, rtol=0, atol=1e-15)
    x2 = rng.standard_normal((M, H))
    w = rng.standard_normal((H, E))
    np.testing.assert_allclose(oracle.router_logits(x + 3 * x2, w),
                               oracle.router_logits(x, w) + 3 * oracle.router_logits(x2, w),
                               rtol=1e-12, atol=1e-12)


def test_router_weight_on_input():
    """FlagDoc section 1.2: multiplying the router weight into the second
    layer's input equals multiplying its output when b2 = 0; with a bias the
    difference is exactly sum_j (1 - a_j) b2[e_j]."""
    rng = np.random.default_rng(13)
    E, H, I, M, k = 5, 12, 16, 9, 2
    w13, w2, b13, b2 = _rand_layer(rng, E, H, I)
    x = rng.standard_normal((M, H))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)])
    a = rng.random((M, k))
    np.testing.assert_allclose(
        oracle.forward(x, a, ids, w13, w2, b13, None, apply_router_weight_on_input=True),
        oracle.forward(x, a, ids, w13, w2, b13, None), rtol=1e-12, atol=1e-12)
    d = (oracle.forward(x, a, ids, w13, w2, b13, b2, apply_router_weight_on_input=True)
         - oracle.forward(x, a, ids, w13, w2, b13, b2))
    expect = sum((1 - a[:, j])[:, None] * b2[ids[:, j]] for j in range(k))
    np.testing.assert_allclose(d, expect, rtol=1e-10, atol=1e-12)
    # closed-form layer: weight on input scales z, bias unscaled
    w13c, b13c, w2c, b2c = _closed_form_case()
    xc = np.array([[1.0, -2.0]])
    y = oracle.forward(xc, np.array([[0.3]]), np.array([[0]]), w13c, w2c, b13c, b2c,
                       apply_router_weight_on_input=True)
    np.testing.assert_allclose(y[0], 0.3 * (_closed_form_expert(0, 1.0, -2.0) - b2c[0]) + b2c[0],
                               rtol=1e-14, atol=1e-14)


def test_expert_map_partition_sums_to_full_layer():
    """Experts split across two holders (expert parallelism): each holder's
    output counts only its experts' items; the two outputs sum to the layer."""
    rng = np.random.default_rng(14)
    E, H, I, M, k = 8, 10, 12, 11, 3
    w13, w2, b13, b2 = _rand_layer(rng, E, H, I)
    x = rng.standard_normal((M, H))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)])
    a = rng.random((M, k))
    full = oracle.forward(x, a, ids, w13, w2, b13, b2)
    owner = rng.permutation(E) % 2
    parts = []
    for r in (0, 1):
        mine = np.flatnonzero(owner == r)
        emap = np.full(E, -1)
        emap[mine] = np.arange(mine.size)
        parts.append(oracle.forward(x, a, ids, w13[mine], w2[mine], b13[mine], b2[mine],
                                    expert_map=emap))
    np.testing.assert_allclose(parts[0] + parts[1], full, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(oracle.forward(x, a, ids, w13, w2, b13, b2,
                                              expert_map=np.arange(E)), full, rtol=0, atol=0)
    assert not oracle.forward(x, a, ids, w13[:1], w2[:1], b13[:1], b2[:1],
                              expert_map=np.full(E, -1)).any()


def _e4m3_table():
    """Every finite E4M3 value, decoded from its bit fields by the format's
    definition (bias 7; exponent field 0 = subnormal; S.1111.111 = NaN)."""
    vals = []
    for code in range(256):
        sgn = -1.0 if code & 0x80 else 1.0
        ef, mf = (code >> 3) & 0xF, code & 0x7
        if ef == 0xF and mf == 0x7:
            continue
        v = (mf / 8.0) * 2.0 ** -6 if ef == 0 else (1.0 + mf / 8.0) * 2.0 ** (ef - 7)
        vals.append(sgn * v)
    return np.array(sorted(set(vals)))


def test_e4m3_rounding_against_the_format():
    """Brute force over the code table: e4m3_round returns the nearest table
    value (ties to the even mantissa), is the identity on the table, and
    saturates at +-448; torch's float8_e4m3fn cast agrees inside the range."""
    table = _e4m3_table()
    assert table.size == 253 and table.max() == 448.0 and table[table > 0].min() == 2.0 ** -9
    np.testing.assert_array_equal(oracle.e4m3_round(table), table)
    rng = np.random.default_rng(21)
    v = np.concatenate([rng.standard_normal(20000) * 10 ** rng.uniform(-4, 2.5, 20000),
                        (table[:-1] + table[1:]) / 2])              # exact midpoints
    v = v.astype(np.float32).astype(np.float64)
    got = oracle.e4m3_round(v)
    def mantissa_field(val):
        a = abs(val)
        if a < 2.0 ** -6:
            return int(round(a / 2.0 ** -9))
        e = np.floor(np.log2(a))
        return int(round((a / 2.0 ** e - 1.0) * 8))

    ties = 0
    for x, g in zip(v[::3], got[::3]):
        d = np.abs(table - min(max(x, -448.0), 448.0))
        best = table[d == d.min()]
        if best.size == 1:
            assert g == best[0], x
        else:  # a tie between two neighbours: the one with the even mantissa
            assert g in best and mantissa_field(g) % 2 == 0, (x, best, g)
            ties += 1
    assert ties > 10
    assert oracle.e4m3_round(np.array([1000.0, -1e6]))[0] == 448.0
    assert oracle.e4m3_round(np.array([-1e6]))[0] == -448.0
    inside = v[np.abs(v) <= 448.0]
    ref = torch.from_numpy(inside.astype(np.float32)).to(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(oracle.e4m3_round(inside), ref)


def test_quantize_rows_error_bound_and_scale():
    rng = np.random.default_rng(22)
    x = rng.standard_normal((50, 300)) * rng.uniform(0.01, 10, (50, 1))
    x[3] = 0.0
    q, s = oracle.quantize_rows_e4m3(x)
    assert s[3] == 1.0 and not q[3].any()
    assert np.allclose(np.abs(q).max(axis=1)[np.arange(50) != 3], 448.0)
    deq = q * s[:, None]
    # relative half-step of a 3-bit mantissa, or half a subnormal step (times scale)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * s[:, None]) * (1 + 1e-6)
    assert (np.abs(deq - x) <= bound).all()


def test_fp8_forward_reduces_to_exact_layer_on_representable_inputs():
    """With every row's values in {0, +-1, +-2, +-4, +-8} and amax 8 (so
    x / scale = 56 x lands on E4M3 values) and FP8 weights w_q with scale s,
    the FP8 layer equals the layer with dequantised weights w_q * s and the
    z quantisation written out by hand; per-expert scales broadcast like
    per-channel ones."""
    rng = np.random.default_rng(23)
    E, H, I, M = 2, 16, 8, 7
    x = rng.choice([0.0, 1.0, -1.0, 2.0, -2.0, 4.0, -4.0], size=(M, H))
    x[:, 0] = 8.0                                     # row amax 8: x / scale = 56 x
    table = _e4m3_table()
    w13q = rng.choice(table[(np.abs(table) <= 4) & (np.abs(table) >= 0.25)], size=(E, H, 2 * I))
    w2q = rng.choice(table[(np.abs(table) <= 4) & (np.abs(table) >= 0.25)], size=(E, I, H))
    s13 = rng.uniform(0.01, 0.03, (E, 2 * I))
    s2 = rng.uniform(0.01, 0.03, (E, H))
    ids = np.stack([rng.permutation(E)[:1] for _ in range(M)])
    a = rng.random((M, 1))
    y8 = oracle.forward_fp8(x, a, ids, w13q, w2q, s13, s2)
    # the same computation with the z quantisation made explicit
    y = np.zeros((M, H))
    for t in range(M):
        e = ids[t, 0]
        h = x[t] @ (w13q[e] * s13[e])
        z = oracle.silu(h[:I]) * h[I:]
        zb = torch.tensor(z, dtype=torch.float32).bfloat16().double().numpy()   # z held in bf16
        qz, sz = oracle.quantize_rows_e4m3(zb[None, :])
        y[t] = a[t, 0] * ((qz[0] * sz[0]) @ (w2q[e] * s2[e]))
    # equal up to the fp32 rounding of the activation scale 8/448 (2^-24 relative)
    np.testing.assert_allclose(y8, y, rtol=1e-6, atol=1e-12)
    # and per-expert (tensor-wise) scales broadcast like per-channel ones
    y8t = oracle.forward_fp8(x, a, ids, w13q, w2q, s13[:, :1] * np.ones((1, 2 * I)),
                             s2[:, :1] * np.ones((1, H)))
    y8e = oracle.forward_fp8(x, a, ids, w13q, w2q, s13[:, 0], s2[:, 0])
    np.testing.assert_allclose(y8t, y8e, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------ FP8 block-wise ---

def _e4m3_grid():
    rng = np.random.default_rng(0)
    return np.unique(np.abs(oracle.e4m3_round(rng.standard_normal(4000) * 100)))


def _exact_group_rows(M, K, group_scales, rng):
    """Rows whose every 128-column group is E4M3 values (max 448) times a
    power of two: their per-group quantisation is exact."""
    grid = _e4m3_grid()
    x = rng.choice(grid, size=(M, K)) * rng.choice([-1.0, 1.0], size=(M, K))
    for g in range(K // 128):
        x[:, g * 128] = 448.0
        x[:, g * 128:(g + 1) * 128] *= group_scales[:, g][:, None]
    return x


def test_quantize_groups_scales_are_per_group():
    rng = np.random.default_rng(5)
    x = _exact_group_rows(2, 384, np.array([[1.0, 0.25, 8.0], [2.0 ** -6, 1.0, 0.5]]), rng)
    q, sc = oracle.quantize_groups_e4m3(x, 128)
    np.testing.assert_array_equal(sc, [[1.0, 0.25, 8.0], [2.0 ** -6, 1.0, 0.5]])
    np.testing.assert_array_equal(q * np.repeat(sc, 128, axis=1), x)
    # a group's codes depend on that group only
    x2 = x.copy()
    x2[:, 128:256] *= 3.0
    q2, sc2 = oracle.quantize_groups_e4m3(x2, 128)
    np.testing.assert_array_equal(q2[:, :128], q[:, :128])
    np.testing.assert_array_equal(q2[:, 256:], q[:, 256:])
    np.testing.assert_array_equal(sc2[:, [0, 2]], sc[:, [0, 2]])


def _block_case(rng, E=3, H=256, I=128, M=6, k=2):
    w13 = oracle.e4m3_round(rng.standard_normal((E, H, 2 * I)) * 2)
    w2 = oracle.e4m3_round(rng.standard_normal((E, I, H)) * 2)
    ids = np.array([rng.choice(E, k, replace=False) for _ in range(M)])
    tw = rng.random((M, k))
    return w13, w2, ids, tw


def test_fp8_block_reduces_to_per_channel_layer():
    """Weight block scales constant along K and equal group maxima within a
    row: the block-wise layer is the per-channel FP8 layer (one z group)."""
    rng = np.random.default_rng(6)
    E, H, I, M = 3, 256, 128, 6
    w13, w2, ids, tw = _block_case(rng, E, H, I, M)
    row_scale = 2.0 ** rng.integers(-8, -3, size=M).astype(float)
    x = _exact_group_rows(M, H, np.stack([row_scale, row_scale], 1), rng)
    c13 = rng.uniform(0.005, 0.02, size=(E, 2 * I // 128))
    c2 = rng.uniform(0.005, 0.02, size=(E, H // 128))
    s13 = np.repeat(c13[:, None, :], H // 128, axis=1)
    s2 = np.repeat(c2[:, None, :], I // 128, axis=1)
    yb = oracle.forward_fp8_block(x, tw, ids, w13, w2, s13, s2)
    yc = oracle.forward_fp8(x, tw, ids, w13, w2, np.repeat(c13, 128, axis=1),
                            np.repeat(c2, 128, axis=1))
    np.testing.assert_allclose(yb, yc, rtol=1e-12, atol=1e-12 * np.abs(yc).max())


def test_fp8_block_matches_exact_layer_within_quantisation_error():
    """Exactly quantisable x with different group scales, weight block scales
    varying along K: the block-wise layer equals the exact layer on the
    dequantised weights up to the E4M3 rounding of z (relative L2 ~2.4e-2)."""
    rng = np.random.default_rng(0)
    E, H, I, M = 3, 256, 128, 6
    w13, w2, ids, tw = _block_case(rng, E, H, I, M)
    x = _exact_group_rows(M, H, 2.0 ** rng.integers(-8, -4, size=(M, 2)).astype(float), rng)
    s13 = rng.choice([0.5, 2.0], size=(E, H // 128, 2 * I // 128)) * 0.01
    s2 = rng.choice([0.5, 2.0], size=(E, I // 128, H // 128)) * 0.01
    yb = oracle.forward_fp8_block(x, tw, ids, w13, w2, s13, s2)
    W13 = w13 * np.repeat(np.repeat(s13, 128, axis=1), 128, axis=2)
    W2 = w2 * np.repeat(np.repeat(s2, 128, axis=1), 128, axis=2)
    ye = oracle.forward(x, tw, ids, W13, W2)
    rel = np.linalg.norm(yb - ye) / np.linalg.norm(ye)
    assert rel < 0.06, rel


# ------------------------------------------------- weight-only quantisation ---

def _bf16_rne_bits(v):
    """bf16 rounding by integer arithmetic on the float32 bit pattern (round to
    nearest, ties to even), independent of the oracle's bf16_round."""
    b = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    r = ((b + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def test_unpack_nibbles_column_order():
    # byte 0x21: column 0 = 1 (low nibble), column 1 = 2; byte 0xF0: 0 then 15
    got = oracle.unpack_nibbles(np.array([[0x21, 0xF0]], dtype=np.uint8))
    assert got.tolist() == [[1, 2, 0, 15]]


def test_mx_element_values_against_the_format_tables():
    # OCP MX v1.0 element values, written out from the format definitions
    e2m1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    got = oracle.mx_decode(np.arange(16), "e2m1")
    np.testing.assert_array_equal(got[:8], e2m1)
    np.testing.assert_array_equal(got[8:], [-v for v in e2m1])
    # FP6 E3M2: bias 3, max 28 = 2^4 * 1.75, smallest subnormal 2^-2 * 1/4
    e3m2 = oracle.mx_decode(np.arange(32), "e3m2")
    assert e3m2[31] == 28.0 and e3m2[1] == 0.0625 and e3m2[12] == 1.0 and e3m2[4] == 0.25
    assert np.all(np.diff(e3m2) > 0)
    # FP6 E2M3: bias 1, max 7.5 = 2^2 * 1.875, smallest subnormal 1/8
    e2m3 = oracle.mx_decode(np.arange(32), "e2m3")
    assert e2m3[31] == 7.5 and e2m3[1] == 0.125 and e2m3[8] == 1.0 and e2m3[7] == 0.875
    assert np.all(np.diff(e2m3) > 0)
    assert oracle.mx_decode([0b100000], "e3m2")[0] == 0.0 and oracle.mx_decode([0b101100], "e3m2")[0] == -1.0
    assert oracle.ue8m0_scale([127, 128, 125]).tolist() == [1.0, 2.0, 0.25]


def test_bf16_round_against_bit_rounding():
    rng = np.random.default_rng(4)
    v = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-6, 6, 2000),
                        # exact ties: 1 + (2k+1) * 2^-8 sit halfway between bf16 values
                        1.0 + (2 * np.arange(20) + 1) * 2.0 ** -8, [0.0, -0.0, 3e38]])
    np.testing.assert_array_equal(oracle.bf16_round(v), _bf16_rne_bits(v))


def test_dequant_int4_groups_and_zero_points_by_hand():
    # E=1, K=4, N=4, group G=2 (two groups), scales and zero points per (group, column)
    codes = np.array([[0, 15, 8, 3], [1, 2, 9, 4], [7, 8, 0, 15], [12, 4, 5, 6]])
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)[None]
    scale = np.array([[[0.5, 1.0, 2.0, 0.25], [0.125, 4.0, 1.0, 0.5]]])
    zero = np.array([[[8, 8, 8, 3], [7, 0, 1, 15]]], dtype=np.uint8)
    want = np.array([[-4.0, 7.0, 0.0, 0.0],        # (q - zp) * s, rows 0-1: group 0
                     [-3.5, -6.0, 2.0, 0.25],
                     [0.0, 32.0, -1.0, 0.0],       # rows 2-3: group 1
                     [0.625, 16.0, 4.0, -4.5]])
    got = oracle.dequant_int(packed, scale, zero, bits=4)
    np.testing.assert_array_equal(got[0], want)
    # symmetric default zero point 8
    got = oracle.dequant_int(packed, np.ones((1, 2, 4)), None, bits=4)
    np.testing.assert_array_equal(got[0], codes - 8)


def test_dequant_rounds_to_bf16_once():
    s = np.float64(_bf16_rne_bits(1.0 / 3.0))       # a bf16 scale
    codes = np.array([[7, 9, 14, 1]])               # (q - 0) * s is not a bf16 value
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)[None]
    got = oracle.dequant_int(packed, np.full((1, 1, 4), s), np.zeros((1, 1, 4), np.uint8), bits=4)
    np.testing.assert_array_equal(got[0, 0], _bf16_rne_bits(codes[0] * s))
    assert not np.array_equal(got[0, 0], codes[0] * s)
    # int8, symmetric: codes are signed, zero point 0
    q8 = np.array([[[-128, -1, 0, 127]]], dtype=np.int8)
    np.testing.assert_array_equal(oracle.dequant_int(q8, np.full((1, 1, 4), 0.5), None, bits=8)[0, 0],
                                  [-64.0, -0.5, 0.0, 63.5])


def test_dequant_mx_blocks_of_32_by_hand():
    K, N = 64, 2
    codes = np.zeros((1, K, N), dtype=np.int64)
    codes[0, 0] = [0b0011, 0b1111]     # 1.5, -6
    codes[0, 31] = [0b0101, 0b0001]    # 3, 0.5
    codes[0, 32] = [0b0111, 0b1010]    # 6, -1
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    scale = np.array([[[127, 128], [125, 130]]], dtype=np.uint8)   # block 0: 1, 2; block 1: 1/4, 8
    got = oracle.dequant_mx(packed, scale, "e2m1")[0]
    assert got[0].tolist() == [1.5, -12.0] and got[31].tolist() == [3.0, 1.0]
    assert got[32].tolist() == [1.5, -8.0] and not got[1:31].any()


# -------------------------------------------------------------- mutations ---

def _pins_fail(golden_dir):
    """Run the cheap pins; return True if at least one fails."""
    checks = [lambda: test_route_golden(golden_dir),
              lambda: test_route_brute_force(0),
              lambda: test_route_with_groups_brute_force(0),
              test_ffn_closed_form,
              test_single_expert_is_dense_swiglu,
              test_uniform_topk_all_is_mean_of_experts,
              test_route_matches_printed_routing_function,
              lambda: test_align_golden(golden_dir),
              test_e4m3_rounding_against_the_format,
              test_quantize_rows_error_bound_and_scale,
              test_fp8_forward_reduces_to_exact_layer_on_representable_inputs,
              test_unpack_nibbles_column_order,
              test_mx_element_values_against_the_format_tables,
              test_dequant_int4_groups_and_zero_points_by_hand,
              test_dequant_rounds_to_bf16_once,
              test_dequant_mx_blocks_of_32_by_hand,
              test_quantize_groups_scales_are_per_group,
              test_fp8_block_reduces_to_per_channel_layer,
              test_fp8_block_matches_exact_layer_within_quantisation_error]
    for c in checks:
        try:
            c()
        except AssertionError:
            return True
    return False


def _mut_gate_up_swapped(x_rows, w13_e, w2_e, b13_e=None, b2_e=None):
    I = w2_e.shape[0]
    h = np.asarray(x_rows, float) @ w13_e + (0 if b13_e is None else b13_e)
    z = om.silu(h[:, I:]) * h[:, :I]
    return z @ w2_e + (0 if b2_e is None else b2_e)


def _mut_b2_dropped(x_rows, w13_e, w2_e, b13_e=None, b2_e=None):
    return _ORIG_FFN(x_rows, w13_e, w2_e, b13_e, None)


def _mut_silu_sign(u):
    u = np.asarray(u, float)
    return u / (1.0 + np.exp(u))


def _mut_tie_high_id(logits, allowed, top_k):
    l = np.where(allowed, np.asarray(logits, float), -np.inf)
    E = l.shape[1]
    order = np.argsort(-l[:, ::-1], axis=1, kind="stable")
    return (E - 1 - order)[:, :top_k]


def _mut_no_renorm(p, ids, method, renormalize, scale):
    return np.take_along_axis(p, ids, axis=1) * scale


def _mut_sort_unstable_align(topk_ids, E, block_m):
    a = _orig_align(topk_ids, E, block_m)
    st = a["sorted_token_ids"].copy()
    off = a["expert_offsets"]
    for e in range(E):
        c = a["expert_num_tokens"][e]
        st[off[e]:off[e] + c] = st[off[e]:off[e] + c][::-1]
    a["sorted_token_ids"] = st
    return a


def _mut_e4m3_half_away(v):
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.clip(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6, 8)
    step = np.exp2(e - 3)
    return np.sign(v) * np.minimum(np.floor(a / step + 0.5) * step, 448.0)


def _mut_quant_wrong_max(x):
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.abs(x32).max(axis=1)
    scale = np.where(amax > 0, amax / np.float32(240.0), np.float32(1.0)).astype(np.float32)
    return om.e4m3_round(x32 / scale[:, None]), scale.astype(np.float64)


def _mut_nibbles_swapped(packed):
    b = np.asarray(packed, dtype=np.uint8).astype(np.int64)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.int64)
    out[..., 0::2] = b >> 4
    out[..., 1::2] = b & 0xF
    return out


def _mut_dequant_group_cyclic(q, scale, zero=None, bits=4):
    codes = om.unpack_nibbles(q) if bits == 4 else np.asarray(q, dtype=np.int64)
    K = codes.shape[1]
    sc = np.asarray(scale, dtype=np.float64)
    zp = np.full(sc.shape, 8 if bits == 4 else 0) if zero is None else np.asarray(zero, np.int64)
    kg = np.arange(K) % sc.shape[1]                 # wrong: k mod groups, not k // G
    return om.bf16_round((codes - zp[:, kg, :]) * sc[:, kg, :])


def _mut_dequant_unrounded(q, scale, zero=None, bits=4):
    codes = om.unpack_nibbles(q) if bits == 4 else np.asarray(q, dtype=np.int64)
    K = codes.shape[1]
    sc = np.asarray(scale, dtype=np.float64)
    zp = np.full(sc.shape, 8 if bits == 4 else 0) if zero is None else np.asarray(zero, np.int64)
    kg = np.arange(K) // (K // sc.shape[1])
    return (codes - zp[:, kg, :]) * sc[:, kg, :]


def _mut_mx_bias(codes, fmt):
    c = np.asarray(codes, dtype=np.int64)
    ebits, mbits, bias = om.MX_FORMATS[fmt]
    bias += 1
    sign = np.where((c >> (ebits + mbits)) & 1, -1.0, 1.0)
    e = (c >> mbits) & ((1 << ebits) - 1)
    m = (c & ((1 << mbits) - 1)).astype(np.float64)
    return sign * np.where(e == 0, m / (1 << mbits) * 2.0 ** (1 - bias),
                           2.0 ** (e - bias) * (1.0 + m / (1 << mbits)))


def _mut_groups_row_scale(x, group=128):
    q, sc = om.quantize_rows_e4m3(x)                 # wrong: one scale per row
    return q, np.repeat(sc[:, None], np.asarray(x).shape[1] // group, axis=1)


_ORIG_BLOCK = om.forward_fp8_block


def _mut_block_first_scale(x, topk_weights, topk_ids, w13_q, w2_q, w13_scale, w2_scale,
                           w13_bias=None, w2_bias=None, block=128):
    s13 = np.repeat(np.asarray(w13_scale)[:, :1], np.asarray(w13_scale).shape[1], axis=1)
    return _ORIG_BLOCK(x, topk_weights, topk_ids, w13_q, w2_q, s13, w2_scale, w13_bias,
                       w2_bias, block)                 # wrong: first K block's scale everywhere


_ORIG_RWG = om.route_with_groups


def _mut_groups_shifted(logits_row, groups, top_k, method, renormalize, group_count,
                        routed_scaling_factor):
    """Group g mapped to experts g*gs+1 .. g*gs+gs (an off-by-one)."""
    l = np.asarray(logits_row, dtype=np.float64)[None, :]
    E = l.shape[1]
    gs = E // group_count
    allowed = np.zeros((1, E), dtype=bool)
    for g in groups:
        allowed[0, (g * gs + 1) % E:min(E, (g + 1) * gs + 1)] = True
    ids = om.topk_select(l, allowed, top_k)
    w = om.route_weights(om.scores(l, method), ids, method, renormalize, routed_scaling_factor)
    return w[0], ids[0].astype(np.int32)


def _mut_groups_strided(logits_row, groups, top_k, method, renormalize, group_count,
                        routed_scaling_factor):
    """Groups taken as strided expert sets e % group_count == g (the mask
    over the wrong axis of an (gs, G) reshape)."""
    l = np.asarray(logits_row, dtype=np.float64)[None, :]
    E = l.shape[1]
    allowed = np.zeros((1, E), dtype=bool)
    for g in groups:
        allowed[0, g::group_count] = True
    ids = om.topk_select(l, allowed, top_k)
    w = om.route_weights(om.scores(l, method), ids, method, renormalize, routed_scaling_factor)
    return w[0], ids[0].astype(np.int32)


_orig_align = om.align
_ORIG_FFN = om.expert_ffn


@pytest.mark.parametrize("target,mutant", [
    ("expert_ffn", _mut_gate_up_swapped),
    ("expert_ffn", _mut_b2_dropped),
    ("silu", _mut_silu_sign),
    ("topk_select", _mut_tie_high_id),
    ("route_weights", _mut_no_renorm),
    ("align", _mut_sort_unstable_align),
    ("e4m3_round", _mut_e4m3_half_away),
    ("quantize_rows_e4m3", _mut_quant_wrong_max),
    ("unpack_nibbles", _mut_nibbles_swapped),
    ("dequant_int", _mut_dequant_group_cyclic),
    ("dequant_int", _mut_dequant_unrounded),
    ("mx_decode", _mut_mx_bias),
    ("quantize_groups_e4m3", _mut_groups_row_scale),
    ("forward_fp8_block", _mut_block_first_scale),
    ("route_with_groups", _mut_groups_shifted),
    ("route_with_groups", _mut_groups_strided),
])
def test_planted_mistakes_are_caught(monkeypatch, golden_dir, target, mutant):
    monkeypatch.setattr(om, target, mutant)
    monkeypatch.setattr(oracle, target, mutant, raising=False)
    assert _pins_fail(golden_dir), f"no pin caught the planted mistake in {target}"
