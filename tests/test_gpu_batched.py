"""GPU parity of moe_forward_batched (the Batched activation format) against
the oracle, per valid row; invalid input rows hold NaN and output rows past
each expert's count must keep their sentinel (never read, never written)."""
import numpy as np
import pytest
import torch

import oracle
import mixture_experts_ffn_softmax_gb300 as pkg
from mixture_experts_ffn_softmax_gb300 import workloads as wl

from helpers import LazyF64, check_out, f64

pytestmark = pytest.mark.gpu

SENTINEL = -1536.0   # exactly representable in bf16 (1.5 * 2^10)


def _run(d):
    out = torch.full_like(d["x"], SENTINEL)
    pkg.moe_forward_batched(d["x"], d["expert_num_tokens"], d["w13"], d["w2"], d["w13_bias"],
                            d["w2_bias"], d["row_weight"], out=out)
    torch.cuda.synchronize()
    return out


def _check_untouched(out, counts):
    o = out.float().cpu().numpy()
    for e, c in enumerate(counts):
        assert (o[e, c:] == SENTINEL).all(), f"expert {e}: rows past the count were written"


@pytest.mark.parametrize("tiles", ["single", "pairs"])
@pytest.mark.parametrize("name", sorted(wl.SMALL_BATCHED_SPECS))
def test_batched_small(name, tiles):
    spec = wl.SMALL_BATCHED_SPECS[name]
    d = wl.make_batched_inputs(spec, device="cuda")
    pkg.set_gemm_tiles(tiles)
    try:
        out = _run(d)
    finally:
        pkg.set_gemm_tiles("auto")
    counts = d["expert_num_tokens"].cpu().numpy()
    ref = oracle.forward_batched(f64(d["x"]), counts, f64(d["w13"]), f64(d["w2"]),
                                 f64(d["w13_bias"]), f64(d["w2_bias"]), f64(d["row_weight"]))
    o = f64(out)
    got = np.concatenate([o[e, :c] for e, c in enumerate(counts)])
    check_out(got, np.concatenate(ref), name)
    _check_untouched(out, counts)


def test_batched_full_size_sampled():
    """Full-size batched layout (E=32, T=512, H=4096, I=2048): for EVERY expert
    with valid rows, its first and last valid row (the first and the last
    row block of its GEMM tiles) and two random rows against the oracle."""
    spec = wl.BATCHED_SPECS["batched"]
    d = wl.make_batched_inputs(spec, device="cuda")
    out = _run(d)
    counts = d["expert_num_tokens"].cpu().numpy()
    _check_untouched(out, counts)
    rng = np.random.default_rng(0)
    x = d["x"]
    o = f64(out)
    w13, w2 = LazyF64(d["w13"]), LazyF64(d["w2"])
    rw = d["row_weight"].cpu().numpy()
    got, ref = [], []
    checked = 0
    for e in range(spec.E):
        c = int(counts[e])
        if c == 0:
            continue
        rows = np.unique(np.r_[0, c - 1, rng.integers(0, c, size=2)])
        xr = f64(x[e][torch.from_numpy(rows).cuda()])
        r = oracle.expert_ffn(xr, w13[e], w2[e]) * rw[e, rows][:, None]
        got.append(o[e, rows])
        ref.append(r)
        checked += 1
    assert checked == int((counts > 0).sum())
    check_out(np.concatenate(got), np.concatenate(ref), "batched full size")


def _scatter_items(x, ids, wts, E):
    """Scatters real tokens' items (token t, slot j -> expert ids[t, j]) into
    the batched layout in item order: returns xb [E, T, H] (NaN past each
    count), row weights [E, T], counts [E] and each item's (expert, row)."""
    M, k = ids.shape
    flat = ids.reshape(-1).astype(np.int64)
    order = np.argsort(flat, kind="stable")
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    starts = np.concatenate([[0], np.cumsum(counts)[:-1]])
    row = np.empty(flat.size, dtype=np.int64)
    row[order] = np.arange(flat.size) - starts[flat[order]]
    T = int(counts.max())
    H = x.shape[1]
    xb = torch.full((E, T, H), float("nan"), device=x.device).bfloat16()
    rw = torch.zeros(E, T, device=x.device)
    e_t = torch.from_numpy(flat).to(x.device)
    r_t = torch.from_numpy(row).to(x.device)
    tok = torch.from_numpy(np.arange(flat.size) // k).to(x.device)
    xb[e_t, r_t] = x[tok]
    rw[e_t, r_t] = torch.from_numpy(wts.reshape(-1)).to(x.device)
    return xb, rw, counts, flat, row


def test_batched_full_size_real_tokens_match_contiguous_items():
    """Real tokens at full size: M=4096 tokens with top_k=4 distinct experts
    each of E=32 (H=4096, I=2048), weights Dirichlet(1), scattered into the
    batched layout.  Every valid batched row equals the contiguous path's
    output for that one item: the contiguous forward of the R = M * top_k
    items as single-expert tokens (top_k=1, the item's weight).  A sample of
    items is also checked against the oracle."""
    g = torch.Generator(device="cuda").manual_seed(5)
    E, H, I, M, k = 32, 4096, 2048, 4096, 4
    x = torch.randn(M, H, generator=g, device="cuda").bfloat16()
    w13 = (torch.randn(E, H, 2 * I, generator=g, device="cuda") * 0.02).bfloat16()
    w2 = (torch.randn(E, I, H, generator=g, device="cuda") * 0.02).bfloat16()
    rng = np.random.default_rng(5)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
    wts = rng.dirichlet(np.ones(k), size=M).astype(np.float32)
    xb, rw, cnt, flat, row = _scatter_items(x, ids, wts, E)
    out = torch.full_like(xb, SENTINEL)
    pkg.moe_forward_batched(xb, torch.from_numpy(cnt).cuda(), w13, w2, row_weight=rw, out=out)
    # the contiguous path, one token per item
    tok = torch.from_numpy(np.arange(M * k) // k).cuda()
    items = pkg.moe_forward(x[tok].contiguous(), torch.from_numpy(wts.reshape(-1, 1)).cuda(),
                            torch.from_numpy(flat.astype(np.int32).reshape(-1, 1)).cuda(),
                            w13, w2)
    torch.cuda.synchronize()
    _check_untouched(out, cnt)
    got = out[torch.from_numpy(flat).cuda(), torch.from_numpy(row).cuda()]
    check_out(f64(got), f64(items), "batched rows vs contiguous items (full size)")
    sel = np.sort(rng.choice(M * k, size=24, replace=False))
    l13, l2 = LazyF64(w13), LazyF64(w2)
    ref = np.stack([wts.reshape(-1)[r] * oracle.expert_ffn(f64(x[int(r) // k])[None, :],
                                                           l13[flat[r]], l2[flat[r]])[0]
                    for r in sel])
    check_out(f64(got)[sel], ref, "batched rows vs oracle (full size)")


def test_batched_matches_contiguous_items():
    """Real tokens (k distinct experts each) scattered into the batched layout:
    each batched row equals the contiguous path's output for that one item."""
    g = torch.Generator(device="cuda").manual_seed(3)
    E, T, H, I, M, k = 8, 96, 256, 192, 150, 4
    x = torch.randn(M, H, generator=g, device="cuda").bfloat16()
    w13 = (torch.randn(E, H, 2 * I, generator=g, device="cuda") * 0.05).bfloat16()
    w2 = (torch.randn(E, I, H, generator=g, device="cuda") * 0.05).bfloat16()
    rng = np.random.default_rng(3)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
    wts = rng.random((M, k)).astype(np.float32)
    xb = torch.full((E, T, H), float("nan"), device="cuda").bfloat16()
    rw = torch.zeros(E, T, device="cuda")
    cnt = np.zeros(E, dtype=np.int32)
    where = []
    for t in range(M):
        for j in range(k):
            e = ids[t, j]
            xb[e, cnt[e]] = x[t]
            rw[e, cnt[e]] = float(wts[t, j])
            where.append((e, cnt[e], t, j))
            cnt[e] += 1
    assert cnt.max() <= T
    out = torch.full_like(xb, SENTINEL)
    pkg.moe_forward_batched(xb, torch.from_numpy(cnt).cuda(), w13, w2, row_weight=rw, out=out)
    y = pkg.moe_forward(x, torch.from_numpy(wts).cuda(), torch.from_numpy(ids).cuda(), w13, w2)
    torch.cuda.synchronize()
    ob = out.float().cpu().numpy()
    acc = np.zeros((M, H))
    for e, i, t, j in where:
        acc[t] += ob[e, i]
    check_out(acc, f64(y), "batched rows summed per token vs contiguous")
    _check_untouched(out, cnt)


def test_batched_bad_counts_report_error():
    E, T, H, I = 4, 16, 64, 64
    x = torch.zeros(E, T, H, device="cuda").bfloat16()
    w13 = torch.zeros(E, H, 2 * I, device="cuda").bfloat16()
    w2 = torch.zeros(E, I, H, device="cuda").bfloat16()
    cnt = torch.tensor([3, 17, -1, 2], dtype=torch.int32, device="cuda")
    ws = pkg.alloc_workspace(pkg.batched_workspace_size(E, T, H, I))
    out = torch.full_like(x, SENTINEL)
    pkg.moe_forward_batched(x, cnt, w13, w2, workspace=ws, out=out)
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 4
    o = out.float().cpu().numpy()
    assert (o[1] == SENTINEL).all() and (o[2] == SENTINEL).all()   # skipped experts
    assert (o[0, :3] == 0).all() and (o[0, 3:] == SENTINEL).all()
