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
    for e in rng.choice(spec.E, size=6, replace=False):
        c = int(counts[e])
        if c == 0:
            continue
        rows = np.sort(rng.choice(c, size=min(c, 4), replace=False))
        xr = f64(x[int(e)][torch.from_numpy(rows).cuda()])
        r = oracle.expert_ffn(xr, w13[e], w2[e]) * rw[e, rows][:, None]
        got.append(o[e, rows])
        ref.append(r)
    check_out(np.concatenate(got), np.concatenate(ref), "batched full size")


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
