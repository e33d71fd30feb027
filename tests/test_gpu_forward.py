"""GPU parity of moe_forward / fused_moe against the oracle.

Small workloads (every routing structure, ragged H/I/M, biases) are compared
element by element; the full-size workloads run in the same launch
configuration the benchmark times and are compared on sampled tokens that the
oracle computes one by one.  Outputs: relative L2 <= 1e-2 and
max abs <= 5e-2 * RMS of the oracle output."""
import numpy as np
import pytest
import torch

import oracle
import mixture_experts_ffn_softmax_gb300 as pkg
from mixture_experts_ffn_softmax_gb300 import workloads as wl

from helpers import LazyF64, check_out, check_route, covering_tokens, f64, route_args

pytestmark = pytest.mark.gpu


def _oracle_route(spec, logits):
    a = route_args(spec)
    return oracle.route(f64(logits), a["top_k"], a["method"], a["renormalize"], a["k_group"],
                        a["group_count"], a["group_select_mode"], a["routed_scaling_factor"])


@pytest.fixture
def tiles(request):
    """Forces the grouped-GEMM tile shape for one test, then restores auto."""
    pkg.set_gemm_tiles(request.param)
    yield request.param
    pkg.set_gemm_tiles("auto")


@pytest.mark.parametrize("tiles", ["single", "pairs"], indirect=True)
@pytest.mark.parametrize("reduce", ["separate", "epilogue_atomic"])
@pytest.mark.parametrize("name", sorted(wl.SMALL_SPECS))
def test_forward_small_workloads(name, reduce, tiles):
    """Both TopKWeightAndReduce choices and both GEMM tile shapes (single CTA,
    CTA pair) against the oracle."""
    spec = wl.SMALL_SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda")
    w, ids, _ = _oracle_route(spec, d["router_logits"])
    tw = torch.from_numpy(w.astype(np.float32)).cuda()
    tids = torch.from_numpy(ids).cuda()
    y = pkg.moe_forward(d["hidden"], tw, tids, d["w13"], d["w2"], d["w13_bias"], d["w2_bias"],
                        reduce=reduce)
    torch.cuda.synchronize()
    ref = oracle.forward(f64(d["hidden"]), w.astype(np.float32).astype(np.float64), ids,
                         f64(d["w13"]), f64(d["w2"]), f64(d["w13_bias"]), f64(d["w2_bias"]))
    check_out(f64(y), ref, name)


@pytest.mark.parametrize("name", ["tiny", "deepseek_small", "qwen_small", "ragged_small"])
def test_fused_layer_small_workloads(name):
    """route + forward through the GPU path vs oracle.moe_layer."""
    spec = wl.SMALL_SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda")
    a = route_args(spec)
    y = pkg.fused_moe(d["hidden"], d["router_logits"], d["w13"], d["w2"], spec.top_k,
                      d["w13_bias"], d["w2_bias"], spec.k_group, spec.group_count,
                      spec.group_select_mode, spec.routing_method, spec.renormalize,
                      spec.routed_scaling_factor)
    gw, gids = pkg.moe_route(d["router_logits"], spec.top_k, a["method"], a["renormalize"],
                             a["k_group"], a["group_count"], a["group_select_mode"],
                             a["routed_scaling_factor"])
    torch.cuda.synchronize()
    check_route(d["router_logits"].cpu().numpy(), gw.cpu().numpy(), gids.cpu().numpy(), a)
    ref, _, _, _ = oracle.moe_layer(f64(d["hidden"]), f64(d["router_logits"]), f64(d["w13"]),
                                    f64(d["w2"]), spec.top_k, spec.routing_method,
                                    spec.renormalize, spec.k_group, spec.group_count,
                                    spec.group_select_mode, spec.routed_scaling_factor,
                                    f64(d["w13_bias"]), f64(d["w2_bias"]))
    check_out(f64(y), ref, name)


def test_intermediate_stages():
    """Inside the forward's workspace: the sorted item list and the inverse
    permutation are bit-exact against the oracle's align, the permuted rows
    (written by the separate gather kernel) are bit-exact copies of the
    routed tokens, and z (GEMM1 output) matches SiLU(gate) * up of the oracle
    within bf16 rounding."""
    spec = wl.SMALL_SPECS["mixtral_small"]
    d = wl.make_moe_inputs(spec, device="cuda")
    w, ids, _ = _oracle_route(spec, d["router_logits"])
    tw = torch.from_numpy(w.astype(np.float32)).cuda()
    tids = torch.from_numpy(ids).cuda()
    M, H, I, E, k = spec.M, spec.H, spec.I, spec.E, spec.top_k
    ws = pkg.alloc_workspace(pkg.workspace_size(M, H, I, E, k))
    pkg.set_gather_mode("separate")
    try:
        pkg.moe_forward(d["hidden"], tw, tids, d["w13"], d["w2"], workspace=ws)
        torch.cuda.synchronize()
    finally:
        pkg.set_gather_mode("auto")
    lay = pkg.workspace_layout(M, H, I, E, k)
    al = oracle.align(ids, E, pkg.BLOCK_M)
    n = al["num_tokens_post_padded"]
    b = ws.cpu()

    def view(off, count, dtype):
        nbytes = count * torch.tensor([], dtype=dtype).element_size()
        return b[off:off + nbytes].view(dtype)

    st = view(lay["sorted_token_ids"], n, torch.int32).numpy()
    assert st.tolist() == al["sorted_token_ids"].tolist()
    inv = view(lay["inv"], M * k, torch.int32).numpy()
    assert (st[inv] == np.arange(M * k)).all()
    a_perm = view(lay["a_perm"], n * H, torch.bfloat16).view(n, H)
    x = d["hidden"].cpu()
    valid = st < M * k
    assert torch.equal(a_perm[torch.from_numpy(valid)], x[torch.from_numpy(st[valid] // k)])
    z = view(lay["z"], n * I, torch.bfloat16).view(n, I).double().numpy()
    xf, w13 = f64(d["hidden"]), f64(d["w13"])
    zref = np.zeros((n, I))
    for p in np.flatnonzero(valid):
        e = ids.reshape(-1)[st[p]]
        h = xf[st[p] // k] @ w13[e]
        zref[p] = oracle.silu(h[:I]) * h[I:]
    check_out(z[valid], zref[valid], "z")


def test_forward_in_place_and_reuse():
    spec = wl.SMALL_SPECS["ragged_small"]
    d = wl.make_moe_inputs(spec, device="cuda")
    w, ids, _ = _oracle_route(spec, d["router_logits"])
    tw = torch.from_numpy(w.astype(np.float32)).cuda()
    tids = torch.from_numpy(ids).cuda()
    ws = pkg.alloc_workspace(pkg.workspace_size(spec.M, spec.H, spec.I, spec.E, spec.top_k))
    ws.fill_(0xFF)  # workspace contents on entry must not matter
    y1 = pkg.moe_forward(d["hidden"], tw, tids, d["w13"], d["w2"], d["w13_bias"],
                         d["w2_bias"], workspace=ws)
    x = d["hidden"].clone()
    y2 = pkg.moe_forward(x, tw, tids, d["w13"], d["w2"], d["w13_bias"], d["w2_bias"],
                         workspace=ws, out=x)                     # in place
    torch.cuda.synchronize()
    assert y2.data_ptr() == x.data_ptr()
    assert torch.equal(y1, y2)
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 0


@pytest.mark.parametrize("tiles", ["auto", "pairs"], indirect=True)
@pytest.mark.parametrize("reduce", ["auto", "separate", "epilogue_atomic"])
@pytest.mark.parametrize("case", [
    dict(M=1, H=64, I=64, E=1, k=1),
    dict(M=5, H=136, I=72, E=3, k=3),      # top_k = E
    dict(M=300, H=256, I=320, E=16, k=1),
    dict(M=129, H=512, I=256, E=4, k=2, one_expert=True),
    dict(M=40, H=64, I=128, E=8, k=4, dup=True),
    dict(M=20000, H=64, I=64, E=4, k=2),   # crosses the 16384-token chunk
    dict(M=3, H=16, I=8, E=2, k=2),        # H, I below one 64-wide TMA box
    dict(M=70, H=8, I=24, E=3, k=1),
    dict(M=100, H=64, I=64, E=1024, k=64),  # the largest expert count and top_k
    dict(M=50, H=64, I=64, E=64, k=64),     # every expert, top_k = E = 64
])
def test_forward_edge_cases(case, reduce, tiles):
    g = torch.Generator(device="cuda").manual_seed(5)
    M, H, I, E, k = case["M"], case["H"], case["I"], case["E"], case["k"]
    x = torch.randn(M, H, generator=g, device="cuda").bfloat16()
    w13 = (torch.randn(E, H, 2 * I, generator=g, device="cuda") * 0.05).bfloat16()
    w2 = (torch.randn(E, I, H, generator=g, device="cuda") * 0.05).bfloat16()
    rng = np.random.default_rng(M)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
    if case.get("one_expert"):
        ids[:, 0] = 2
        ids[:, 1] = np.where(ids[:, 1] == 2, 0, ids[:, 1])
    if case.get("dup"):
        ids[:, 1] = ids[:, 0]
    wts = rng.random((M, k)).astype(np.float32)
    y = pkg.moe_forward(x, torch.from_numpy(wts).cuda(), torch.from_numpy(ids).cuda(), w13, w2,
                        reduce=reduce)
    torch.cuda.synchronize()
    if M > 4096:   # oracle on a sample of tokens (both chunks)
        sel = np.r_[0:64, 16380:16400, M - 64:M]
        ref = oracle.forward(f64(x)[sel], wts[sel], ids[sel], f64(w13), f64(w2))
        check_out(f64(y)[sel], ref, str(case))
    else:
        ref = oracle.forward(f64(x), wts, ids, f64(w13), f64(w2))
        check_out(f64(y), ref, str(case))


def test_forward_uniform_topk_is_mean():
    """All logits equal and top_k = E through the GPU path: the output is the
    mean of the dense expert outputs."""
    g = torch.Generator(device="cuda").manual_seed(9)
    M, H, I, E = 70, 128, 192, 4
    x = torch.randn(M, H, generator=g, device="cuda").bfloat16()
    w13 = (torch.randn(E, H, 2 * I, generator=g, device="cuda") * 0.05).bfloat16()
    w2 = (torch.randn(E, I, H, generator=g, device="cuda") * 0.05).bfloat16()
    y = pkg.fused_moe(x, torch.zeros(M, E, device="cuda"), w13, w2, E, renormalize=False)
    torch.cuda.synchronize()
    xf, a, b = f64(x), f64(w13), f64(w2)
    mean = sum(oracle.expert_ffn(xf, a[e], b[e]) for e in range(E)) / E
    check_out(f64(y), mean, "uniform top-k")


def test_reduce_choices_agree_full_size_qwen():
    """Both reduce choices on the full Qwen-shape layer (k = 8, skewed experts)
    give the same output up to fp32 summation order."""
    spec = wl.SPECS["qwen_skew"]
    d = wl.make_moe_inputs(spec, device="cuda")
    w, ids = pkg.moe_route(d["router_logits"], spec.top_k, "softmax", False)
    ys = [pkg.moe_forward(d["hidden"], w, ids, d["w13"], d["w2"], d["w13_bias"], d["w2_bias"],
                          reduce=r) for r in ("separate", "epilogue_atomic")]
    torch.cuda.synchronize()
    check_out(f64(ys[1]), f64(ys[0]), "atomic vs separate")


def test_forward_bad_ids_report_error():
    g = torch.Generator(device="cuda").manual_seed(2)
    M, H, I, E, k = 16, 64, 64, 4, 2
    x = torch.randn(M, H, generator=g, device="cuda").bfloat16()
    w13 = torch.randn(E, H, 2 * I, generator=g, device="cuda").bfloat16()
    w2 = torch.randn(E, I, H, generator=g, device="cuda").bfloat16()
    ids = torch.zeros(M, k, dtype=torch.int32, device="cuda")
    ids[3, 1] = 7
    ws = pkg.alloc_workspace(pkg.workspace_size(M, H, I, E, k))
    pkg.moe_forward(x, torch.ones(M, k, device="cuda"), ids, w13, w2, workspace=ws)
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 4   # MOE_ERR_BAD_EXPERT_ID


def test_tile_shapes_agree_full_size_mixtral():
    """Single-CTA and CTA-pair GEMMs on the full Mixtral-shape prefill: same
    result up to fp32 summation order."""
    spec = wl.SPECS["mixtral_prefill"]
    d = wl.make_moe_inputs(spec, device="cuda")
    w, ids = pkg.moe_route(d["router_logits"], spec.top_k, "softmax", True)
    ys = []
    for mode in ("single", "pairs"):
        pkg.set_gemm_tiles(mode)
        ys.append(pkg.moe_forward(d["hidden"], w, ids, d["w13"], d["w2"]))
    pkg.set_gemm_tiles("auto")
    torch.cuda.synchronize()
    check_out(f64(ys[1]), f64(ys[0]), "pairs vs single")


@pytest.mark.parametrize("tiles", ["single", "pairs"], indirect=True)
@pytest.mark.parametrize("reduce", ["separate", "epilogue_atomic"])
def test_odd_and_even_row_blocks(reduce, tiles):
    """Experts with 0, 1, 2, 3 and 5 row blocks (a pair tile's second row
    block is absent for the odd ones: its rows are computed, never stored),
    ragged N in both GEMMs, biases, and a repeated call giving the same bits."""
    counts = [0, 100, 128, 129, 300, 600, 256, 1, 17, 33]
    E, H, I = len(counts), 392, 328
    rng = np.random.default_rng(21)
    ids = np.concatenate([np.full(c, e) for e, c in enumerate(counts)]).astype(np.int32)
    rng.shuffle(ids)
    M, k = ids.size, 1
    ids = ids.reshape(M, k)
    wts = rng.random((M, k)).astype(np.float32)
    g = torch.Generator(device="cuda").manual_seed(21)
    x = torch.randn(M, H, generator=g, device="cuda").bfloat16()
    w13 = (torch.randn(E, H, 2 * I, generator=g, device="cuda") * 0.05).bfloat16()
    w2 = (torch.randn(E, I, H, generator=g, device="cuda") * 0.05).bfloat16()
    b13 = (torch.randn(E, 2 * I, generator=g, device="cuda") * 0.1).bfloat16()
    b2 = (torch.randn(E, H, generator=g, device="cuda") * 0.1).bfloat16()
    tw, tids = torch.from_numpy(wts).cuda(), torch.from_numpy(ids).cuda()
    ys = [pkg.moe_forward(x, tw, tids, w13, w2, b13, b2, reduce=reduce) for _ in range(2)]
    torch.cuda.synchronize()
    ref = oracle.forward(f64(x), wts, ids, f64(w13), f64(w2), f64(b13), f64(b2))
    check_out(f64(ys[0]), ref, f"odd/even row blocks {tiles} {reduce}")
    assert torch.equal(ys[0], ys[1])


FULL = ["mixtral_prefill", "mixtral_decode", "deepseek_m64", "deepseek_m8192", "qwen_skew",
        "qwen_skew_lit"]


@pytest.mark.parametrize("name", FULL)
def test_forward_full_size_sampled(name):
    """Full-size layer in the benchmark's launch configuration; sampled tokens
    checked against the oracle.  The sample holds, for every expert that
    receives items, the tokens of its first item, of the first item of its
    last 128-row block and of its last item (so every touched expert's first
    and last row block of the grouped GEMMs is compared), plus random
    tokens."""
    spec = wl.SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda")
    a = route_args(spec)
    ws = pkg.alloc_workspace(pkg.workspace_size(spec.M, spec.H, spec.I, spec.E, spec.top_k))
    gw, gids = pkg.moe_route(d["router_logits"], spec.top_k, a["method"], a["renormalize"],
                             a["k_group"], a["group_count"], a["group_select_mode"],
                             a["routed_scaling_factor"])
    y = pkg.moe_forward(d["hidden"], gw, gids, d["w13"], d["w2"], d["w13_bias"], d["w2_bias"],
                        workspace=ws)
    torch.cuda.synchronize()
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 0
    gw_np, gids_np = gw.cpu().numpy(), gids.cpu().numpy()
    check_route(d["router_logits"].cpu().numpy(), gw_np, gids_np, a)
    rng = np.random.default_rng(0)
    sel = covering_tokens(gids_np, 12 if spec.E > 64 else 24, rng)
    touched = np.unique(gids_np)
    assert set(np.unique(gids_np[sel])) == set(touched)
    xs = f64(d["hidden"][torch.from_numpy(sel).cuda()])
    ref = oracle.forward(xs, gw_np[sel].astype(np.float64), gids_np[sel], LazyF64(d["w13"]),
                         LazyF64(d["w2"]),
                         None if d["w13_bias"] is None else LazyF64(d["w13_bias"]),
                         None if d["w2_bias"] is None else LazyF64(d["w2_bias"]))
    check_out(f64(y)[sel], ref, name)
    assert np.isfinite(f64(y)).all()


@pytest.mark.parametrize("reduce", ["separate", "epilogue_atomic"])
def test_forward_dynamic_schedule_across_chunks_and_calls(reduce):
    """CTA-pair GEMMs with K >= 3072 take their tiles from a counter that each
    launch resets when it ends: a forward of two token chunks (20000 > 16384
    tokens) repeated three times gives the oracle's result and the same bits
    every time."""
    M, H, I, E, k = 20000, 3072, 64, 4, 2
    g = torch.Generator(device="cuda").manual_seed(11)
    x = torch.randn(M, H, generator=g, device="cuda").bfloat16()
    w13 = (torch.randn(E, H, 2 * I, generator=g, device="cuda") * 0.02).bfloat16()
    w2 = (torch.randn(E, I, H, generator=g, device="cuda") * 0.05).bfloat16()
    rng = np.random.default_rng(3)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
    wts = rng.random((M, k)).astype(np.float32)
    tw, tids = torch.from_numpy(wts).cuda(), torch.from_numpy(ids).cuda()
    ws = pkg.alloc_workspace(pkg.workspace_size(M, H, I, E, k, reduce))
    outs = []
    for _ in range(3):
        outs.append(pkg.moe_forward(x, tw, tids, w13, w2, workspace=ws, reduce=reduce))
        torch.cuda.synchronize()
        assert pkg.read_error(pkg.workspace_error_word(ws)) == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    sel = np.r_[0:16, 16376:16392, M - 16:M]
    ref = oracle.forward(f64(x)[sel], wts[sel], ids[sel], f64(w13), f64(w2))
    check_out(f64(outs[0])[sel], ref, f"dynamic schedule {reduce}")
