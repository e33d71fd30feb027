"""GPU parity of the rows next to the hot path: the router logits GEMM
(s = x W_g + b_g), bf16 router logits, the router weight applied to the
second layer's input, and expert-parallel local compute (expert_map)."""
import numpy as np
import pytest
import torch

import oracle
import mixture_experts_ffn_softmax_gb300 as pkg
from mixture_experts_ffn_softmax_gb300 import workloads as wl

from helpers import check_out, check_route, f64, route_args

pytestmark = pytest.mark.gpu


def _router_weights(H, E, seed, bias=True):
    g = torch.Generator(device="cuda").manual_seed(seed)
    wg = (torch.randn(H, E, generator=g, device="cuda") * 0.05).bfloat16()
    bg = (torch.randn(E, generator=g, device="cuda") * 0.1).bfloat16() if bias else None
    return wg, bg


def _check_logits(got, ref):
    """fp32 accumulation of exact bf16 products over H terms."""
    got = np.asarray(got, dtype=np.float64)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= 1e-5, f"router logits relative L2 {rel:.3g}"
    assert np.abs(got - ref).max() <= 1e-4 * np.sqrt(np.mean(ref ** 2)) * 10


@pytest.mark.parametrize("M,H,E,bias", [(1, 64, 8, False), (333, 512, 8, True),
                                         (97, 384, 256, True), (517, 256, 128, False),
                                         (129, 328, 1024, True), (70, 1024, 16, True),
                                         (300, 768, 24, False), (5, 4096, 32, True)])
def test_router_logits(M, H, E, bias):
    g = torch.Generator(device="cuda").manual_seed(M)
    x = torch.randn(M, H, generator=g, device="cuda").bfloat16()
    wg, bg = _router_weights(H, E, M + 1, bias)
    s = pkg.moe_router_logits(x, wg, bg)
    torch.cuda.synchronize()
    _check_logits(s.cpu().numpy(), oracle.router_logits(f64(x), f64(wg), f64(bg)))


@pytest.mark.parametrize("name", ["mixtral_prefill", "deepseek_m8192"])
def test_router_logits_full_size(name):
    spec = wl.SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    wg, bg = _router_weights(spec.H, spec.E, 7)
    s = pkg.moe_router_logits(d["hidden"], wg, bg)
    torch.cuda.synchronize()
    rows = np.random.default_rng(0).choice(spec.M, 64, replace=False)
    ref = oracle.router_logits(f64(d["hidden"])[rows], f64(wg), f64(bg))
    _check_logits(s.cpu().numpy()[rows], ref)


def test_router_logits_rejects_unaligned_expert_count():
    x = torch.zeros(4, 64, device="cuda").bfloat16()
    wg = torch.zeros(64, 6, device="cuda").bfloat16()
    with pytest.raises(pkg.MoEError) as ei:
        pkg.moe_router_logits(x, wg)
    assert ei.value.status == 2   # MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("name", ["tiny", "deepseek_small", "qwen_small"])
def test_layer_from_hidden(name):
    """Router GEMM -> route -> forward.  The routing decision is taken on the
    GPU's fp32 logits on both sides (the oracle routes the same logits)."""
    spec = wl.SMALL_SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda")
    wg, bg = _router_weights(spec.H, spec.E, 3)
    y = pkg.moe_layer(d["hidden"], wg, d["w13"], d["w2"], spec.top_k, bg, d["w13_bias"],
                      d["w2_bias"], spec.k_group, spec.group_count, spec.group_select_mode,
                      spec.routing_method, spec.renormalize, spec.routed_scaling_factor)
    s = pkg.moe_router_logits(d["hidden"], wg, bg)
    torch.cuda.synchronize()
    s_np = s.cpu().numpy()
    _check_logits(s_np, oracle.router_logits(f64(d["hidden"]), f64(wg), f64(bg)))
    a = route_args(spec)
    w, ids, _ = oracle.route(s_np.astype(np.float64), a["top_k"], a["method"], a["renormalize"],
                             a["k_group"], a["group_count"], a["group_select_mode"],
                             a["routed_scaling_factor"])
    ref = oracle.forward(f64(d["hidden"]), w, ids, f64(d["w13"]), f64(d["w2"]),
                         f64(d["w13_bias"]), f64(d["w2_bias"]))
    check_out(f64(y), ref, name)


@pytest.mark.parametrize("name", ["tiny", "deepseek_small", "qwen_small", "mixtral_small"])
def test_route_bf16_logits(name):
    spec = wl.SMALL_SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    lb = d["router_logits"].bfloat16()
    a = route_args(spec)
    w, ids = pkg.moe_route(lb, spec.top_k, a["method"], a["renormalize"], a["k_group"],
                           a["group_count"], a["group_select_mode"], a["routed_scaling_factor"])
    torch.cuda.synchronize()
    check_route(lb.float().cpu().numpy(), w.cpu().numpy(), ids.cpu().numpy(), a)


@pytest.mark.parametrize("reduce", ["separate", "epilogue_atomic"])
@pytest.mark.parametrize("name", ["ragged_small", "qwen_small", "mixtral_small"])
def test_router_weight_on_input(name, reduce):
    spec = wl.SMALL_SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda")
    a = route_args(spec)
    w, ids, _ = oracle.route(f64(d["router_logits"]), a["top_k"], a["method"], a["renormalize"],
                             a["k_group"], a["group_count"], a["group_select_mode"],
                             a["routed_scaling_factor"])
    w32 = w.astype(np.float32)
    y = pkg.moe_forward(d["hidden"], torch.from_numpy(w32).cuda(), torch.from_numpy(ids).cuda(),
                        d["w13"], d["w2"], d["w13_bias"], d["w2_bias"], reduce=reduce,
                        apply_router_weight_on_input=True)
    torch.cuda.synchronize()
    ref = oracle.forward(f64(d["hidden"]), w32.astype(np.float64), ids, f64(d["w13"]),
                         f64(d["w2"]), f64(d["w13_bias"]), f64(d["w2_bias"]),
                         apply_router_weight_on_input=True)
    check_out(f64(y), ref, name)


@pytest.mark.parametrize("name", ["mixtral_small", "deepseek_small", "qwen_small"])
def test_expert_map_two_holders(name):
    """Experts split between two holders: each holder's output matches the
    oracle's expert-parallel forward, and the two sum to the full layer."""
    spec = wl.SMALL_SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda")
    a = route_args(spec)
    w, ids, _ = oracle.route(f64(d["router_logits"]), a["top_k"], a["method"], a["renormalize"],
                             a["k_group"], a["group_count"], a["group_select_mode"],
                             a["routed_scaling_factor"])
    w32 = w.astype(np.float32)
    tw, tids = torch.from_numpy(w32).cuda(), torch.from_numpy(ids).cuda()
    owner = np.random.default_rng(1).permutation(spec.E) % 2
    full = pkg.moe_forward(d["hidden"], tw, tids, d["w13"], d["w2"], d["w13_bias"], d["w2_bias"])
    parts = []
    for r in (0, 1):
        mine = np.flatnonzero(owner == r)
        emap = np.full(spec.E, -1, dtype=np.int32)
        emap[mine] = np.arange(mine.size, dtype=np.int32)
        sel = torch.from_numpy(mine).cuda()
        lw = [None if t is None else t[sel].contiguous()
              for t in (d["w13"], d["w2"], d["w13_bias"], d["w2_bias"])]
        y = pkg.moe_forward(d["hidden"], tw, tids, lw[0], lw[1], lw[2], lw[3],
                            expert_map=torch.from_numpy(emap).cuda())
        torch.cuda.synchronize()
        ref = oracle.forward(f64(d["hidden"]), w32.astype(np.float64), ids, f64(lw[0]),
                             f64(lw[1]), f64(lw[2]), f64(lw[3]), expert_map=emap)
        check_out(f64(y), ref, f"{name} holder {r}")
        parts.append(f64(y))
    check_out(parts[0] + parts[1], f64(full), f"{name} sum of holders")


def test_expert_map_bad_entries_report_error():
    M, H, I, E, Eg, k = 16, 64, 64, 2, 4, 2
    x = torch.ones(M, H, device="cuda").bfloat16()
    w13 = torch.zeros(E, H, 2 * I, device="cuda").bfloat16()
    w2 = torch.zeros(E, I, H, device="cuda").bfloat16()
    ids = torch.zeros(M, k, dtype=torch.int32, device="cuda")
    ids[:, 1] = 3
    ws = pkg.alloc_workspace(pkg.workspace_size(M, H, I, E, k))
    good = torch.tensor([0, -1, 1, -1], dtype=torch.int32, device="cuda")
    y = pkg.moe_forward(x, torch.ones(M, k, device="cuda"), ids, w13, w2, workspace=ws,
                        expert_map=good)
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 0
    assert (y.float() == 0).all()
    bad = torch.tensor([0, -1, 1, 5], dtype=torch.int32, device="cuda")   # maps past E
    pkg.moe_forward(x, torch.ones(M, k, device="cuda"), ids, w13, w2, workspace=ws,
                    expert_map=bad)
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 4
    ids[0, 0] = 9                                                          # id past Eg
    pkg.moe_forward(x, torch.ones(M, k, device="cuda"), ids, w13, w2, workspace=ws,
                    expert_map=good)
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 4
