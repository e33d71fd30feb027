"""GEMM1 with the gather fused (its gather warp copies A's rows from the
token rows): the layer's output equals the separate-gather path bit for bit
on every workload shape, on single-CTA and CTA-pair tiles, and matches the
oracle at full size on sampled tokens."""
import numpy as np
import pytest
import torch

import oracle
import mixture_experts_ffn_softmax_gb300 as pkg
from mixture_experts_ffn_softmax_gb300 import workloads as wl

from helpers import LazyF64, check_out, f64, route_args

pytestmark = pytest.mark.gpu


def _layer(spec, d, **kw):
    a = route_args(spec)
    w, ids = pkg.moe_route(d["router_logits"], a["top_k"], a["method"], a["renormalize"],
                           a["k_group"], a["group_count"], a["group_select_mode"],
                           a["routed_scaling_factor"])
    ws = pkg.alloc_workspace(pkg.workspace_size(spec.M, spec.H, spec.I, spec.E, spec.top_k))
    y = pkg.moe_forward(d["hidden"], w, ids, d["w13"], d["w2"], d["w13_bias"], d["w2_bias"],
                        workspace=ws, **kw)
    torch.cuda.synchronize()
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 0
    return y, w, ids


@pytest.fixture
def modes():
    yield
    pkg.set_gather_mode("auto")
    pkg.set_gemm_tiles("auto")


@pytest.mark.parametrize("tiles", ["single", "pairs"])
@pytest.mark.parametrize("name", ["tiny", "mixtral_small", "deepseek_small", "qwen_small",
                                  "qwen_lit_small"])
def test_fused_gather_equals_separate(name, tiles, modes):
    spec = wl.SMALL_SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda")
    pkg.set_gemm_tiles(tiles)
    pkg.set_gather_mode("separate")
    y0, _, _ = _layer(spec, d)
    pkg.set_gather_mode("fused")
    y1, _, _ = _layer(spec, d)
    assert torch.equal(y0, y1)


def test_fused_gather_options(modes):
    """Router weight on the input and the expert map go through GEMM1's
    epilogue and the plan: the same with the gather fused."""
    spec = wl.SMALL_SPECS["mixtral_small"]
    d = wl.make_moe_inputs(spec, device="cuda")
    emap = torch.tensor([0, -1, 1, -1, 2, 3, -1, 4], dtype=torch.int32, device="cuda")
    local = [0, 2, 4, 5, 7]
    kw = dict(apply_router_weight_on_input=True, expert_map=emap)
    a = route_args(spec)
    w, ids = pkg.moe_route(d["router_logits"], a["top_k"], a["method"], a["renormalize"])
    outs = []
    for mode in ("separate", "fused"):
        pkg.set_gather_mode(mode)
        outs.append(pkg.moe_forward(d["hidden"], w, ids, d["w13"][local], d["w2"][local],
                                    None, None, **kw))
        torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("name", ["mixtral_prefill", "qwen_skew"])
def test_fused_gather_full_size_sampled(name, modes):
    spec = wl.SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda")
    pkg.set_gather_mode("fused")
    y, w, ids = _layer(spec, d)
    sel = np.sort(np.random.default_rng(7).choice(spec.M, 12 if spec.E > 64 else 24,
                                                  replace=False))
    xs = f64(d["hidden"][torch.from_numpy(sel).cuda()])
    ref = oracle.forward(xs, w.cpu().numpy()[sel].astype(np.float64), ids.cpu().numpy()[sel],
                         LazyF64(d["w13"]), LazyF64(d["w2"]),
                         None if d["w13_bias"] is None else LazyF64(d["w13_bias"]),
                         None if d["w2_bias"] is None else LazyF64(d["w2_bias"]))
    check_out(f64(y)[sel], ref, f"{name} fused gather")
