"""Programmatic dependent launch between the library's kernels: each kernel
waits on the device for the one before it, so the chain gives exactly the
results of plain stream order -- eagerly, across back-to-back calls that
reuse the same buffers, and replayed from a CUDA graph.  (The epilogue-atomic
reduce adds a token's rows in no fixed order, so that path is compared up to
rounding.)"""
import numpy as np
import pytest
import torch

import oracle
import mixture_experts_ffn_softmax_gb300 as pkg
from mixture_experts_ffn_softmax_gb300 import workloads as wl

from helpers import check_out, f64, route_args

pytestmark = pytest.mark.gpu


@pytest.fixture
def pdl_restore():
    yield
    pkg.set_pdl(True)


def _layer(spec, d, w, ids, ws, out, **kw):
    pkg.moe_route(d["router_logits"], spec.top_k, spec.routing_method, spec.renormalize,
                  spec.k_group, spec.group_count, spec.group_select_mode,
                  spec.routed_scaling_factor, w, ids)
    pkg.moe_forward(d["hidden"], w, ids, d["w13"], d["w2"], d["w13_bias"], d["w2_bias"], ws, out,
                    **kw)


@pytest.mark.parametrize("reduce", ["separate", "epilogue_atomic"])
@pytest.mark.parametrize("name", sorted(wl.SMALL_SPECS))
def test_pdl_chain_equals_plain_stream_order(name, reduce, pdl_restore):
    spec = wl.SMALL_SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda")
    w = torch.empty(spec.M, spec.top_k, device="cuda")
    ids = torch.empty(spec.M, spec.top_k, dtype=torch.int32, device="cuda")
    ws = pkg.alloc_workspace(pkg.workspace_size(spec.M, spec.H, spec.I, spec.E, spec.top_k,
                                                reduce))
    outs = {}
    for on in (False, True):
        pkg.set_pdl(on)
        out = torch.empty_like(d["hidden"])
        for _ in range(3):   # back to back on the same workspace
            _layer(spec, d, w, ids, ws, out, reduce=reduce)
        torch.cuda.synchronize()
        assert pkg.read_error(pkg.workspace_error_word(ws)) == 0
        outs[on] = out
    if reduce == "separate":
        assert torch.equal(outs[False], outs[True])
    else:
        # fp32 atomics add a token's rows in no fixed order: equal up to rounding
        check_out(f64(outs[True]), f64(outs[False]), f"{name} atomic, pdl on vs off")
    a = route_args(spec)
    ref, rw, rids, _ = oracle.moe_layer(f64(d["hidden"]), f64(d["router_logits"]), f64(d["w13"]),
                                        f64(d["w2"]), spec.top_k, a["method"], a["renormalize"],
                                        a["k_group"], a["group_count"], a["group_select_mode"],
                                        a["routed_scaling_factor"], f64(d["w13_bias"]),
                                        f64(d["w2_bias"]))
    if np.array_equal(ids.cpu().numpy(), rids):
        check_out(f64(outs[True]), ref, name)


@pytest.mark.parametrize("name", ["tiny", "qwen_small", "deepseek_small"])
def test_pdl_graph_replay_equals_plain_eager(name, pdl_restore):
    """A graph captured with the launches' programmatic edges replays to the
    bits of an eager run in plain stream order."""
    spec = wl.SMALL_SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda")
    w = torch.empty(spec.M, spec.top_k, device="cuda")
    ids = torch.empty(spec.M, spec.top_k, dtype=torch.int32, device="cuda")
    ws = pkg.alloc_workspace(pkg.workspace_size(spec.M, spec.H, spec.I, spec.E, spec.top_k))
    out = torch.empty_like(d["hidden"])
    pkg.set_pdl(True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _layer(spec, d, w, ids, ws, out)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _layer(spec, d, w, ids, ws, out)
    for seed in (1, 2):
        new = wl.make_moe_inputs(spec, device="cuda", seed=seed, weights=False)
        d["hidden"].copy_(new["hidden"])
        d["router_logits"].copy_(new["router_logits"])
        g.replay()
        torch.cuda.synchronize()
        got = out.clone()
        pkg.set_pdl(False)
        _layer(spec, d, w, ids, ws, out)
        torch.cuda.synchronize()
        pkg.set_pdl(True)
        assert torch.equal(got, out)
        assert pkg.read_error(pkg.workspace_error_word(ws)) == 0


def test_pdl_fp8_and_weight_only_layers(pdl_restore):
    """The FP8 (per-channel and block scales) and weight-only int4 layers on a
    small Mixtral-shape copy: identical with and without PDL."""
    spec = wl.SPECS["mixtral_prefill"].scaled("mixtral_pdl", M=300, H=512, I=640)
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    w, ids = pkg.moe_route(d["router_logits"], spec.top_k, "softmax", True)
    q = wl.make_fp8_weights(spec, device="cuda")
    qb = wl.make_fp8_weights(spec, device="cuda", block=True)
    qi = wl.make_wq_weights(spec, "int4", 128, device="cuda")
    res = {}
    for on in (False, True):
        pkg.set_pdl(on)
        r = [pkg.moe_forward_fp8(d["hidden"], w, ids, q["w13_q"], q["w2_q"], q["w13_scale"],
                                 q["w2_scale"]),
             pkg.moe_forward_fp8(d["hidden"], w, ids, qb["w13_q"], qb["w2_q"], qb["w13_scale"],
                                 qb["w2_scale"]),
             pkg.moe_forward_wq(d["hidden"], w, ids, "int4", qi["w13_q"], qi["w2_q"],
                                qi["w13_scale"], qi["w2_scale"], qi["w13_zero"], qi["w2_zero"],
                                qi["group_size"])]
        torch.cuda.synchronize()
        res[on] = r
    for a, b in zip(res[False], res[True]):
        assert torch.equal(a, b)
