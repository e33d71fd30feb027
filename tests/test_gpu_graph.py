"""The forward is stream-ordered, allocates nothing and never synchronises,
so route + forward can be captured into a CUDA graph: replays on new inputs
(copied into the captured buffers) give the eager results bit for bit."""
import pytest
import torch

import mixture_experts_ffn_softmax_gb300 as pkg
from mixture_experts_ffn_softmax_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _layer(spec, d, w, ids, ws, out):
    pkg.moe_route(d["router_logits"], spec.top_k, spec.routing_method, spec.renormalize,
                  spec.k_group, spec.group_count, spec.group_select_mode,
                  spec.routed_scaling_factor, w, ids)
    pkg.moe_forward(d["hidden"], w, ids, d["w13"], d["w2"], d["w13_bias"], d["w2_bias"], ws, out)


@pytest.mark.parametrize("name", ["tiny", "deepseek_small", "qwen_small", "mixtral_decode_small"])
def test_forward_graph_replay_matches_eager(name):
    spec = wl.SMALL_SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda")
    w = torch.empty(spec.M, spec.top_k, device="cuda")
    ids = torch.empty(spec.M, spec.top_k, dtype=torch.int32, device="cuda")
    ws = pkg.alloc_workspace(pkg.workspace_size(spec.M, spec.H, spec.I, spec.E, spec.top_k))
    out = torch.empty_like(d["hidden"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _layer(spec, d, w, ids, ws, out)          # first calls set up outside the capture
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
        _layer(spec, d, w, ids, ws, out)          # eager on the same inputs
        torch.cuda.synchronize()
        assert torch.equal(got, out)
        assert pkg.read_error(pkg.workspace_error_word(ws)) == 0
