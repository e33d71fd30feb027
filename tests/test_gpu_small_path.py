"""GPU parity of the small-call path: moe_forward with the automatic reduce
for at most 256 routed items and small expert weights runs the layer in two
kernels, GEMM1 finding each expert's items in topk_ids itself and GEMM2 adding
the weighted rows into an fp32 token accumulator ("fused_moe.py 分析": the
fused_moe kernel and the reduce after it).  Checked against the oracle on
shapes with one token, all experts touched, an expert holding every item,
duplicate ids, ids outside [0, E), biases; against the general path; the two
kernels are the ones that ran; a CUDA graph replays it; and moe_forward_host
takes it."""
import numpy as np
import pytest
import torch

import oracle
import mixture_experts_ffn_softmax_gb300 as pkg
from mixture_experts_ffn_softmax_gb300 import workloads as wl

from helpers import check_out, f64, route_args

pytestmark = pytest.mark.gpu

# (M, H, I, E, top_k, bias): the tiny layer; one token, one item; the Mixtral
# decode proportions scaled down; 200 items over 16 experts; 256 items over
# 64 experts (k = 8); a handful of items over 3 experts; 240 items over 2
# experts (four 32-item passes, GEMM1's ring wrapping 16 K stages); K = 4096
# (64 stages) at the largest M * H; I = 2048 (GEMM2's ring over 32 stages)
SHAPES = [(64, 256, 512, 8, 2, True), (1, 64, 64, 4, 1, False), (16, 512, 640, 8, 2, True),
          (100, 128, 192, 16, 2, True), (32, 256, 128, 64, 8, False), (5, 64, 128, 3, 3, True),
          (120, 1024, 256, 2, 2, True), (64, 4096, 64, 4, 2, False), (8, 64, 2048, 4, 2, True)]


@pytest.fixture
def small_restore():
    yield
    pkg.set_small_path(True)


def _spec(M, H, I, E, k, bias):
    return wl.SMALL_SPECS["tiny"].scaled("small", M=M, H=H, I=I, E=E, top_k=k, bias=bias)


def _route(spec, d):
    a = route_args(spec)
    w, ids, _ = oracle.route(f64(d["router_logits"]), a["top_k"], a["method"], a["renormalize"],
                             a["k_group"], a["group_count"], a["group_select_mode"],
                             a["routed_scaling_factor"])
    return w.astype(np.float32), ids


def _oracle(d, w, ids):
    return oracle.forward(f64(d["hidden"]), w.astype(np.float64), ids, f64(d["w13"]), f64(d["w2"]),
                          f64(d["w13_bias"]), f64(d["w2_bias"]))


def _forward(d, w, ids, ws=None):
    return pkg.moe_forward(d["hidden"], torch.as_tensor(w).cuda(), torch.as_tensor(ids).cuda(),
                           d["w13"], d["w2"], d["w13_bias"], d["w2_bias"], workspace=ws)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "M%d_H%d_I%d_E%d_k%d_b%d" % s)
def test_small_path_matches_oracle(shape):
    spec = _spec(*shape)
    d = wl.make_moe_inputs(spec, device="cuda")
    w, ids = _route(spec, d)
    ws = pkg.alloc_workspace(pkg.workspace_size(spec.M, spec.H, spec.I, spec.E, spec.top_k))
    n0 = pkg.launch_count()
    pkg.profiler_start()
    y = _forward(d, w, ids, ws)
    ran = pkg.profiler_stop()
    torch.cuda.synchronize()
    assert set(ran) == {"small_gemm1", "small_gemm2"}, sorted(ran)
    assert pkg.launch_count() - n0 == 2
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 0
    check_out(f64(y), _oracle(d, w, ids), f"small {shape}")


@pytest.mark.parametrize("shape", SHAPES[:3], ids=lambda s: "M%d_H%d_I%d_E%d_k%d_b%d" % s)
def test_small_path_equals_general_path(shape, small_restore):
    spec = _spec(*shape)
    d = wl.make_moe_inputs(spec, device="cuda")
    w, ids = _route(spec, d)
    y_small = _forward(d, w, ids)
    pkg.set_small_path(False)
    pkg.profiler_start()
    y_gen = _forward(d, w, ids)
    ran = pkg.profiler_stop()
    torch.cuda.synchronize()
    assert "small_gemm1" not in ran
    check_out(f64(y_small), f64(y_gen), f"small vs general {shape}")


def test_small_path_skewed_and_duplicate_ids():
    """Every item on expert 0 but a few, some tokens routing both items to
    the same expert: experts with 0, a few and 250 items; rows in several
    32-item passes."""
    spec = _spec(125, 128, 128, 5, 2, True)
    d = wl.make_moe_inputs(spec, device="cuda")
    g = np.random.default_rng(4)
    ids = np.zeros((spec.M, 2), np.int32)
    ids[:, 1] = g.integers(0, 2, spec.M)        # (0, 0) for about half the tokens
    ids[:5, 1] = 3
    w = g.random((spec.M, 2)).astype(np.float32)
    y = _forward(d, w, ids)
    torch.cuda.synchronize()
    check_out(f64(y), _oracle(d, w, ids), "skewed and duplicate ids")


def test_small_path_ids_outside_the_experts():
    """Items routed to an id outside [0, E) contribute nothing and set the
    error word (MOE_ERR_BAD_EXPERT_ID); the others match the oracle."""
    spec = _spec(12, 128, 128, 6, 2, False)
    d = wl.make_moe_inputs(spec, device="cuda")
    w, ids = _route(spec, d)
    ids = ids.copy()
    ids[3, 1] = spec.E + 2
    ids[7, 0] = -1
    ws = pkg.alloc_workspace(pkg.workspace_size(spec.M, spec.H, spec.I, spec.E, spec.top_k))
    y = _forward(d, w, ids, ws)
    torch.cuda.synchronize()
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 4   # MOE_ERR_BAD_EXPERT_ID
    wk, idk = w.copy(), ids.copy()
    wk[3, 1] = wk[7, 0] = 0.0
    idk[3, 1] = idk[7, 0] = 0
    check_out(f64(y), _oracle(d, wk, idk), "ids outside the experts")
    # the next call on the same workspace starts with a clear error word
    _forward(d, w, np.clip(ids, 0, spec.E - 1).astype(np.int32), ws)
    torch.cuda.synchronize()
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 0


def test_small_path_graph_replay():
    spec = _spec(64, 256, 512, 8, 2, True)
    d = wl.make_moe_inputs(spec, device="cuda")
    a = route_args(spec)
    ws = pkg.alloc_workspace(pkg.workspace_size(spec.M, spec.H, spec.I, spec.E, spec.top_k))
    out = torch.empty_like(d["hidden"])
    x = d["hidden"].clone()
    logits = d["router_logits"].clone()

    def step():
        tw, tids = pkg.moe_route(logits, spec.top_k, a["method"], a["renormalize"])
        pkg.moe_forward(x, tw, tids, d["w13"], d["w2"], d["w13_bias"], d["w2_bias"],
                        workspace=ws, out=out)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step()
    for seed in (3, 4):
        new = wl.make_moe_inputs(spec, device="cuda", seed=seed, weights=False)
        x.copy_(new["hidden"])
        logits.copy_(new["router_logits"])
        graph.replay()
        torch.cuda.synchronize()
        ref = out.clone()
        with torch.cuda.stream(s):
            step()
        s.synchronize()
        assert torch.equal(out, ref) or float((out.float() - ref.float()).abs().max()) < 1e-2


def test_small_path_host_step():
    """moe_forward_host (host buffers in and out) takes the small path too."""
    spec = _spec(64, 256, 512, 8, 2, True)
    d = wl.make_moe_inputs(spec, device="cuda")
    a = route_args(spec)
    hx, hl = d["hidden"].cpu().pin_memory(), d["router_logits"].cpu().pin_memory()
    pkg.profiler_start()
    y = pkg.moe_forward_host(hx, hl, d["w13"], d["w2"], spec.top_k, a["method"], a["renormalize"],
                             w13_bias=d["w13_bias"], w2_bias=d["w2_bias"],
                             stream=torch.cuda.current_stream())
    ran = pkg.profiler_stop()
    torch.cuda.synchronize()
    assert "small_gemm1" in ran
    w, ids = _route(spec, d)
    check_out(f64(y), _oracle(d, w, ids), "host step small")


@pytest.mark.parametrize("M,H,small", [(128, 64, True), (129, 64, False), (64, 4096, True),
                                       (65, 4096, False)])
def test_small_path_bounds(M, H, small):
    """At most 256 routed items and M * H <= 2^18 take the small path; one
    more token takes the general one; both match the oracle."""
    spec = _spec(M, H, 64, 4, 2, False)
    d = wl.make_moe_inputs(spec, device="cuda")
    w, ids = _route(spec, d)
    pkg.profiler_start()
    y = _forward(d, w, ids)
    ran = pkg.profiler_stop()
    torch.cuda.synchronize()
    assert ("small_gemm1" in ran) == small, sorted(ran)
    check_out(f64(y), _oracle(d, w, ids), f"bounds M={M} H={H}")
