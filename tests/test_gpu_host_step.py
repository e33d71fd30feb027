"""The host-memory step (moe_forward_host): host inputs and output, the
copies inside the call.  Its output equals routing + the device forward on
the same inputs bit for bit, also when the call is captured in a CUDA graph
and replayed on new host data."""
import pytest
import torch

import mixture_experts_ffn_softmax_gb300 as pkg
from mixture_experts_ffn_softmax_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _route_kw(spec):
    return dict(top_k=spec.top_k, routing_method=spec.routing_method,
                renormalize=spec.renormalize, k_group=spec.k_group,
                group_count=spec.group_count, group_select_mode=spec.group_select_mode,
                routed_scaling_factor=spec.routed_scaling_factor)


def _device_layer(spec, d):
    w, ids = pkg.moe_route(d["router_logits"], spec.top_k, spec.routing_method, spec.renormalize,
                           spec.k_group, spec.group_count, spec.group_select_mode,
                           spec.routed_scaling_factor)
    return pkg.moe_forward(d["hidden"], w, ids, d["w13"], d["w2"], d["w13_bias"], d["w2_bias"])


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("name", ["tiny", "mixtral_small", "deepseek_small", "qwen_small"])
def test_host_step_equals_device_layer(name, pinned):
    spec = wl.SMALL_SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda")
    hx = d["hidden"].cpu()
    hl = d["router_logits"].cpu()
    if pinned:
        hx, hl = hx.pin_memory(), hl.pin_memory()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = pkg.moe_forward_host(hx, hl, d["w13"], d["w2"], w13_bias=d["w13_bias"],
                                 w2_bias=d["w2_bias"], stream=s, **_route_kw(spec))
    s.synchronize()
    want = _device_layer(spec, d)
    torch.cuda.synchronize()
    assert torch.equal(y, want.cpu())


@pytest.mark.parametrize("name", ["mixtral_prefill", "qwen_skew", "deepseek_m64"])
def test_host_step_full_size(name):
    """Full-size layers: the Qwen shape runs as two token chunks with the
    copies overlapping the compute, the Mixtral and DeepSeek shapes in one
    pass; the output equals one device pass bit for bit."""
    spec = wl.SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda")
    hx, hl = d["hidden"].cpu().pin_memory(), d["router_logits"].cpu().pin_memory()
    y = pkg.moe_forward_host(hx, hl, d["w13"], d["w2"], w13_bias=d["w13_bias"],
                             w2_bias=d["w2_bias"], stream=torch.cuda.current_stream(),
                             **_route_kw(spec))
    torch.cuda.synchronize()
    assert torch.equal(y, _device_layer(spec, d).cpu())


def test_host_step_graph_replay():
    spec = wl.SMALL_SPECS["qwen_small"]
    d = wl.make_moe_inputs(spec, device="cuda")
    hx = d["hidden"].cpu().pin_memory()
    hl = d["router_logits"].cpu().pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    st = pkg.HostStaging(spec.M, spec.H, spec.I, spec.E, spec.top_k)
    kw = dict(w13_bias=d["w13_bias"], w2_bias=d["w2_bias"], out=hy, staging=st,
              **_route_kw(spec))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pkg.moe_forward_host(hx, hl, d["w13"], d["w2"], stream=s, **kw)   # set-up outside
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkg.moe_forward_host(hx, hl, d["w13"], d["w2"], stream=s, **kw)
    for seed in (1, 2):
        new = wl.make_moe_inputs(spec, device="cuda", seed=seed, weights=False)
        hx.copy_(new["hidden"].cpu())
        hl.copy_(new["router_logits"].cpu())
        g.replay()
        torch.cuda.synchronize()
        d["hidden"], d["router_logits"] = new["hidden"], new["router_logits"]
        assert torch.equal(hy, _device_layer(spec, d).cpu())
    assert pkg.read_error(pkg.workspace_error_word(st.workspace)) == 0


def test_host_step_validation_enqueues_nothing():
    spec = wl.SMALL_SPECS["tiny"]
    d = wl.make_moe_inputs(spec, device="cuda")
    hx, hl = d["hidden"].cpu(), d["router_logits"].cpu()
    kw = _route_kw(spec)
    kw["top_k"] = spec.E + 1
    with pytest.raises(pkg.MoEError) as ei:
        pkg.moe_forward_host(hx, hl, d["w13"], d["w2"], **kw)
    assert ei.value.status == 1
    kw = _route_kw(spec)
    y = pkg.moe_forward_host(hx[:0], hl[:0], d["w13"], d["w2"], **kw)   # M = 0: nothing to do
    assert y.shape == (0, spec.H)


@pytest.fixture
def direct_restore():
    yield
    pkg.set_host_out_direct(True)


@pytest.mark.parametrize("name", ["mixtral_small", "qwen_small"])
def test_host_step_output_buffers(name, direct_restore):
    """The output's way back to the host: written by the reduce straight into
    a pinned `out` (the default), through the device staging buffer and a
    copy (switch off, pageable `out`, or a pinned `out` that is not 16-byte
    aligned) -- the same bits every way."""
    spec = wl.SMALL_SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda")
    hx, hl = d["hidden"].cpu().pin_memory(), d["router_logits"].cpu().pin_memory()
    want = _device_layer(spec, d).cpu()
    n = spec.M * spec.H
    outs = {
        "pinned": torch.empty(spec.M, spec.H, dtype=torch.bfloat16).pin_memory(),
        "pageable": torch.empty(spec.M, spec.H, dtype=torch.bfloat16),
        "pinned_unaligned":
            torch.empty(n + 1, dtype=torch.bfloat16).pin_memory()[1:].view(spec.M, spec.H),
    }
    for direct in (True, False):
        pkg.set_host_out_direct(direct)
        for key, out in outs.items():
            out.fill_(float("nan"))
            y = pkg.moe_forward_host(hx, hl, d["w13"], d["w2"], w13_bias=d["w13_bias"],
                                     w2_bias=d["w2_bias"], out=out,
                                     stream=torch.cuda.current_stream(), **_route_kw(spec))
            torch.cuda.synchronize()
            assert y.data_ptr() == out.data_ptr()
            assert torch.equal(out, want), (key, direct)
