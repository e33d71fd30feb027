"""Several host threads calling the library at once, each on its own stream
with its own workspace: every result equals the one computed alone (the
library's lazily set per-device state and its per-thread copy streams are
safe to share)."""
import threading

import pytest
import torch

import mixture_experts_ffn_softmax_gb300 as pkg
from mixture_experts_ffn_softmax_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _inputs(name, seed):
    spec = wl.SMALL_SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda", seed=seed)
    w, ids = pkg.moe_route(d["router_logits"], spec.top_k, spec.routing_method, spec.renormalize,
                           spec.k_group, spec.group_count, spec.group_select_mode,
                           spec.routed_scaling_factor)
    torch.cuda.synchronize()
    return spec, d, w, ids


def _forward(spec, d, w, ids, stream, ws):
    with torch.cuda.stream(stream):
        return pkg.moe_forward(d["hidden"], w, ids, d["w13"], d["w2"], d["w13_bias"],
                               d["w2_bias"], workspace=ws, stream=stream)


def _host_step(spec, d, stream):
    with torch.cuda.stream(stream):
        return pkg.moe_forward_host(d["hidden"].cpu().pin_memory(),
                                    d["router_logits"].cpu().pin_memory(), d["w13"], d["w2"],
                                    spec.top_k, spec.routing_method, spec.renormalize,
                                    spec.k_group, spec.group_count, spec.group_select_mode,
                                    spec.routed_scaling_factor, d["w13_bias"], d["w2_bias"],
                                    stream=stream)


def test_concurrent_threads_match_serial():
    jobs = [_inputs(name, seed) for seed, name in enumerate(
        ["mixtral_small", "deepseek_small", "qwen_small", "tiny"])]
    want_dev, want_host = [], []
    for spec, d, w, ids in jobs:
        ws = pkg.alloc_workspace(pkg.workspace_size(spec.M, spec.H, spec.I, spec.E, spec.top_k))
        s = torch.cuda.Stream()
        want_dev.append(_forward(spec, d, w, ids, s, ws))
        want_host.append(_host_step(spec, d, s))
        s.synchronize()
    got = [[None, None] for _ in jobs]
    errors = []

    def run(i):
        try:
            spec, d, w, ids = jobs[i]
            ws = pkg.alloc_workspace(pkg.workspace_size(spec.M, spec.H, spec.I, spec.E,
                                                        spec.top_k))
            s = torch.cuda.Stream()
            for _ in range(5):
                got[i][0] = _forward(spec, d, w, ids, s, ws)
                got[i][1] = _host_step(spec, d, s)
            s.synchronize()
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(len(jobs)):
        assert torch.equal(got[i][0], want_dev[i])
        assert torch.equal(got[i][1], want_host[i])


def test_default_stream_is_the_current_stream():
    """With no stream given the binding launches on torch's current stream:
    the default one, one entered with torch.cuda.stream, and in another
    host thread that thread's own."""
    from mixture_experts_ffn_softmax_gb300 import _stream
    assert _stream() == torch.cuda.current_stream().cuda_stream
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert _stream() == s.cuda_stream
    assert _stream() == torch.cuda.current_stream().cuda_stream
    seen = {}

    def other():
        t = torch.cuda.Stream()
        with torch.cuda.stream(t):
            seen["got"], seen["want"] = _stream(), t.cuda_stream

    th = threading.Thread(target=other)
    th.start()
    th.join()
    assert seen["got"] == seen["want"]
