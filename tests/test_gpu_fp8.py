"""GPU parity of the FP8 W8A8 layer (moe_forward_fp8) against the oracle's
FP8 layer: E4M3 weights with per-channel or per-expert scales, activations
quantised per row before each GEMM.  Same output bar as the bf16 layer
(relative L2 <= 1e-2, max abs <= 5e-2 * RMS) against the oracle's FP8
computation."""
import numpy as np
import pytest
import torch

import oracle
import mixture_experts_ffn_softmax_gb300 as pkg
from mixture_experts_ffn_softmax_gb300 import workloads as wl

from helpers import LazyF64, check_out, f64, route_args

pytestmark = pytest.mark.gpu


def _route(spec, d):
    a = route_args(spec)
    w, ids, _ = oracle.route(f64(d["router_logits"]), a["top_k"], a["method"], a["renormalize"],
                             a["k_group"], a["group_count"], a["group_select_mode"],
                             a["routed_scaling_factor"])
    return w.astype(np.float32), ids


@pytest.mark.parametrize("tiles", ["single", "pairs"])
@pytest.mark.parametrize("per_channel", [True, False])
@pytest.mark.parametrize("name", ["tiny", "mixtral_small", "deepseek_small", "qwen_small"])
def test_fp8_small_workloads(name, per_channel, tiles):
    spec = wl.SMALL_SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda")
    q = wl.make_fp8_weights(spec, device="cuda", per_channel=per_channel)
    w32, ids = _route(spec, d)
    pkg.set_gemm_tiles(tiles)
    try:
        y = pkg.moe_forward_fp8(d["hidden"], torch.from_numpy(w32).cuda(),
                                torch.from_numpy(ids).cuda(), q["w13_q"], q["w2_q"],
                                q["w13_scale"], q["w2_scale"], d["w13_bias"], d["w2_bias"])
        torch.cuda.synchronize()
    finally:
        pkg.set_gemm_tiles("auto")
    ref = oracle.forward_fp8(f64(d["hidden"]), w32.astype(np.float64), ids, f64(q["w13_q"]),
                             f64(q["w2_q"]), f64(q["w13_scale"]), f64(q["w2_scale"]),
                             f64(d["w13_bias"]), f64(d["w2_bias"]))
    check_out(f64(y), ref, f"{name} fp8")


def test_fp8_full_size_mixtral_sampled():
    spec = wl.SPECS["mixtral_prefill"]
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    q = wl.make_fp8_weights(spec, device="cuda")
    w, ids = pkg.moe_route(d["router_logits"], spec.top_k, "softmax", True)
    ws = pkg.alloc_workspace(pkg.workspace_size_fp8(spec.M, spec.H, spec.I, spec.E, spec.top_k))
    y = pkg.moe_forward_fp8(d["hidden"], w, ids, q["w13_q"], q["w2_q"], q["w13_scale"],
                            q["w2_scale"], workspace=ws)
    torch.cuda.synchronize()
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 0
    sel = np.sort(np.random.default_rng(0).choice(spec.M, 16, replace=False))
    ref = oracle.forward_fp8(f64(d["hidden"])[sel], w.cpu().numpy()[sel].astype(np.float64),
                             ids.cpu().numpy()[sel], LazyF64(q["w13_q"]), LazyF64(q["w2_q"]),
                             f64(q["w13_scale"]), f64(q["w2_scale"]))
    check_out(f64(y)[sel], ref, "mixtral fp8")


def test_fp8_close_to_bf16_layer_with_dequantised_weights():
    """Sanity of scale placement: the FP8 layer is within FP8 quantisation
    error of the bf16 layer run on the dequantised weights."""
    spec = wl.SMALL_SPECS["mixtral_small"]
    d = wl.make_moe_inputs(spec, device="cuda")
    q = wl.make_fp8_weights(spec, device="cuda")
    w32, ids = _route(spec, d)
    tw, tids = torch.from_numpy(w32).cuda(), torch.from_numpy(ids).cuda()
    y8 = pkg.moe_forward_fp8(d["hidden"], tw, tids, q["w13_q"], q["w2_q"], q["w13_scale"],
                             q["w2_scale"])
    w13 = (q["w13_q"].float() * q["w13_scale"][:, None, :]).bfloat16()
    w2 = (q["w2_q"].float() * q["w2_scale"][:, None, :]).bfloat16()
    yb = pkg.moe_forward(d["hidden"], tw, tids, w13, w2)
    torch.cuda.synchronize()
    a, b = f64(y8), f64(yb)
    rel = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert rel < 0.08, rel        # two E4M3 activation quantisations: a few percent


def test_fp8_validation():
    x = torch.zeros(4, 40, device="cuda").bfloat16()          # H % 16 != 0
    w13 = torch.zeros(2, 40, 64, device="cuda", dtype=torch.uint8)
    w2 = torch.zeros(2, 32, 40, device="cuda", dtype=torch.uint8)
    s = torch.ones(2, device="cuda")
    with pytest.raises(pkg.MoEError) as ei:
        pkg.moe_forward_fp8(x, torch.ones(4, 1, device="cuda"),
                            torch.zeros(4, 1, dtype=torch.int32, device="cuda"), w13, w2, s, s)
    assert ei.value.status == 1
