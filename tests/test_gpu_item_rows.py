"""The separate weight-and-reduce with its item rows as fp32 and as fp16 with
a power-of-two exponent per row and 32-column chunk ("fused_moe.py 分析": the
weighted rows o_r, summed per token by the reduce): both formats against the
oracle on every small workload and the edge shapes, with both tile shapes;
outputs whose magnitudes exceed fp16's range (the exponents at work); the
per-channel FP8 layer; and the two formats against each other at the full
Qwen-MoE shape."""
import numpy as np
import pytest
import torch

import oracle
import mixture_experts_ffn_softmax_gb300 as pkg
from mixture_experts_ffn_softmax_gb300 import workloads as wl

from helpers import check_out, f64

pytestmark = pytest.mark.gpu


@pytest.fixture
def rows_restore():
    yield
    pkg.set_item_rows("auto")
    pkg.set_gemm_tiles("auto")


def _oracle_route(spec, logits):
    w, ids, _ = oracle.route(f64(logits), spec.top_k, spec.routing_method, spec.renormalize,
                             spec.k_group, spec.group_count, spec.group_select_mode,
                             spec.routed_scaling_factor)
    return w.astype(np.float32), ids


def _layer(spec, d, w, ids, scale=1.0):
    x = d["hidden"] if scale == 1.0 else (d["hidden"].float() * scale).bfloat16()
    y = pkg.moe_forward(x, torch.from_numpy(w).cuda(), torch.from_numpy(ids).cuda(), d["w13"],
                        d["w2"], d["w13_bias"], d["w2_bias"], reduce="separate")
    torch.cuda.synchronize()
    ref = oracle.forward(f64(x), w.astype(np.float64), ids, f64(d["w13"]), f64(d["w2"]),
                         f64(d["w13_bias"]), f64(d["w2_bias"]))
    return y, ref


@pytest.mark.parametrize("tiles", ["single", "pairs"])
@pytest.mark.parametrize("fmt", ["fp16", "fp32"])
@pytest.mark.parametrize("name", sorted(wl.SMALL_SPECS))
def test_item_row_formats_small_workloads(name, fmt, tiles, rows_restore):
    spec = wl.SMALL_SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda")
    w, ids = _oracle_route(spec, d["router_logits"])
    pkg.set_item_rows(fmt)
    pkg.set_gemm_tiles(tiles)
    y, ref = _layer(spec, d, w, ids)
    check_out(f64(y), ref, f"{name} {fmt} {tiles}")


@pytest.mark.parametrize("shape", [(5, 136, 72, 3, 3), (70, 8, 24, 3, 1), (300, 256, 320, 16, 4),
                                   (40, 64, 128, 8, 4), (20000, 64, 64, 8, 4)])
def test_item_rows_fp16_edge_shapes(shape, rows_restore):
    """H not a multiple of 32 (a ragged last chunk), H = 8 (one chunk of eight
    columns), top_k = E, and 20000 tokens (two token chunks of the forward, each
    with its own rows and exponents)."""
    M, H, I, E, k = shape
    spec = wl.SMALL_SPECS["mixtral_small"].scaled("rows", M=M, H=H, I=I, E=E, top_k=k)
    d = wl.make_moe_inputs(spec, device="cuda")
    w, ids = _oracle_route(spec, d["router_logits"])
    pkg.set_item_rows("fp16")
    y, ref = _layer(spec, d, w, ids)
    check_out(f64(y), ref, f"fp16 rows {shape}")


@pytest.mark.parametrize("scale", [2.0 ** 12, 2.0 ** 24])
def test_item_rows_fp16_beyond_fp16_range(scale, rows_restore):
    """Inputs scaled so that the weighted rows reach ~1e4 / ~5e7, past fp16's
    65504: the exponents keep every chunk finite and the result matches the
    oracle as closely as at unit scale."""
    spec = wl.SMALL_SPECS["qwen_small"]
    d = wl.make_moe_inputs(spec, device="cuda")
    w, ids = _oracle_route(spec, d["router_logits"])
    pkg.set_item_rows("fp16")
    y, ref = _layer(spec, d, w, ids, scale=scale)
    assert np.abs(ref).max() > 65504.0
    check_out(f64(y), ref, f"fp16 rows, inputs x {scale:g}")


def test_item_rows_fp16_fp8_layer(rows_restore):
    spec = wl.SPECS["mixtral_prefill"].scaled("rows_fp8", M=300, H=512, I=640, top_k=4)
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    w, ids = pkg.moe_route(d["router_logits"], spec.top_k, "softmax", True)
    q = wl.make_fp8_weights(spec, device="cuda")
    ys = {}
    for fmt in ("fp32", "fp16"):
        pkg.set_item_rows(fmt)
        ys[fmt] = pkg.moe_forward_fp8(d["hidden"], w, ids, q["w13_q"], q["w2_q"], q["w13_scale"],
                                      q["w2_scale"])
        torch.cuda.synchronize()
    # the same quantised operands and MMAs: the formats differ by the fp16
    # rounding of each weighted row before the k-sum
    check_out(f64(ys["fp16"]), f64(ys["fp32"]), "fp8 layer fp16 vs fp32 rows")
    ref = oracle.forward_fp8(f64(d["hidden"]), w.cpu().numpy().astype(np.float64),
                             ids.cpu().numpy(), f64(q["w13_q"]), f64(q["w2_q"]),
                             f64(q["w13_scale"]), f64(q["w2_scale"]))
    check_out(f64(ys["fp16"]), ref, "fp8 layer fp16 rows vs oracle")


def test_item_row_formats_agree_full_size_qwen(rows_restore):
    spec = wl.SPECS["qwen_skew"]
    d = wl.make_moe_inputs(spec, device="cuda")
    w, ids = pkg.moe_route(d["router_logits"], spec.top_k, spec.routing_method, spec.renormalize)
    ys = {}
    for fmt in ("fp32", "fp16"):
        pkg.set_item_rows(fmt)
        ws = pkg.alloc_workspace(pkg.workspace_size(spec.M, spec.H, spec.I, spec.E, spec.top_k))
        ys[fmt] = pkg.moe_forward(d["hidden"], w, ids, d["w13"], d["w2"], d["w13_bias"],
                                  d["w2_bias"], ws, reduce="separate")
        torch.cuda.synchronize()
        assert pkg.read_error(pkg.workspace_error_word(ws)) == 0
    check_out(f64(ys["fp16"]), f64(ys["fp32"]), "qwen fp16 vs fp32 item rows")
