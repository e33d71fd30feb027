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


def _quant_cases():
    g = torch.Generator().manual_seed(5)
    H = 272                                                   # 17 16-byte groups: ragged lanes
    rows = [torch.randn(64, H, generator=g),                  # plain values
            torch.randint(-9, 10, (64, H), generator=g).float(),   # tie-heavy small integers
            torch.randint(-448, 449, (32, H), generator=g).float() / 7.0,
            torch.randn(8, H, generator=g) * 1e30,
            torch.randn(8, H, generator=g) * 1e-3,
            torch.zeros(2, H)]                                # all-zero rows: scale 1
    # rows whose quotients sit on E4M3 rounding midpoints: amax fixed at 448 * 2^j
    mids = []
    for j in (-3, 0, 5):
        r = torch.zeros(H)
        v = torch.tensor([1.0625, 2.125, 9.0, 17.0, 68.0, 104.0, 232.0, 440.0, 0.0009765625 * 3])
        r[: v.numel()] = v * 2.0 ** j
        r[-1] = 448.0 * 2.0 ** j
        mids.append(r)
    rows.append(torch.stack(mids))
    tiny = torch.full((1, H), 1e-37)                          # scale below the normal range
    tiny[0, ::3] = -3e-38
    rows.append(tiny)
    return torch.cat(rows).bfloat16()


def test_quant_rows_codes_match_oracle_bit_exactly():
    """The code of each element is an integer decided by floating point: both
    sides decide it in fp32 (scale = amax / 448, quotient x / scale correctly
    rounded), so codes and scales agree exactly."""
    x = _quant_cases()
    q8, s = pkg.moe_quant_rows_fp8(x.cuda())
    torch.cuda.synchronize()
    qo, so = oracle.quantize_rows_e4m3(x.float().numpy())
    np.testing.assert_array_equal(s.cpu().numpy(), so.astype(np.float32))
    got = q8.cpu().float().double().numpy()
    bad = np.argwhere(got != qo)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[:4].tolist()}"


def test_quant_rows_full_size_sampled():
    spec = wl.SPECS["mixtral_prefill"]
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    q8, s = pkg.moe_quant_rows_fp8(d["hidden"])
    torch.cuda.synchronize()
    sel = np.random.default_rng(3).choice(spec.M, 64, replace=False)
    qo, so = oracle.quantize_rows_e4m3(d["hidden"][sel].float().cpu().numpy())
    np.testing.assert_array_equal(s.cpu().numpy()[sel], so.astype(np.float32))
    np.testing.assert_array_equal(q8[sel].cpu().float().double().numpy(), qo)


def test_quant_rows_validation_and_empty():
    pkg.moe_quant_rows_fp8(torch.empty(0, 32, device="cuda").bfloat16())
    with pytest.raises(pkg.MoEError) as ei:
        pkg.moe_quant_rows_fp8(torch.zeros(4, 40, device="cuda").bfloat16())
    assert ei.value.status == 1


@pytest.mark.parametrize("name", ["tiny", "mixtral_small", "deepseek_small"])
def test_fp8_block_scales_small_workloads(name):
    """128 x 128 weight-block scales, activations per (row, group of 128):
    against the oracle's block-wise FP8 layer."""
    spec = wl.SMALL_SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda")
    q = wl.make_fp8_weights(spec, device="cuda", block=True)
    w32, ids = _route(spec, d)
    y = pkg.moe_forward_fp8(d["hidden"], torch.from_numpy(w32).cuda(), torch.from_numpy(ids).cuda(),
                            q["w13_q"], q["w2_q"], q["w13_scale"], q["w2_scale"], d["w13_bias"],
                            d["w2_bias"])
    torch.cuda.synchronize()
    ref = oracle.forward_fp8_block(f64(d["hidden"]), w32.astype(np.float64), ids, f64(q["w13_q"]),
                                   f64(q["w2_q"]), f64(q["w13_scale"]), f64(q["w2_scale"]),
                                   f64(d["w13_bias"]), f64(d["w2_bias"]))
    check_out(f64(y), ref, f"{name} fp8 block")


def test_fp8_block_scales_with_bias_and_ragged_rows():
    """Biases, M not a multiple of the tile, experts with a few rows each."""
    spec = wl.MoESpec(name="block_ragged", M=77, H=256, I=384, E=6, top_k=3,
                      routing_method="softmax", renormalize=True, bias=True)
    d = wl.make_moe_inputs(spec, device="cuda")
    q = wl.make_fp8_weights(spec, device="cuda", block=True)
    w32, ids = _route(spec, d)
    y = pkg.moe_forward_fp8(d["hidden"], torch.from_numpy(w32).cuda(), torch.from_numpy(ids).cuda(),
                            q["w13_q"], q["w2_q"], q["w13_scale"], q["w2_scale"], d["w13_bias"],
                            d["w2_bias"])
    torch.cuda.synchronize()
    ref = oracle.forward_fp8_block(f64(d["hidden"]), w32.astype(np.float64), ids, f64(q["w13_q"]),
                                   f64(q["w2_q"]), f64(q["w13_scale"]), f64(q["w2_scale"]),
                                   f64(d["w13_bias"]), f64(d["w2_bias"]))
    check_out(f64(y), ref, "ragged fp8 block")


@pytest.mark.parametrize("M,H,I,E,k", [(1, 128, 128, 3, 2), (5, 256, 128, 4, 3), (3, 128, 384, 2, 1)])
def test_fp8_block_scales_edge_shapes(M, H, I, E, k):
    """One token or a few, a single 128-wide z group (one z column tile), and
    tiles that are almost all padding: z's codes and group scales come from
    GEMM1's epilogue, whose per-row maxima are exchanged across warps."""
    spec = wl.MoESpec(name="block_edge", M=M, H=H, I=I, E=E, top_k=k,
                      routing_method="softmax", renormalize=True, bias=True)
    d = wl.make_moe_inputs(spec, device="cuda")
    q = wl.make_fp8_weights(spec, device="cuda", block=True)
    w32, ids = _route(spec, d)
    y = pkg.moe_forward_fp8(d["hidden"], torch.from_numpy(w32).cuda(), torch.from_numpy(ids).cuda(),
                            q["w13_q"], q["w2_q"], q["w13_scale"], q["w2_scale"], d["w13_bias"],
                            d["w2_bias"])
    torch.cuda.synchronize()
    ref = oracle.forward_fp8_block(f64(d["hidden"]), w32.astype(np.float64), ids, f64(q["w13_q"]),
                                   f64(q["w2_q"]), f64(q["w13_scale"]), f64(q["w2_scale"]),
                                   f64(d["w13_bias"]), f64(d["w2_bias"]))
    check_out(f64(y), ref, f"fp8 block M={M} H={H} I={I} E={E} k={k}")


def test_fp8_block_scales_full_size_mixtral_sampled():
    spec = wl.SPECS["mixtral_prefill"]
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    q = wl.make_fp8_weights(spec, device="cuda", block=True)
    w, ids = pkg.moe_route(d["router_logits"], spec.top_k, "softmax", True)
    ws = pkg.alloc_workspace(pkg.workspace_size_fp8(spec.M, spec.H, spec.I, spec.E, spec.top_k))
    y = pkg.moe_forward_fp8(d["hidden"], w, ids, q["w13_q"], q["w2_q"], q["w13_scale"],
                            q["w2_scale"], workspace=ws)
    torch.cuda.synchronize()
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 0
    sel = np.sort(np.random.default_rng(2).choice(spec.M, 12, replace=False))
    ref = oracle.forward_fp8_block(f64(d["hidden"])[sel], w.cpu().numpy()[sel].astype(np.float64),
                                   ids.cpu().numpy()[sel], LazyF64(q["w13_q"]), LazyF64(q["w2_q"]),
                                   f64(q["w13_scale"]), f64(q["w2_scale"]))
    check_out(f64(y)[sel], ref, "mixtral fp8 block")


def test_fp8_block_scales_validation():
    spec = wl.MoESpec(name="bad", M=8, H=192, I=256, E=2, top_k=1)   # H % 128 != 0
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    w13 = torch.zeros(2, 192, 512, dtype=torch.uint8, device="cuda")
    w2 = torch.zeros(2, 256, 192, dtype=torch.uint8, device="cuda")
    s13 = torch.ones(2, 1, 4, device="cuda")
    s2 = torch.ones(2, 2, 1, device="cuda")
    with pytest.raises(pkg.MoEError) as ei:
        pkg.moe_forward_fp8(d["hidden"], torch.ones(8, 1, device="cuda"),
                            torch.zeros(8, 1, dtype=torch.int32, device="cuda"), w13, w2, s13, s2)
    assert ei.value.status == 1
