"""GPU parity of the weight-only quantised layer (int4 / int8 with group
scales and zero points, MX FP4) against the oracle: the dequantised weights
bit-exactly, the layer within the output bar (relative L2 <= 1e-2, max abs
<= 5e-2 * RMS), and the fused layer equal to the bf16 layer run on the
dequantised weights."""
import numpy as np
import pytest
import torch

import oracle
import mixture_experts_ffn_softmax_gb300 as pkg
from mixture_experts_ffn_softmax_gb300 import workloads as wl

from helpers import check_out, f64, route_args

pytestmark = pytest.mark.gpu


MX_ELEMENT = {"mxfp4": "e2m1", "mxfp6_e3m2": "e3m2", "mxfp6_e2m3": "e2m3"}


def _oracle_dequant(fmt, q, scale, zero):
    q = q.cpu().numpy()
    if fmt in MX_ELEMENT:
        return oracle.dequant_mx(q, scale.cpu().numpy(), MX_ELEMENT[fmt])
    z = None if zero is None else zero.cpu().numpy()
    return oracle.dequant_int(q, scale.float().cpu().numpy(), z, bits=4 if fmt == "int4" else 8)


class LazyDequant:
    """Indexable per-expert view of quantised weights, dequantised by the
    oracle on the host one expert at a time."""

    def __init__(self, fmt, q, scale, zero):
        self.args = (fmt, q, scale, zero)
        E, K, n = q.shape
        self.shape = (E, K, 2 * n if fmt in ("int4", "mxfp4") else n)
        self._cache = {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self._cache:
            self._cache.clear()
            fmt, q, s, z = self.args
            self._cache[e] = _oracle_dequant(fmt, q[e:e + 1], s[e:e + 1],
                                             None if z is None else z[e:e + 1])[0]
        return self._cache[e]


def _route(spec, d):
    a = route_args(spec)
    w, ids, _ = oracle.route(f64(d["router_logits"]), a["top_k"], a["method"], a["renormalize"],
                             a["k_group"], a["group_count"], a["group_select_mode"],
                             a["routed_scaling_factor"])
    return w.astype(np.float32), ids


CASES = [("int4", 128, True), ("int4", 32, False), ("int4", 64, True),
         ("int8", 64, True), ("int8", 128, False), ("mxfp4", 32, False),
         ("mxfp6_e3m2", 32, False), ("mxfp6_e2m3", 32, False)]


@pytest.mark.parametrize("fmt,G,zero", CASES)
def test_dequant_weights_bit_exact(fmt, G, zero):
    spec = wl.SMALL_SPECS["mixtral_small"]
    q = wl.make_wq_weights(spec, fmt, G, device="cuda", zero=zero)
    for name in ("w13", "w2"):
        got = pkg.moe_dequant_weights(fmt, q[name + "_q"], q[name + "_scale"], q[name + "_zero"],
                                      q["group_size"])
        torch.cuda.synchronize()
        want = _oracle_dequant(fmt, q[name + "_q"], q[name + "_scale"], q[name + "_zero"])
        np.testing.assert_array_equal(got.float().cpu().numpy(), want.astype(np.float32))


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp6_e3m2", "mxfp6_e2m3"])
def test_dequant_mx_extreme_scales_bit_exact(fmt):
    """Every element code with UE8M0 scales at the ends of the range: bf16
    subnormal results (2^-127), and powers of two far above one."""
    E, K, N = 2, 64, 64
    g = torch.Generator().manual_seed(3)
    if fmt == "mxfp4":
        codes = torch.randint(0, 256, (E, K, N // 2), generator=g, dtype=torch.int32).to(torch.uint8)
    else:
        codes = torch.arange(E * K * N, dtype=torch.int32).reshape(E, K, N).remainder(64)
        codes = codes.to(torch.uint8)
    scale = torch.tensor([0, 1, 2, 100, 127, 130, 200, 250], dtype=torch.uint8)
    scale = scale[torch.randint(0, 8, (E, K // 32, N), generator=g)]
    got = pkg.moe_dequant_weights(fmt, codes.cuda(), scale.cuda(), None, 32)
    torch.cuda.synchronize()
    want = oracle.dequant_mx(codes.numpy(), scale.numpy(), MX_ELEMENT[fmt])
    np.testing.assert_array_equal(got.float().cpu().numpy(), want.astype(np.float32))


@pytest.fixture(params=["single", "pairs"])
def tiles(request):
    pkg.set_gemm_tiles(request.param)
    yield request.param
    pkg.set_gemm_tiles("auto")


@pytest.mark.parametrize("fmt,G,zero", CASES)
@pytest.mark.parametrize("name", ["tiny", "mixtral_small", "deepseek_small", "qwen_small"])
def test_wq_layer_small_workloads(name, fmt, G, zero, tiles):
    spec = wl.SMALL_SPECS[name]
    if spec.H % G or spec.I % G:
        pytest.skip("group size does not divide H and I")
    d = wl.make_moe_inputs(spec, device="cuda")
    q = wl.make_wq_weights(spec, fmt, G, device="cuda", zero=zero)
    b13, b2 = d["w13_bias"], d["w2_bias"]
    w32, ids = _route(spec, d)
    y = pkg.moe_forward_wq(d["hidden"], torch.from_numpy(w32).cuda(), torch.from_numpy(ids).cuda(),
                           fmt, q["w13_q"], q["w2_q"], q["w13_scale"], q["w2_scale"],
                           q["w13_zero"], q["w2_zero"], q["group_size"], b13, b2)
    torch.cuda.synchronize()
    w13 = _oracle_dequant(fmt, q["w13_q"], q["w13_scale"], q["w13_zero"])
    w2 = _oracle_dequant(fmt, q["w2_q"], q["w2_scale"], q["w2_zero"])
    ref = oracle.forward_wq(f64(d["hidden"]), w32.astype(np.float64), ids, w13, w2, f64(b13),
                            f64(b2))
    check_out(f64(y), ref, f"{name} {fmt} G={G} {tiles}")


@pytest.mark.parametrize("mode", ["single", "pairs"])
@pytest.mark.parametrize("fmt", ["int4", "int8", "mxfp4", "mxfp6_e3m2", "mxfp6_e2m3"])
def test_wq_layer_equals_bf16_layer_on_dequantised_weights(fmt, mode):
    """The fused conversion feeds the same bf16 weights to the same MMA
    sequence as the bf16 layer (same tile shape): identical outputs."""
    spec = wl.SMALL_SPECS["mixtral_small"]
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    q = wl.make_wq_weights(spec, fmt, 64, device="cuda")
    w32, ids = _route(spec, d)
    tw, tids = torch.from_numpy(w32).cuda(), torch.from_numpy(ids).cuda()
    w13 = pkg.moe_dequant_weights(fmt, q["w13_q"], q["w13_scale"], q["w13_zero"], q["group_size"])
    w2 = pkg.moe_dequant_weights(fmt, q["w2_q"], q["w2_scale"], q["w2_zero"], q["group_size"])
    pkg.set_gemm_tiles(mode)
    try:
        y = pkg.moe_forward_wq(d["hidden"], tw, tids, fmt, q["w13_q"], q["w2_q"], q["w13_scale"],
                               q["w2_scale"], q["w13_zero"], q["w2_zero"], q["group_size"])
        yb = pkg.moe_forward(d["hidden"], tw, tids, w13, w2, reduce="separate")
        torch.cuda.synchronize()
    finally:
        pkg.set_gemm_tiles("auto")
    assert torch.equal(y, yb)


def test_wq_full_size_mixtral_int4_sampled():
    spec = wl.SPECS["mixtral_prefill"]
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    q = wl.make_wq_weights(spec, "int4", 128, device="cuda")
    w, ids = pkg.moe_route(d["router_logits"], spec.top_k, "softmax", True)
    ws = pkg.alloc_workspace(pkg.workspace_size(spec.M, spec.H, spec.I, spec.E, spec.top_k,
                                                "separate"))
    y = pkg.moe_forward_wq(d["hidden"], w, ids, "int4", q["w13_q"], q["w2_q"], q["w13_scale"],
                           q["w2_scale"], q["w13_zero"], q["w2_zero"], 128, workspace=ws)
    torch.cuda.synchronize()
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 0
    # tokens routed to experts 0 and 1 only: the oracle dequantises two experts
    ids_np = ids.cpu().numpy()
    cand = np.flatnonzero(np.all(np.isin(ids_np, [0, 1]), axis=1))
    assert cand.size >= 12
    sel = np.sort(np.random.default_rng(1).choice(cand, 12, replace=False))
    ref = oracle.forward_wq(f64(d["hidden"])[sel], w.cpu().numpy()[sel].astype(np.float64),
                            ids.cpu().numpy()[sel],
                            LazyDequant("int4", q["w13_q"], q["w13_scale"], q["w13_zero"]),
                            LazyDequant("int4", q["w2_q"], q["w2_scale"], q["w2_zero"]))
    check_out(f64(y)[sel], ref, "mixtral int4")


def test_wq_decode_shape_int4():
    spec = wl.SMALL_SPECS["mixtral_decode_small"]
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    q = wl.make_wq_weights(spec, "int4", 128, device="cuda")
    w32, ids = _route(spec, d)
    y = pkg.moe_forward_wq(d["hidden"], torch.from_numpy(w32).cuda(), torch.from_numpy(ids).cuda(),
                           "int4", q["w13_q"], q["w2_q"], q["w13_scale"], q["w2_scale"],
                           q["w13_zero"], q["w2_zero"], 128)
    torch.cuda.synchronize()
    ref = oracle.forward_wq(f64(d["hidden"]), w32.astype(np.float64), ids,
                            LazyDequant("int4", q["w13_q"], q["w13_scale"], q["w13_zero"]),
                            LazyDequant("int4", q["w2_q"], q["w2_scale"], q["w2_zero"]))
    check_out(f64(y), ref, "mixtral decode int4")


def test_wq_validation():
    spec = wl.SMALL_SPECS["tiny"]
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    q = wl.make_wq_weights(spec, "int4", 64, device="cuda")
    w, ids = pkg.moe_route(d["router_logits"], spec.top_k, "softmax", True)
    args = (d["hidden"], w, ids, "int4", q["w13_q"], q["w2_q"], q["w13_scale"], q["w2_scale"],
            q["w13_zero"], q["w2_zero"])
    for G in (48, 16, 512):                       # not a multiple of 32 / does not divide H
        with pytest.raises(pkg.MoEError) as ei:
            pkg.moe_forward_wq(*args, group_size=G)
        assert ei.value.status == 1
    with pytest.raises(pkg.MoEError):              # zero points for one of the two only
        pkg.moe_forward_wq(d["hidden"], w, ids, "int4", q["w13_q"], q["w2_q"], q["w13_scale"],
                           q["w2_scale"], q["w13_zero"], None, 64)
    with pytest.raises(pkg.MoEError):              # MX FP4 takes no zero points
        pkg.moe_dequant_weights("mxfp4", q["w13_q"],
                                torch.zeros(8, 8, 1024, dtype=torch.uint8, device="cuda"),
                                q["w13_zero"], 32)
    pkg.moe_forward_wq(d["hidden"][:0], w[:0], ids[:0], "int4", q["w13_q"], q["w2_q"],
                       q["w13_scale"], q["w2_scale"], q["w13_zero"], q["w2_zero"], 64)


@pytest.mark.parametrize("fmt,G", [("int4", 128), ("mxfp4", 32), ("int8", 64)])
def test_wq_pair_tiles_every_block_count(fmt, G):
    """CTA-pair tiles hold four row blocks of one expert: experts with 0..9
    row blocks (every remainder mod 4, a ragged last block) give the same
    outputs on pairs as on single-CTA tiles, bit for bit."""
    E, H, I, k = 10, 256, 384, 1
    counts = [0, 128, 256, 384, 512, 640, 700, 896, 1024, 1100]   # rows per expert
    M = sum(counts)
    ids = torch.cat([torch.full((c,), e, dtype=torch.int32) for e, c in enumerate(counts)])
    ids = ids[torch.randperm(M, generator=torch.Generator().manual_seed(5))].view(M, k).cuda()
    w = torch.rand(M, k, generator=torch.Generator().manual_seed(6)).cuda()
    spec = wl.SMALL_SPECS["mixtral_small"].scaled("blocks", M=M, H=H, I=I, E=E, top_k=k)
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    q = wl.make_wq_weights(spec, fmt, G, device="cuda")
    args = (d["hidden"], w, ids, fmt, q["w13_q"], q["w2_q"], q["w13_scale"], q["w2_scale"],
            q["w13_zero"], q["w2_zero"], q["group_size"])
    ys = {}
    for mode in ("single", "pairs"):
        pkg.set_gemm_tiles(mode)
        try:
            ws = pkg.alloc_workspace(pkg.workspace_size(M, H, I, E, k, "separate"))
            ys[mode] = pkg.moe_forward_wq(*args, workspace=ws)
            torch.cuda.synchronize()
            assert pkg.read_error(pkg.workspace_error_word(ws)) == 0
        finally:
            pkg.set_gemm_tiles("auto")
    assert torch.equal(ys["single"], ys["pairs"])
    # and against the oracle on a row sample from every expert
    sel = np.sort(np.concatenate([np.flatnonzero(ids.cpu().numpy()[:, 0] == e)[:3]
                                  for e in range(E) if counts[e]]))
    ref = oracle.forward_wq(f64(d["hidden"])[sel], w.cpu().numpy()[sel].astype(np.float64),
                            ids.cpu().numpy()[sel],
                            LazyDequant(fmt, q["w13_q"], q["w13_scale"], q["w13_zero"]),
                            LazyDequant(fmt, q["w2_q"], q["w2_scale"], q["w2_zero"]))
    check_out(f64(ys["pairs"])[sel], ref, f"{fmt} every block count")
