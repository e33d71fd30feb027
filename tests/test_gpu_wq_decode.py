"""GPU parity of the weight-only decode GEMMs -- the path moe_forward_wq takes
for calls of at most 32 tokens: each expert's few rows as the MMA's N, the
quantised weights expanded in registers, GEMM2's K in parts that the
weight-and-reduce adds -- against the oracle ("fused_moe.py 分析", "WNA16
路径" and "5. 特殊量化格式处理": the layer on the dequantised weights), for
every format, group size and zero-point choice; against the grouped
tensor-core path on the same call; with duplicate expert ids in a token (an
expert holding more rows than one pass takes); and at the Mixtral-8x7B decode
shape (M = 16) on every token."""
import numpy as np
import pytest
import torch

import oracle
import mixture_experts_ffn_softmax_gb300 as pkg
from mixture_experts_ffn_softmax_gb300 import workloads as wl

from helpers import check_out, f64
from test_gpu_wq import CASES, LazyDequant, _oracle_dequant, _route

pytestmark = pytest.mark.gpu

# (M, H, I, E, top_k): one, two and four 8-row tiles per pass; a GEMM2 K
# (= I) ending in half a 64-row stage; few of many experts touched; a K long
# enough for GEMM2 to be split into many parts
SHAPES = [(16, 512, 640, 8, 2), (5, 256, 96, 6, 3), (32, 128, 256, 64, 4), (1, 64, 64, 4, 2),
          (9, 192, 1024, 3, 2)]


@pytest.fixture
def decode_restore():
    yield
    pkg.set_wq_decode(True)


def _spec(M, H, I, E, k, bias=True):
    return wl.SMALL_SPECS["mixtral_small"].scaled("wq_decode", M=M, H=H, I=I, E=E, top_k=k,
                                                   bias=bias)


def _biases(spec, seed=7):
    g = torch.Generator(device="cuda").manual_seed(seed)
    b13 = (torch.randn(spec.E, 2 * spec.I, generator=g, device="cuda") * 0.05).bfloat16()
    b2 = (torch.randn(spec.E, spec.H, generator=g, device="cuda") * 0.05).bfloat16()
    return b13, b2


def _run(d, w, ids, fmt, q, b13=None, b2=None, ws=None):
    return pkg.moe_forward_wq(d["hidden"], w, ids, fmt, q["w13_q"], q["w2_q"], q["w13_scale"],
                              q["w2_scale"], q["w13_zero"], q["w2_zero"], q["group_size"], b13, b2,
                              workspace=ws)


@pytest.mark.parametrize("fmt,G,zero", CASES)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "M%d_H%d_I%d_E%d_k%d" % s)
def test_decode_layer_matches_oracle(shape, fmt, G, zero):
    spec = _spec(*shape)
    if spec.H % G or spec.I % G:
        pytest.skip("group size does not divide H and I")
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    q = wl.make_wq_weights(spec, fmt, G, device="cuda", zero=zero)
    b13, b2 = _biases(spec)
    w32, ids = _route(spec, d)
    ws = pkg.alloc_workspace(pkg.workspace_size(spec.M, spec.H, spec.I, spec.E, spec.top_k,
                                                "separate"))
    y = _run(d, torch.from_numpy(w32).cuda(), torch.from_numpy(ids).cuda(), fmt, q, b13, b2, ws)
    torch.cuda.synchronize()
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 0
    w13 = _oracle_dequant(fmt, q["w13_q"], q["w13_scale"], q["w13_zero"])
    w2 = _oracle_dequant(fmt, q["w2_q"], q["w2_scale"], q["w2_zero"])
    ref = oracle.forward_wq(f64(d["hidden"]), w32.astype(np.float64), ids, w13, w2, f64(b13),
                            f64(b2))
    check_out(f64(y), ref, f"decode {shape} {fmt} G={G} zero={zero}")


@pytest.mark.parametrize("fmt,G", [("int4", 128), ("int4", 32), ("int8", 64), ("mxfp4", 32),
                                   ("mxfp6_e3m2", 32), ("mxfp6_e2m3", 32)])
def test_decode_equals_grouped_gemm_path(fmt, G, decode_restore):
    """The same call through the decode GEMMs and through the grouped
    tensor-core GEMMs: equal up to fp32 summation order (and the bf16
    rounding of z that follows from it)."""
    spec = _spec(16, 512, 640, 8, 2)
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    q = wl.make_wq_weights(spec, fmt, G, device="cuda")
    b13, b2 = _biases(spec)
    w, ids = pkg.moe_route(d["router_logits"], spec.top_k, "softmax", True)
    ys = {}
    for on in (True, False):
        pkg.set_wq_decode(on)
        ys[on] = _run(d, w, ids, fmt, q, b13, b2)
        torch.cuda.synchronize()
    check_out(f64(ys[True]), f64(ys[False]), f"{fmt} decode vs grouped")


@pytest.mark.parametrize("fmt,G", [("int4", 64), ("mxfp4", 32), ("int8", 128)])
def test_decode_duplicate_ids_take_row_groups(fmt, G):
    """Caller-supplied ids may repeat an expert within a token, so an expert
    can hold more rows than the call has tokens: with M = 8 (one 8-row tile
    per pass) and every token's four items on experts 0..1, experts hold up
    to 32 rows, taken in row groups."""
    M, H, I, E, k = 8, 128, 256, 4, 4
    spec = _spec(M, H, I, E, k)
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    q = wl.make_wq_weights(spec, fmt, G, device="cuda")
    b13, b2 = _biases(spec)
    gen = torch.Generator().manual_seed(11)
    ids = torch.randint(0, 2, (M, k), generator=gen, dtype=torch.int32)
    ids[0] = 0                      # expert 0 gets at least 4 items of token 0
    w = torch.rand(M, k, generator=gen)
    ws = pkg.alloc_workspace(pkg.workspace_size(M, H, I, E, k, "separate"))
    y = _run(d, w.cuda(), ids.cuda(), fmt, q, b13, b2, ws)
    torch.cuda.synchronize()
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 0
    assert int((ids == 0).sum()) > 8 or int((ids == 1).sum()) > 8
    w13 = _oracle_dequant(fmt, q["w13_q"], q["w13_scale"], q["w13_zero"])
    w2 = _oracle_dequant(fmt, q["w2_q"], q["w2_scale"], q["w2_zero"])
    ref = oracle.forward_wq(f64(d["hidden"]), w.numpy().astype(np.float64), ids.numpy(), w13, w2,
                            f64(b13), f64(b2))
    check_out(f64(y), ref, f"{fmt} duplicate ids")


def test_decode_dropped_items_and_empty_call():
    """Items routed to an id outside [0, E) are dropped (error word set) and
    contribute nothing; the others match the oracle on the remaining items."""
    M, H, I, E, k = 12, 128, 128, 6, 2
    spec = _spec(M, H, I, E, k, bias=False)
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    q = wl.make_wq_weights(spec, "int4", 64, device="cuda")
    w, ids = pkg.moe_route(d["router_logits"], k, "softmax", True)
    ids = ids.clone()
    ids[3, 1] = E + 2
    ws = pkg.alloc_workspace(pkg.workspace_size(M, H, I, E, k, "separate"))
    y = _run(d, w, ids, "int4", q, ws=ws)
    torch.cuda.synchronize()
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 4   # MOE_ERR_BAD_EXPERT_ID
    wk = w.cpu().numpy().astype(np.float64)
    wk[3, 1] = 0.0
    idk = ids.cpu().numpy().copy()
    idk[3, 1] = 0
    w13 = _oracle_dequant("int4", q["w13_q"], q["w13_scale"], q["w13_zero"])
    w2 = _oracle_dequant("int4", q["w2_q"], q["w2_scale"], q["w2_zero"])
    check_out(f64(y), oracle.forward_wq(f64(d["hidden"]), wk, idk, w13, w2), "dropped item")


@pytest.mark.parametrize("fmt,G", [("int4", 128), ("mxfp4", 32)])
def test_decode_full_size_mixtral_every_token(fmt, G):
    """Mixtral-8x7B shape at decode (M = 16, H = 4096, I = 14336, E = 8,
    k = 2): every token against the oracle, which dequantises the experts
    one at a time."""
    spec = wl.SPECS["mixtral_decode"]
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    q = wl.make_wq_weights(spec, fmt, G, device="cuda")
    w, ids = pkg.moe_route(d["router_logits"], spec.top_k, "softmax", True)
    ws = pkg.alloc_workspace(pkg.workspace_size(spec.M, spec.H, spec.I, spec.E, spec.top_k,
                                                "separate"))
    y = _run(d, w, ids, fmt, q, ws=ws)
    torch.cuda.synchronize()
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 0
    ref = oracle.forward_wq(f64(d["hidden"]), w.cpu().numpy().astype(np.float64),
                            ids.cpu().numpy(),
                            LazyDequant(fmt, q["w13_q"], q["w13_scale"], q["w13_zero"]),
                            LazyDequant(fmt, q["w2_q"], q["w2_scale"], q["w2_zero"]))
    check_out(f64(y), ref, f"mixtral decode {fmt}")
