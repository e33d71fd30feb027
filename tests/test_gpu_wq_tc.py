"""GPU parity of the int4 decode GEMMs on tcgen05, the path moe_forward_wq
takes for calls of at most 32 tokens when the codes repacked along K are
given: the repacked layout bit for bit against a numpy restatement of its
definition; the layer against the oracle ("fused_moe.py 分析", "WNA16 路径":
the layer on the dequantised weights) for group sizes 128 and 256, with and
without zero points, 16- and 32-row passes; against the mma.sync decode GEMMs
on the same call; with duplicate expert ids (row groups); groups of 64 rows
left to the mma.sync path; and at the Mixtral-8x7B decode shape on every
token."""
import numpy as np
import pytest
import torch

import oracle
import mixture_experts_ffn_softmax_gb300 as pkg
from mixture_experts_ffn_softmax_gb300 import workloads as wl

from helpers import check_out, f64
from test_gpu_wq import LazyDequant, _oracle_dequant, _route

pytestmark = pytest.mark.gpu

# (M, H, I, E, top_k): one 256-column unit per expert and part; GEMM2 parts
# ending inside a group; few of many experts touched; 32-row passes; one
# token; a long GEMM2 K split into parts
SHAPES = [(16, 256, 256, 8, 2), (5, 256, 384, 6, 3), (32, 256, 128, 16, 4), (1, 256, 128, 4, 2),
          (9, 256, 1024, 3, 2), (24, 512, 640, 5, 2)]
GROUPS = [(128, True), (128, False), (256, True)]


def _spec(M, H, I, E, k, bias=True):
    return wl.SMALL_SPECS["mixtral_small"].scaled("wq_tc", M=M, H=H, I=I, E=E, top_k=k, bias=bias)


def _biases(spec, seed=7):
    g = torch.Generator(device="cuda").manual_seed(seed)
    b13 = (torch.randn(spec.E, 2 * spec.I, generator=g, device="cuda") * 0.05).bfloat16()
    b2 = (torch.randn(spec.E, spec.H, generator=g, device="cuda") * 0.05).bfloat16()
    return b13, b2


def _packed(q):
    return pkg.wq_pack_k("int4", q["w13_q"]), pkg.wq_pack_k("int4", q["w2_q"])


def _run(d, w, ids, q, packed, b13=None, b2=None, ws=None):
    p13, p2 = packed if packed is not None else (None, None)
    return pkg.moe_forward_wq(d["hidden"], w, ids, "int4", q["w13_q"], q["w2_q"], q["w13_scale"],
                              q["w2_scale"], q["w13_zero"], q["w2_zero"], q["group_size"], b13, b2,
                              workspace=ws, w13_kpack=p13, w2_kpack=p2)


def _pack_reference(codes):
    """The documented layout, restated: word w of column n holds K rows
    8w..8w+7, row 8w + 2t in nibble t and row 8w + 2t + 1 in nibble t + 4."""
    c = codes.cpu().numpy()
    E, K, half = c.shape
    q = np.empty((E, K, 2 * half), np.uint32)
    q[:, :, 0::2] = c & 0xF
    q[:, :, 1::2] = c >> 4
    q = q.transpose(0, 2, 1).reshape(E, 2 * half, K // 8, 8)   # [E, N, word, row in word]
    words = np.zeros((E, 2 * half, K // 8), np.uint32)
    for t in range(4):
        words |= q[..., 2 * t] << (4 * t)
        words |= q[..., 2 * t + 1] << (4 * (t + 4))
    return words.view(np.uint8).reshape(E, 2 * half, K // 2)


@pytest.mark.parametrize("shape", [(3, 64, 40), (2, 256, 128), (1, 8, 2)])
def test_pack_k_layout_bit_exact(shape):
    E, K, N = shape
    g = torch.Generator().manual_seed(5)
    codes = torch.randint(0, 256, (E, K, N // 2), generator=g, dtype=torch.uint8)
    got = pkg.wq_pack_k("int4", codes.cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got.cpu().numpy(), _pack_reference(codes))


def test_pack_k_rejects_other_formats():
    codes = torch.zeros(1, 64, 32, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkg.MoEError):
        pkg.wq_pack_k("mxfp4", codes)


@pytest.mark.parametrize("G,zero", GROUPS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "M%d_H%d_I%d_E%d_k%d" % s)
def test_tc_layer_matches_oracle(shape, G, zero):
    spec = _spec(*shape)
    if spec.H % G or spec.I % G:
        pytest.skip("group size does not divide H and I")
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    q = wl.make_wq_weights(spec, "int4", G, device="cuda", zero=zero)
    b13, b2 = _biases(spec)
    w32, ids = _route(spec, d)
    ws = pkg.alloc_workspace(pkg.workspace_size(spec.M, spec.H, spec.I, spec.E, spec.top_k,
                                                "separate"))
    packed = _packed(q)
    pkg.profiler_start()
    y = _run(d, torch.from_numpy(w32).cuda(), torch.from_numpy(ids).cuda(), q, packed, b13,
             b2, ws)
    ran = pkg.profiler_stop()
    torch.cuda.synchronize()
    assert "gemm1_swiglu_int4_tc" in ran and "gemm2_int4_tc" in ran, sorted(ran)
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 0
    w13 = _oracle_dequant("int4", q["w13_q"], q["w13_scale"], q["w13_zero"])
    w2 = _oracle_dequant("int4", q["w2_q"], q["w2_scale"], q["w2_zero"])
    ref = oracle.forward_wq(f64(d["hidden"]), w32.astype(np.float64), ids, w13, w2, f64(b13),
                            f64(b2))
    check_out(f64(y), ref, f"tc {shape} G={G} zero={zero}")


def test_tc_equals_register_decode():
    """The same call through the tcgen05 decode GEMMs and the mma.sync ones
    (which round each dequantised weight to bf16): equal within the bar."""
    spec = _spec(16, 512, 640, 8, 2)
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    q = wl.make_wq_weights(spec, "int4", 128, device="cuda")
    b13, b2 = _biases(spec)
    w, ids = pkg.moe_route(d["router_logits"], spec.top_k, "softmax", True)
    y_tc = _run(d, w, ids, q, _packed(q), b13, b2)
    y_reg = _run(d, w, ids, q, None, b13, b2)
    torch.cuda.synchronize()
    check_out(f64(y_tc), f64(y_reg), "tc vs register decode")


def test_tc_duplicate_ids_take_row_groups():
    """Experts holding more rows than a 16-row pass (duplicate ids within a
    token) are taken in row groups."""
    M, H, I, E, k = 8, 256, 256, 4, 4
    spec = _spec(M, H, I, E, k)
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    q = wl.make_wq_weights(spec, "int4", 128, device="cuda")
    b13, b2 = _biases(spec)
    gen = torch.Generator().manual_seed(11)
    ids = torch.randint(0, 2, (M, k), generator=gen, dtype=torch.int32)
    ids[0] = 0
    w = torch.rand(M, k, generator=gen)
    assert int((ids == 0).sum()) > 16 or int((ids == 1).sum()) > 16
    ws = pkg.alloc_workspace(pkg.workspace_size(M, H, I, E, k, "separate"))
    y = _run(d, w.cuda(), ids.cuda(), q, _packed(q), b13, b2, ws)
    torch.cuda.synchronize()
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 0
    w13 = _oracle_dequant("int4", q["w13_q"], q["w13_scale"], q["w13_zero"])
    w2 = _oracle_dequant("int4", q["w2_q"], q["w2_scale"], q["w2_zero"])
    ref = oracle.forward_wq(f64(d["hidden"]), w.numpy().astype(np.float64), ids.numpy(), w13, w2,
                            f64(b13), f64(b2))
    check_out(f64(y), ref, "tc duplicate ids")


def test_group_64_takes_the_register_decode():
    """Groups of 64 rows are shorter than a stage of the tcgen05 kernels: the
    call takes the mma.sync decode GEMMs even with the repacked codes given,
    and matches the oracle."""
    spec = _spec(16, 256, 256, 8, 2)
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    q = wl.make_wq_weights(spec, "int4", 64, device="cuda")
    w32, ids = _route(spec, d)
    pkg.profiler_start()
    y = _run(d, torch.from_numpy(w32).cuda(), torch.from_numpy(ids).cuda(), q, _packed(q))
    ran = pkg.profiler_stop()
    torch.cuda.synchronize()
    assert "gemm1_swiglu_int4_decode" in ran and "gemm1_swiglu_int4_tc" not in ran, sorted(ran)
    w13 = _oracle_dequant("int4", q["w13_q"], q["w13_scale"], q["w13_zero"])
    w2 = _oracle_dequant("int4", q["w2_q"], q["w2_scale"], q["w2_zero"])
    ref = oracle.forward_wq(f64(d["hidden"]), w32.astype(np.float64), ids, w13, w2)
    check_out(f64(y), ref, "group 64 register decode")


def test_tc_full_size_mixtral_every_token():
    """Mixtral-8x7B shape at decode (M = 16, H = 4096, I = 14336, E = 8,
    k = 2), int4 group 128 with zero points: every token against the oracle."""
    spec = wl.SPECS["mixtral_decode"]
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    q = wl.make_wq_weights(spec, "int4", 128, device="cuda")
    w, ids = pkg.moe_route(d["router_logits"], spec.top_k, "softmax", True)
    ws = pkg.alloc_workspace(pkg.workspace_size(spec.M, spec.H, spec.I, spec.E, spec.top_k,
                                                "separate"))
    y = _run(d, w, ids, q, _packed(q), ws=ws)
    torch.cuda.synchronize()
    assert pkg.read_error(pkg.workspace_error_word(ws)) == 0
    ref = oracle.forward_wq(f64(d["hidden"]), w.cpu().numpy().astype(np.float64),
                            ids.cpu().numpy(),
                            LazyDequant("int4", q["w13_q"], q["w13_scale"], q["w13_zero"]),
                            LazyDequant("int4", q["w2_q"], q["w2_scale"], q["w2_zero"]))
    check_out(f64(y), ref, "mixtral decode int4 tc")
