"""GPU parity of moe_route against the oracle: ids bit-exact (ties to the
lower expert id), weights within 1e-5 absolute."""
import json
import math
import os

import numpy as np
import pytest
import torch

import mixture_experts_ffn_softmax_gb300 as pkg
from mixture_experts_ffn_softmax_gb300 import workloads as wl

from helpers import check_route, route_args

pytestmark = pytest.mark.gpu


def _gpu_route(logits, a):
    w, ids = pkg.moe_route(logits, a["top_k"], a["method"], a["renormalize"], a["k_group"],
                           a["group_count"], a["group_select_mode"], a["routed_scaling_factor"])
    torch.cuda.synchronize()
    return w.cpu().numpy(), ids.cpu().numpy()


@pytest.mark.parametrize("name", sorted(wl.SPECS))
def test_route_full_size_workloads(name):
    spec = wl.SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    a = route_args(spec)
    w, ids = _gpu_route(d["router_logits"], a)
    ties = check_route(d["router_logits"].cpu().numpy(), w, ids, a)
    assert ties <= max(4, spec.M // 1000)


@pytest.mark.parametrize("name", sorted(wl.SMALL_SPECS))
def test_route_small_workloads(name):
    spec = wl.SMALL_SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    a = route_args(spec)
    w, ids = _gpu_route(d["router_logits"], a)
    check_route(d["router_logits"].cpu().numpy(), w, ids, a)


def test_route_golden_cases(golden_dir):
    with open(os.path.join(golden_dir, "route_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        logits = torch.tensor([[math.log(q) for q in c["logits_ln"]]], dtype=torch.float32,
                              device="cuda")
        a = dict(top_k=c["top_k"], method=c["method"], renormalize=c["renormalize"],
                 k_group=c["k_group"], group_count=c["group_count"],
                 group_select_mode=c["group_select_mode"], routed_scaling_factor=c["scale"])
        w, ids = _gpu_route(logits, a)
        assert ids[0].tolist() == c["ids"], c["name"]
        np.testing.assert_allclose(w[0], c["weights"], atol=1e-6, err_msg=c["name"])


CASES = [
    # (E, top_k, method, renorm, k_group, group_count, mode, scale)
    (1, 1, "softmax", True, 1, 1, 0, 1.0),
    (3, 2, "softmax", False, 1, 1, 0, 1.0),
    (33, 5, "sigmoid", False, 1, 1, 0, 0.5),
    (64, 64, "softmax", True, 1, 1, 0, 1.0),
    (96, 6, "softmax", True, 2, 3, 0, 1.0),
    (160, 7, "sigmoid", False, 3, 5, 1, 2.5),
    (256, 8, "softmax", False, 4, 8, 1, 1.0),
    (512, 16, "sigmoid", True, 2, 64, 1, 1.0),
    (1024, 33, "softmax", True, 1, 1, 0, 1.0),
    (1024, 8, "sigmoid", False, 5, 16, 0, 3.0),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("ties", [False, True])
def test_route_shapes_and_ties(case, ties):
    E, k, method, renorm, kg, G, mode, scale = case
    g = torch.Generator().manual_seed(E * 31 + k)
    M = 257
    if ties:
        # few distinct values -> many exactly equal logits (tie rule)
        logits = torch.randint(-3, 4, (M, E), generator=g).float()
    else:
        logits = torch.randn(M, E, generator=g) * 2.0
    a = dict(top_k=k, method=method, renormalize=renorm, k_group=kg, group_count=G,
             group_select_mode=mode, routed_scaling_factor=scale)
    w, ids = _gpu_route(logits.cuda(), a)
    check_route(logits.numpy(), w, ids, a)


def test_route_signed_zero_ties():
    """-0.0 and +0.0 are equal logits: the lower expert id wins."""
    logits = torch.tensor([[0.0, -0.0, -1.0, 0.0, -0.0, 0.5, -0.0, 0.0]]).repeat(3, 1)
    logits[1] = torch.tensor([-0.0, 0.0, -0.0, -2.0, 0.0, -0.0, 0.0, -0.0])
    a = dict(top_k=4, method="softmax", renormalize=True, k_group=1, group_count=1,
             group_select_mode=0, routed_scaling_factor=1.0)
    w, ids = _gpu_route(logits.cuda(), a)
    check_route(logits.numpy(), w, ids, a)
    assert ids[0].tolist() == [5, 0, 1, 3]


def test_route_large_logits_and_empty():
    # sigmoid saturates in fp32 for large logits; selection is still exact
    logits = torch.tensor([[30.0, 40.0, 35.0, -50.0, 39.0, 41.0, 0.0, 20.0]]).repeat(9, 1)
    a = dict(top_k=3, method="sigmoid", renormalize=False, k_group=1, group_count=1,
             group_select_mode=0, routed_scaling_factor=1.0)
    w, ids = _gpu_route(logits.cuda(), a)
    assert (ids == np.array([5, 1, 4])).all()
    check_route(logits.numpy(), w, ids, a)
    # M = 0 is a no-op
    pkg.moe_route(torch.empty(0, 8, device="cuda"), 2)
