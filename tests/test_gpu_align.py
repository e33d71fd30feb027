"""GPU parity of moe_align against the oracle: sorted_token_ids, offsets,
counts, per-block expert ids and the padding sentinel, bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import mixture_experts_ffn_softmax_gb300 as pkg
from mixture_experts_ffn_softmax_gb300 import workloads as wl

from helpers import route_args

pytestmark = pytest.mark.gpu


def _check_align(ids_np, E, bm):
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = pkg.moe_align(ids, E, bm, error_word=err)
    torch.cuda.synchronize()
    ref = oracle.align(ids_np, E, bm)
    n = ref["num_tokens_post_padded"]
    off = g["expert_offsets"].cpu().numpy()
    assert off.tolist() == ref["expert_offsets"].tolist()
    assert g["expert_num_tokens"].cpu().numpy().tolist() == ref["expert_num_tokens"].tolist()
    assert g["sorted_token_ids"][:n].cpu().numpy().tolist() == ref["sorted_token_ids"].tolist()
    blk = g["block_expert_ids"].cpu().numpy()
    assert blk[: n // bm].tolist() == ref["block_expert_ids"].tolist()
    assert (blk[n // bm:] == -1).all()
    assert int(err.item()) == 0


@pytest.mark.parametrize("name", sorted(wl.SPECS))
def test_align_full_size_routing(name):
    spec = wl.SPECS[name]
    d = wl.make_moe_inputs(spec, device="cuda", weights=False)
    a = route_args(spec)
    _, ids = pkg.moe_route(d["router_logits"], a["top_k"], a["method"], a["renormalize"],
                           a["k_group"], a["group_count"], a["group_select_mode"],
                           a["routed_scaling_factor"])
    _check_align(ids.cpu().numpy(), spec.E, pkg.BLOCK_M)


@pytest.mark.parametrize("bm", [1, 7, 16, 128, 1024])
@pytest.mark.parametrize("E,M,k", [(1, 5, 1), (8, 1, 2), (8, 777, 2), (37, 300, 4),
                                   (256, 513, 8), (1024, 300, 3)])
def test_align_shapes(E, M, k, bm):
    rng = np.random.default_rng(E * 7 + M)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]) if k <= E else None
    _check_align(ids, E, bm)


def test_align_skewed_and_empty_experts():
    rng = np.random.default_rng(1)
    E, M, k = 64, 3000, 4
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)])
    ids[:2500] = [3, 9, 10, 11]          # most items on four experts, many experts empty
    ids[:, 0][ids[:, 0] > 40] = 3
    _check_align(ids, E, 128)
    # every item on one expert (duplicates allowed in ids)
    _check_align(np.full((1000, 2), 5, dtype=np.int32), 8, 128)


def test_align_bad_ids_set_error_word():
    ids = torch.tensor([[0, 1], [2, 9], [-1, 3]], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = pkg.moe_align(ids, 4, 4, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 4                       # MOE_ERR_BAD_EXPERT_ID
    counts = g["expert_num_tokens"].cpu().numpy().tolist()
    assert counts == [1, 1, 1, 1]                     # bad items dropped, others placed
    assert pkg.read_error(err.data_ptr()) == 4
    assert int(err.item()) == 0                       # reset by read_error


@pytest.mark.parametrize("E,M,k", [(8, 2049, 2), (8, 8192, 2), (16, 4096, 4), (8, 8193, 2),
                                   (17, 1500, 3), (2, 16384, 1)])
def test_align_one_block_plan_bounds(E, M, k):
    """Around the bounds of the one-block plan for few experts (items up to
    16384 with at most 16 experts) and just past them; a skewed draw."""
    rng = np.random.default_rng(M + E)
    p = rng.dirichlet(np.ones(E) * 0.3)
    ids = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(M)]).astype(np.int32)
    _check_align(ids, E, 128)
    _check_align(ids, E, 16)
