"""The seeded generators follow their recipes (tree rules, distinct slots)."""
import math

import pytest
import torch

from speculative_decode_mla_tree_gb300 import workloads as W


def _children_depth(par):
    ch = [0] * len(par)
    dep = []
    for i, p in enumerate(par):
        assert -1 <= p < i
        dep.append(1 if p < 0 else dep[p] + 1)
        if p >= 0:
            ch[p] += 1
    return ch, dep


@pytest.mark.parametrize("cid", [1, 2, 3])
def test_config_recipes(cid):
    w = W.config(cid)
    qo = w.qo_indptr.tolist()
    for b in range(w.batch):
        par = w.parents[qo[b]:qo[b + 1]].tolist()
        ch, dep = _children_depth(par)
        if cid == 2:
            assert par[0] == -1 and max(ch) <= 3 and len(par) == 16
            assert 1024 <= w.prefix_lens[b] <= 4096
        if cid == 3:
            assert max(ch) <= 4 and max(dep) <= 8 and len(par) == 64
    slots = torch.cat([w.prefix_indices, w.out_cache_loc])
    assert slots.unique().numel() == slots.numel()
    assert int(slots.max()) < w.num_slots
    assert w.q.shape == (w.total_q, w.heads, 576)


def test_config5_shape_only():
    """Config 5 is large: check its drawn sizes without building the pool."""
    g = torch.Generator().manual_seed(1005)
    lo, hi = math.log(128.0), math.log(131072.0)
    P = [int(math.floor(math.exp(lo + (hi - lo) * float(torch.rand((1,), generator=g))))) for _ in range(64)]
    assert all(128 <= p <= 131072 for p in P)


def test_seed_reproducible():
    a, b = W.config(1), W.config(1)
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    assert torch.equal(a.parents, b.parents)
