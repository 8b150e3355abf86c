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


def test_redraw_keeps_shapes_and_changes_contents():
    w = W.config(2)
    v = W.redraw(w, 2002)
    assert v.prefix_lens == w.prefix_lens and v.tree_sizes == w.tree_sizes
    assert v.heads == w.heads and v.num_slots == w.num_slots and v.sm_scale == w.sm_scale
    assert torch.equal(v.qo_indptr, w.qo_indptr) and torch.equal(v.prefix_indptr, w.prefix_indptr)
    assert v.q.shape == w.q.shape and v.pool_rows.shape == w.pool_rows.shape
    assert not torch.equal(v.q.view(torch.int16), w.q.view(torch.int16))
    qo = v.qo_indptr.tolist()
    for b in range(v.batch):          # the same tree rule (branching <= 3, node 0 the root)
        ch, _ = _children_depth(v.parents[qo[b]:qo[b + 1]].tolist())
        assert max(ch) <= 3


def _f64(t):
    return t.double()


def test_stress_cancel_zeroes_the_latent_dot_product_exactly():
    w = W.small(seed=3)
    s = W.stress(w, "cancel")
    q, k = _f64(s.q), _f64(s.pool_rows)
    lat = torch.einsum("thd,rd->thr", q[..., :512], k[:, :512])
    assert float(lat.abs().max()) == 0.0
    half = torch.einsum("thd,rd->thr", q[..., :256], k[:, :256])
    assert float(half.abs().max()) > 1000.0     # each half alone is large


def test_stress_huge_v_keeps_scores_and_scales_values():
    w = W.small(seed=4)
    s = W.stress(w, "huge_v")
    sw = torch.einsum("thd,rd->thr", _f64(w.q), _f64(w.pool_rows))
    ss = torch.einsum("thd,rd->thr", _f64(s.q), _f64(s.pool_rows))
    assert torch.equal(sw, ss)                   # power-of-two factors: exact
    assert float(_f64(s.pool_rows)[:, :512].abs().max()) > 65504.0
    assert torch.equal(_f64(s.pool_rows)[:, :512], _f64(w.pool_rows)[:, :512] * 2.0 ** 17)


def test_stress_peaked_scales_queries_by_eight():
    w = W.small(seed=5)
    s = W.stress(w, "peaked")
    assert torch.equal(_f64(s.q), _f64(w.q) * 8.0)
    assert torch.equal(s.pool_rows.view(torch.int16), w.pool_rows.view(torch.int16))
