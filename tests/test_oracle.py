"""Pins for the fp64 oracle: each test ties it to something other than itself
(a hand-worked example, the shapes the pages log, a library routine, brute
force, a closed form or an invariant). CPU only."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decode_mla_tree_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _bf16(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def _prepare(w):
    """Scatter + index build + mask for a workload, all through the oracle."""
    pool = oracle.draft_kv_scatter(_bits(w.dense_pool()), _bits(w.draft_kv), w.out_cache_loc)
    kv_indices, kv_indptr = oracle.kv_indices_build(w.prefix_indices, w.prefix_indptr,
                                                    w.out_cache_loc, w.qo_indptr)
    mask_indptr, mask = oracle.tree_mask_pack(w.parents, w.qo_indptr, kv_indptr)
    return pool, kv_indices, kv_indptr, mask_indptr, mask


def _attend(w, pool, kv_indices, kv_indptr, mask_indptr, mask, q=None, **kw):
    return oracle.verify_attention(_bits(w.q) if q is None else q, pool, kv_indices, kv_indptr,
                                   w.qo_indptr, mask, mask_indptr, w.heads, w.sm_scale, **kw)


# ------------------------------------------------------------------ golden

def test_page_shapes_log():
    """Config 1 reproduces the logged live shapes: q (9, 8, 576), prefix 21,
    mask of 270 = 9 x 30 elements."""
    g = json.load(open(os.path.join(GOLDEN, "verify_shapes_log.json")))
    w = W.config(1)
    assert list(w.q.shape) == g["q_shape"]
    assert w.prefix_lens == [g["kv_len_max"]]
    assert w.tree_sizes == [g["draft_tokens"]]
    _, kv_indices, kv_indptr, mask_indptr, mask = _prepare(w)
    assert int(mask_indptr[-1]) == g["mask_numel"] == mask.size
    assert int(kv_indptr[1] - kv_indptr[0]) == g["mask_row_stride"]


def test_small_tree_mask_by_hand():
    g = json.load(open(os.path.join(GOLDEN, "small_tree_mask.json")))
    parents, qo, pidx, pptr, loc = [], [0], [], [0], []
    for r, ps, ds in zip(g["requests"], g["prefix_slots"], g["draft_slots"]):
        parents += r["parents"]
        qo.append(qo[-1] + len(r["parents"]))
        pidx += ps
        pptr.append(pptr[-1] + len(ps))
        loc += ds
    kv_indices, kv_indptr = oracle.kv_indices_build(np.array(pidx), np.array(pptr),
                                                    np.array(loc), np.array(qo))
    assert kv_indices.tolist() == g["kv_indices"]
    assert kv_indptr.tolist() == g["kv_indptr"]
    mask_indptr, mask = oracle.tree_mask_pack(np.array(parents), np.array(qo), kv_indptr)
    assert mask_indptr.tolist() == g["mask_indptr"]
    expect = np.concatenate([np.array(r["mask"], dtype=np.uint8).reshape(-1) for r in g["requests"]])
    assert mask.tolist() == expect.tolist()


# ------------------------------------------------------------------ mask

def _all_forests(n):
    return itertools.product(*[range(-1, i) for i in range(n)])


def test_ancestors_match_networkx_exhaustive():
    """Every parent array with n <= 6 (873 forests): ancestor-or-self sets
    equal networkx's graph ancestors plus the node itself."""
    nx = pytest.importorskip("networkx")
    count = 0
    for n in range(1, 7):
        for par in _all_forests(n):
            G = nx.DiGraph()
            G.add_nodes_from(range(n))
            G.add_edges_from((p, i) for i, p in enumerate(par) if p >= 0)
            got = oracle.ancestors_or_self(par)
            for i in range(n):
                assert got[i] == nx.ancestors(G, i) | {i}
            count += 1
    assert count == sum(math.factorial(n) for n in range(1, 7))


def test_mask_chain_is_causal_and_star_is_diagonal():
    n, P = 12, 5
    qo = np.array([0, n]); kv_indptr = np.array([0, P + n])
    _, chain = oracle.tree_mask_pack(np.arange(-1, n - 1), qo, kv_indptr)
    chain = chain.reshape(n, P + n)
    causal = np.concatenate([np.ones((n, P), np.uint8), np.tril(np.ones((n, n), np.uint8))], 1)
    assert (chain == causal).all()
    _, star = oracle.tree_mask_pack(np.full(n, -1), qo, kv_indptr)
    star = star.reshape(n, P + n)
    diag = np.concatenate([np.ones((n, P), np.uint8), np.eye(n, dtype=np.uint8)], 1)
    assert (star == diag).all()


def test_small_tree_mask_bits_by_hand():
    """The bit encoding of the hand-worked masks (words also worked by hand)."""
    g = json.load(open(os.path.join(GOLDEN, "small_tree_mask.json")))
    parents, qo, kv = [], [0], [0]
    for r in g["requests"]:
        parents += r["parents"]
        qo.append(qo[-1] + len(r["parents"]))
        kv.append(kv[-1] + r["prefix"] + len(r["parents"]))
    indptr, words = oracle.tree_mask_pack_bits(np.array(parents), np.array(qo), np.array(kv))
    assert indptr.tolist() == g["mask_word_indptr"]
    assert words.dtype == np.uint32
    assert words.tolist() == g["mask_words"]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_mask_bits_unpack_to_mask_bytes(seed):
    """Rows of several words (prefixes 0..130, trees up to 40 nodes): unpacking
    each row's words with numpy's bit order gives the byte mask, and the bits
    past the row's last column are zero."""
    rng = np.random.default_rng(seed)
    batch = 5
    n = rng.integers(1, 41, batch)
    P = rng.integers(0, 131, batch)
    parents = np.concatenate([[int(rng.integers(-1, i)) for i in range(k)] for k in n])
    qo = np.concatenate([[0], np.cumsum(n)])
    kv = np.concatenate([[0], np.cumsum(n + P)])
    bi, words = oracle.tree_mask_pack_bits(parents, qo, kv)
    mi, mask = oracle.tree_mask_pack(parents, qo, kv)
    for b in range(batch):
        L, W = int(n[b] + P[b]), int((n[b] + P[b] + 31) // 32)
        rows = words[bi[b]:bi[b + 1]].reshape(int(n[b]), W)
        bits = np.unpackbits(rows.astype("<u4").view(np.uint8), bitorder="little").reshape(int(n[b]), 32 * W)
        assert (bits[:, :L] == mask[mi[b]:mi[b + 1]].reshape(int(n[b]), L)).all()
        assert not bits[:, L:].any()


def test_mask_rejects_non_topological_parent():
    with pytest.raises(ValueError):
        oracle.ancestors_or_self([-1, 2, 0])


# ------------------------------------------------------------------ marshaling

def test_kv_indices_config1_is_the_drawn_permutation():
    """Config 1 drew kv_indices as 30 distinct slots with out_cache_loc = the
    last 9: the oracle's marshaling must give back exactly that list."""
    w = W.config(1)
    kv_indices, kv_indptr = oracle.kv_indices_build(w.prefix_indices, w.prefix_indptr,
                                                    w.out_cache_loc, w.qo_indptr)
    assert kv_indptr.tolist() == [0, 30]
    assert kv_indices.tolist() == w.pool_slots[:30].tolist()
    assert kv_indices[21:].tolist() == w.out_cache_loc.tolist()
    assert len(set(kv_indices.tolist())) == 30


def test_scatter_writes_rows_and_nothing_else():
    w = W.small(seed=3)
    pool0 = _bits(w.dense_pool())
    pool1 = oracle.draft_kv_scatter(pool0, _bits(w.draft_kv), w.out_cache_loc)
    loc = w.out_cache_loc.numpy()
    assert (pool1[loc] == _bits(w.draft_kv)).all()
    other = np.ones(w.num_slots, bool); other[loc] = False
    assert (pool1[other] == pool0[other]).all()


# ------------------------------------------------------------------ attention

def test_bf16_widening_exact():
    x = torch.randn(1000, generator=torch.Generator().manual_seed(0)).to(torch.bfloat16)
    assert (oracle.bf16_bits_to_f64(_bits(x)) == x.to(torch.float64).numpy()).all()


def test_dense_matches_torch_softmax():
    """All-visible rows reduce to softmax(scale * q k^T) v, checked against
    torch.softmax / torch.logsumexp in float64."""
    w = W.small(seed=5, batch=1, prefix=(50,), tree=(6,), rule="uniform")
    pool, kv_indices, kv_indptr, mask_indptr, mask = _prepare(w)
    mask = np.ones_like(mask)
    out, lse = _attend(w, pool, kv_indices, kv_indptr, mask_indptr, mask)
    K = torch.from_numpy(oracle.bf16_bits_to_f64(pool[kv_indices.astype(np.int64)]))
    Q = w.q.to(torch.float64)
    scale = float(np.float32(w.sm_scale))
    S = scale * torch.einsum("thd,ld->thl", Q, K)
    ref = torch.softmax(S, dim=-1) @ K[:, :512]
    assert np.abs(out - ref.numpy()).max() < 1e-12
    assert np.abs(lse - torch.logsumexp(S, -1).numpy()).max() < 1e-12


def _plain_decode(qv, keys, scale):
    """Ordinary single-query attention written with Python loops."""
    s = [scale * sum(a * b for a, b in zip(qv, k)) for k in keys]
    m = max(s)
    e = [math.exp(x - m) for x in s]
    tot = sum(e)
    out = [sum(e[j] * keys[j][d] for j in range(len(keys))) / tot for d in range(512)]
    return out, m + math.log(tot)


def test_chain_is_causal_decode():
    """A chain tree: draft row i is ordinary decode over prefix + drafts 0..i."""
    P, n, H = 7, 5, 2
    w = W.make_workload("chain", H, [P], "chain", [n], 64, seed=11)
    pool, kv_indices, kv_indptr, mask_indptr, mask = _prepare(w)
    out, lse = _attend(w, pool, kv_indices, kv_indptr, mask_indptr, mask)
    Kf = oracle.bf16_bits_to_f64(pool[kv_indices.astype(np.int64)]).tolist()
    Qf = w.q.to(torch.float64).numpy()
    scale = float(np.float32(w.sm_scale))
    for i in range(n):
        for h in range(H):
            o, l = _plain_decode(Qf[i, h].tolist(), Kf[:P + i + 1], scale)
            assert abs(l - lse[i, h]) < 1e-11
            assert np.abs(np.array(o) - out[i, h]).max() < 1e-11


def test_skip_prefix_reads_no_prefix_mask():
    """The prefix-skip switch: the first L_b - n_b positions are visible
    whatever their mask bytes hold, the draft positions still follow the tree."""
    w = W.make_workload("skip", 2, [6, 9], "uniform", [5, 7], 128, seed=21)
    pool, kv_indices, kv_indptr, mask_indptr, mask = _prepare(w)
    out, lse = _attend(w, pool, kv_indices, kv_indptr, mask_indptr, mask)
    # a tree mask already shows the whole prefix: the switch changes nothing
    o2, l2 = _attend(w, pool, kv_indices, kv_indptr, mask_indptr, mask, skip_prefix=True)
    assert np.array_equal(o2, out) and np.array_equal(l2, lse)
    # clear every prefix byte
    cleared = mask.copy()
    qptr = w.qo_indptr.numpy()
    for b in range(len(qptr) - 1):
        n, L = int(qptr[b + 1] - qptr[b]), int(kv_indptr[b + 1] - kv_indptr[b])
        for i in range(n):
            cleared[mask_indptr[b] + i * L:mask_indptr[b] + i * L + L - n] = 0
    o3, l3 = _attend(w, pool, kv_indices, kv_indptr, mask_indptr, cleared, skip_prefix=True)
    assert np.array_equal(o3, out) and np.array_equal(l3, lse)
    # without the switch the cleared prefix is gone: a root (parent -1) sees
    # only itself, so its row is that key's value row and its own score
    o4, l4 = _attend(w, pool, kv_indices, kv_indptr, mask_indptr, cleared)
    scale = float(np.float32(w.sm_scale))
    for b in range(len(qptr) - 1):
        n, L = int(qptr[b + 1] - qptr[b]), int(kv_indptr[b + 1] - kv_indptr[b])
        for i in range(n):
            if int(w.parents[qptr[b] + i]) != -1:
                continue
            t = int(qptr[b]) + i
            k = oracle.bf16_bits_to_f64(pool[int(kv_indices[kv_indptr[b] + L - n + i])])
            for h in range(w.heads):
                qf = oracle.bf16_bits_to_f64(_bits(w.q)[t, h])
                assert abs(l4[t, h] - scale * float(qf @ k)) < 1e-9
                assert np.abs(o4[t, h] - k[:512]).max() < 1e-12
    assert not np.allclose(o4, out)


def test_constant_scores_give_uniform_mean():
    """Zero latent query dims and one shared rope key make every score equal:
    out is the plain mean of the visible V rows, lse = s + ln(#visible)."""
    w = W.small(seed=7)
    pool, kv_indices, kv_indptr, mask_indptr, mask = _prepare(w)
    pool = pool.copy()
    rope = _bits(_bf16(np.linspace(-1, 1, 64)))
    pool[:, 512:] = rope
    q = _bits(w.q).copy()
    q[:, :, :512] = 0
    out, lse = _attend(w, pool, kv_indices, kv_indptr, mask_indptr, mask, q=q)
    qf = oracle.bf16_bits_to_f64(q)
    rf = oracle.bf16_bits_to_f64(rope)
    scale = np.float64(np.float32(w.sm_scale))
    qo = w.qo_indptr.numpy()
    for b in range(w.batch):
        L = kv_indptr[b + 1] - kv_indptr[b]
        n = qo[b + 1] - qo[b]
        V = oracle.bf16_bits_to_f64(pool[kv_indices[kv_indptr[b]:kv_indptr[b + 1]].astype(np.int64), :512])
        vis = mask[mask_indptr[b]:mask_indptr[b + 1]].reshape(n, L) != 0
        for i in range(n):
            t = qo[b] + i
            mean = V[vis[i]].mean(axis=0)
            for h in range(w.heads):
                s = scale * float(qf[t, h, 512:] @ rf)
                assert abs(lse[t, h] - (s + math.log(vis[i].sum()))) < 1e-12
                assert np.abs(out[t, h] - mean).max() < 1e-12


def test_single_visible_key():
    w = W.small(seed=9)
    pool, kv_indices, kv_indptr, mask_indptr, mask = _prepare(w)
    rng = np.random.default_rng(0)
    mask = np.zeros_like(mask)
    qo = w.qo_indptr.numpy()
    pick = {}
    for b in range(w.batch):
        L = kv_indptr[b + 1] - kv_indptr[b]
        for i in range(qo[b + 1] - qo[b]):
            j = int(rng.integers(0, L))
            mask[mask_indptr[b] + i * L + j] = 1
            pick[qo[b] + i] = kv_indices[kv_indptr[b] + j]
    out, lse = _attend(w, pool, kv_indices, kv_indptr, mask_indptr, mask)
    qf = oracle.bf16_bits_to_f64(_bits(w.q))
    scale = np.float64(np.float32(w.sm_scale))
    for t, slot in pick.items():
        row = oracle.bf16_bits_to_f64(pool[slot])
        assert (out[t] == row[None, :512]).all()
        assert np.abs(lse[t] - scale * (qf[t] @ row)).max() < 1e-12


def test_empty_row_gives_zero_and_minus_inf():
    w = W.small(seed=13)
    pool, kv_indices, kv_indptr, mask_indptr, mask = _prepare(w)
    mask = mask.copy()
    L0 = kv_indptr[1] - kv_indptr[0]
    mask[mask_indptr[0]:mask_indptr[0] + L0] = 0    # row 0 of request 0 sees nothing
    out, lse = _attend(w, pool, kv_indices, kv_indptr, mask_indptr, mask)
    assert (out[0] == 0).all() and np.isneginf(lse[0]).all()
    assert np.isfinite(lse[1:]).all()


def test_pool_permutation_invariance():
    """Moving pool rows and remapping slots gives bit-identical results."""
    w = W.small(seed=17)
    pool, kv_indices, kv_indptr, mask_indptr, mask = _prepare(w)
    out, lse = _attend(w, pool, kv_indices, kv_indptr, mask_indptr, mask)
    perm = np.random.default_rng(1).permutation(w.num_slots)
    pool2 = np.empty_like(pool); pool2[perm] = pool
    out2, lse2 = _attend(w, pool2, perm[kv_indices].astype(np.int32), kv_indptr, mask_indptr, mask)
    assert (out == out2).all() and (lse == lse2).all()


def test_duplicated_head_gives_identical_rows():
    w = W.small(seed=19)
    pool, kv_indices, kv_indptr, mask_indptr, mask = _prepare(w)
    q = _bits(w.q).copy()
    q[:, 3] = q[:, 1]
    out, lse = _attend(w, pool, kv_indices, kv_indptr, mask_indptr, mask, q=q)
    assert (out[:, 3] == out[:, 1]).all() and (lse[:, 3] == lse[:, 1]).all()


def test_uniform_score_shift():
    """With every key sharing one rope vector u, moving the query's rope part
    along u adds the same amount to every score: out is unchanged and lse
    moves by exactly that amount."""
    w = W.small(seed=23)
    pool, kv_indices, kv_indptr, mask_indptr, mask = _prepare(w)
    pool = pool.copy()
    u = np.zeros(64, np.float32); u[0] = 1.0
    pool[:, 512:] = _bits(_bf16(u))
    q = _bits(w.q).copy()
    q[:, :, 512:] = _bits(_bf16(np.zeros(64)))
    out0, lse0 = _attend(w, pool, kv_indices, kv_indptr, mask_indptr, mask, q=q)
    q[:, :, 512] = _bits(_bf16([3.0]))[0]
    out1, lse1 = _attend(w, pool, kv_indices, kv_indptr, mask_indptr, mask, q=q)
    scale = np.float64(np.float32(w.sm_scale))
    assert np.abs(lse1 - lse0 - 3.0 * scale).max() < 1e-12
    assert np.abs(out1 - out0).max() < 1e-12


def test_scale_enters_as_float32():
    w = W.small(seed=29, sm_scale=0.1)
    pool, kv_indices, kv_indptr, mask_indptr, mask = _prepare(w)
    a = _attend(w, pool, kv_indices, kv_indptr, mask_indptr, mask)
    w.sm_scale = float(np.float32(0.1))
    b = _attend(w, pool, kv_indices, kv_indptr, mask_indptr, mask)
    assert (a[0] == b[0]).all()


@pytest.mark.parametrize("splits", [1, 3, 7, 64])
def test_split_merge_equals_unsplit(splits):
    """Split partials merged by log-sum-exp equal the unsplit result; 64
    splits leave some pieces empty for the shortest request."""
    w = W.small(seed=31, prefix=(5, 40, 130), tree=(4, 9, 17))
    pool, kv_indices, kv_indptr, mask_indptr, mask = _prepare(w)
    out, lse = _attend(w, pool, kv_indices, kv_indptr, mask_indptr, mask)
    parts = oracle.verify_attention_split(_bits(w.q), pool, kv_indices, kv_indptr, w.qo_indptr,
                                          mask, mask_indptr, w.heads, w.sm_scale, splits)
    out2, lse2 = oracle.lse_merge(parts)
    assert np.abs(out2 - out).max() < 1e-12
    assert np.abs(lse2 - lse).max() < 1e-12


def test_split_bounds_cover():
    for L in [0, 1, 5, 63, 64, 1000]:
        for s in [1, 2, 7, 64]:
            b = oracle.split_bounds(L, s)
            assert b[0][0] == 0 and b[-1][1] == L
            assert all(b[k][1] == b[k + 1][0] for k in range(s - 1))
            lens = [hi - lo for lo, hi in b]
            assert max(lens) - min(lens) <= 1


def test_row_sampling_matches_full():
    w = W.small(seed=37)
    pool, kv_indices, kv_indptr, mask_indptr, mask = _prepare(w)
    out, lse = _attend(w, pool, kv_indices, kv_indptr, mask_indptr, mask)
    rows = [(0, 0), (5, 7), (w.total_q - 1, 3)]
    o2, l2 = _attend(w, pool, kv_indices, kv_indptr, mask_indptr, mask, rows=rows)
    for t, h in rows:
        # BLAS blocks a different row count differently: equal up to rounding
        assert np.abs(o2[t, h] - out[t, h]).max() < 1e-12 and abs(l2[t, h] - lse[t, h]) < 1e-12
