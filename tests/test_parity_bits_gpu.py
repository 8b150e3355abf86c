"""GPU parity of the bit-form tree mask (tree_mask_pack_bits,
mla_tree_verify_bits) through the C ABI: the words bit for bit against the
fp64 oracle, attention within the verify tolerances, and the same outputs as
the byte-mask call bit for bit."""
import numpy as np
import pytest
import torch

import __graft_entry__
import oracle
from speculative_decode_mla_tree_gb300 import abi, workloads as W
from speculative_decode_mla_tree_gb300.step import VerifyStep

from parity import OracleRun, compare_attention, sample_rows

pytestmark = pytest.mark.gpu
PATHS = [pytest.param(abi.PATH_SIMT, id="simt"), pytest.param(abi.PATH_TC, id="tcgen05")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    __graft_entry__.build()


def _edge_workload():
    parents = [[-1], list(range(-1, 63)), [-1] + [0] * 15, [-1, -1, 0, 2, 1, -1, 5, 3, 3, -1],
               [-1, 0, 1]]
    return W.make_workload("edges", 8, [7, 100, 33, 500, 0], None, None, 8192, seed=77,
                           parents=parents)


def _check_words(st, ref_kv_indptr):
    w = st.w
    bi, words = oracle.tree_mask_pack_bits(w.parents, w.qo_indptr, ref_kv_indptr)
    assert int(st.status.item()) == 0
    assert (st.mask_word_indptr.cpu().numpy() == bi).all()
    assert (st.mask_words.cpu().numpy().view(np.uint32) == words).all()


@pytest.mark.parametrize("cid", ["small", "edges", 2, 4, 5])
def test_mask_words_bit_exact(cid):
    w = {"small": lambda: W.small(seed=1), "edges": _edge_workload}.get(cid, lambda: W.config(cid))()
    st = VerifyStep(w, path=abi.PATH_TC, mask_bits=True)
    st.load(w)
    abi.mla_tree_kv_indices_build(st.prefix_indices, st.prefix_indptr, st.out_cache_loc, st.qo_indptr,
                                  st.kv_indices, st.kv_indptr, st.status)
    st.pack_mask(); torch.cuda.synchronize()
    _, kv_indptr = oracle.kv_indices_build(w.prefix_indices, w.prefix_indptr, w.out_cache_loc, w.qo_indptr)
    _check_words(st, kv_indptr)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("wl", ["small", "edges", "c2"])
def test_bits_attention_full(wl, path):
    w = {"small": lambda: W.small(seed=1), "edges": _edge_workload, "c2": lambda: W.config(2)}[wl]()
    st = VerifyStep(w, path=path, mask_bits=True); st.run(); torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    ref = OracleRun(w)
    out, lse = ref.attention()
    compare_attention(st.out, st.lse, out, lse)


@pytest.mark.parametrize("path", PATHS)
def test_bits_equal_bytes(path):
    """Same kernel, same inputs, mask in either form: identical outputs."""
    w = W.config(2)
    a = VerifyStep(w, path=path); a.run()
    b = VerifyStep(w, path=path, mask_bits=True, pool=a.pool); b.run()
    torch.cuda.synchronize()
    assert torch.equal(a.out, b.out)
    assert torch.equal(a.lse, b.lse)


@pytest.mark.parametrize("splits", [1, 7, 64])
def test_bits_forced_splits_tc(splits):
    w = W.make_workload("splits", 16, [3000, 20000], "uniform", [32, 8], 65536, seed=5)
    st = VerifyStep(w, path=abi.PATH_TC, max_splits=splits, mask_bits=True); st.run()
    torch.cuda.synchronize()
    ref = OracleRun(w)
    rows = sample_rows(w, 12, seed=2)
    out, lse = ref.attention(rows=rows)
    compare_attention(st.out, st.lse, out, lse, rows=rows)


@pytest.mark.parametrize("cid", [3, 4, 5])
def test_bits_config_sampled_tc(cid):
    w = W.config(cid)
    st = VerifyStep(w, path=abi.PATH_TC, mask_bits=True); st.run(); torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    ref = OracleRun(w)
    rows = sample_rows(w, 6, seed=cid)
    out, lse = ref.attention(rows=rows)
    compare_attention(st.out, st.lse, out, lse, rows=rows)


@pytest.mark.parametrize("n", [8192, 8193], ids=["at_limit", "over_limit"])
def test_mask_tree_size_limit(n):
    """A request of exactly MT_MAX_TREE = 8192 draft nodes packs bit for bit
    (bytes and words); one node more is flagged MT_DEV_TREE_TOO_BIG and its
    rows are left unwritten; the other request is still packed."""
    sizes = [n, 5]
    rng = np.random.default_rng(n)
    parents = []
    for k in sizes:
        par = [-1] + [int(rng.integers(-1, i)) for i in range(1, k)]
        parents.append(par)
    w = W.make_workload("limit", 1, [16, 40], None, None, 16384, seed=3, parents=parents)
    kv_indices, kv_indptr = oracle.kv_indices_build(w.prefix_indices, w.prefix_indptr,
                                                    w.out_cache_loc, w.qo_indptr)
    dev = torch.device("cuda")
    par = w.parents.to(dev)
    qptr = w.qo_indptr.to(dev)
    kptr = torch.from_numpy(np.asarray(kv_indptr, dtype=np.int32)).to(dev)
    B = w.batch
    mi_ref, m_ref = oracle.tree_mask_pack(w.parents, w.qo_indptr, kv_indptr)
    wi_ref, w_ref = oracle.tree_mask_pack_bits(w.parents, w.qo_indptr, kv_indptr)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    mask = torch.full((int(mi_ref[-1]),), 7, dtype=torch.uint8, device=dev)
    mind = torch.empty(B + 1, dtype=torch.int64, device=dev)
    abi.tree_mask_pack(par, qptr, kptr, mind, mask, status)
    words = torch.full((int(wi_ref[-1]),), 7, dtype=torch.int32, device=dev)
    wind = torch.empty(B + 1, dtype=torch.int64, device=dev)
    abi.tree_mask_pack_bits(par, qptr, kptr, wind, words, status)
    torch.cuda.synchronize()
    assert (mind.cpu().numpy() == mi_ref).all() and (wind.cpu().numpy() == wi_ref).all()
    m, wd = mask.cpu().numpy(), words.cpu().numpy().view(np.uint32)
    if n <= 8192:
        assert int(status.item()) == 0
        assert (m == m_ref).all() and (wd == w_ref).all()
    else:
        assert int(status.item()) == abi.DEV_TREE_TOO_BIG
        # request 0 untouched, request 1 packed
        assert (m[:mi_ref[1]] == 7).all() and (m[mi_ref[1]:] == m_ref[mi_ref[1]:]).all()
        assert (wd[:wi_ref[1]] == 7).all() and (wd[wi_ref[1]:] == w_ref[wi_ref[1]:]).all()


def test_short_work_two_rounds_of_items():
    """90 requests of one 128-row tile and 56-106 keys: the short-work
    kernel variant (dry passes on a cluster's first item), with more items
    than clusters, so clusters also run a second item without the dry pass."""
    rng = np.random.default_rng(9)
    prefix = [int(x) for x in rng.integers(40, 91, size=90)]
    w = W.make_workload("rounds", 8, prefix, "uniform", [16] * 90, 65536, seed=9)
    # the host's choice of the short-work variant: every tile against the
    # whole kv_indices stays within 512 key blocks per cluster
    tiles_ub = (w.total_q * w.heads + 127) // 128 + w.batch
    assert tiles_ub * (sum(prefix) + w.total_q) <= 512 * 48 * 76
    st = VerifyStep(w, path=abi.PATH_TC, fused=True)
    st.run()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    out, lse = OracleRun(w).attention()
    compare_attention(st.out, st.lse, out, lse)


def test_bits_graph_capture_and_replay():
    w1 = W.make_workload("g", 8, [300, 1200, 77], "uniform", [16, 9, 30], 16384, seed=101)
    w2 = W.make_workload("g", 8, [300, 1200, 77], "uniform", [16, 9, 30], 16384, seed=202)
    st = VerifyStep(w1, path=abi.PATH_TC, mask_bits=True)
    st.run(); torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        st.run()
    for w in (w1, w2):
        st.pool.copy_(w.dense_pool("cuda"))
        st.load(w)
        g.replay(); torch.cuda.synchronize()
        ref = OracleRun(w)
        out, lse = ref.attention()
        compare_attention(st.out, st.lse, out, lse)


def test_bits_capacity_overflow_is_flagged():
    w = W.small(seed=10)
    st = VerifyStep(w, mask_bits=True)
    st.mask_words = st.mask_words[: st.mask_words.numel() // 2]
    st.run(); torch.cuda.synchronize()
    assert int(st.status.item()) & abi.DEV_BAD_INDPTR


@pytest.mark.parametrize("wl", ["small", "edges", "c2", "c4"])
def test_prepare_matches_separate_calls(wl):
    """mla_tree_prepare writes exactly what the three separate entry points
    write (pool rows, kv_indices, kv_indptr, mask words and offsets), and
    those match the oracle."""
    w = {"small": lambda: W.small(seed=1), "edges": _edge_workload, "c2": lambda: W.config(2),
         "c4": lambda: W.config(4)}[wl]()
    a = VerifyStep(w, path=abi.PATH_TC, mask_bits=True)
    a.load(w)
    abi.mla_tree_draft_kv_scatter(a.draft_kv, a.out_cache_loc, a.pool, a.status)
    abi.mla_tree_kv_indices_build(a.prefix_indices, a.prefix_indptr, a.out_cache_loc, a.qo_indptr,
                                  a.kv_indices, a.kv_indptr, a.status)
    a.pack_mask()
    b = VerifyStep(w, path=abi.PATH_TC, fused=True)
    b.load(w)
    b.prepare()
    torch.cuda.synchronize()
    assert int(a.status.item()) == 0 and int(b.status.item()) == 0
    for x, y in [(a.pool, b.pool), (a.kv_indices, b.kv_indices), (a.kv_indptr, b.kv_indptr),
                 (a.mask_word_indptr, b.mask_word_indptr), (a.mask_words, b.mask_words)]:
        assert torch.equal(x, y)
    kv_indices, kv_indptr = oracle.kv_indices_build(w.prefix_indices, w.prefix_indptr, w.out_cache_loc,
                                                    w.qo_indptr)
    assert (b.kv_indices.cpu().numpy() == kv_indices).all()
    _check_words(b, kv_indptr)


@pytest.mark.parametrize("path", PATHS)
def test_fused_step_attention(path):
    w = W.config(2)
    st = VerifyStep(w, path=path, fused=True); st.run(); torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    ref = OracleRun(w)
    out, lse = ref.attention()
    compare_attention(st.out, st.lse, out, lse)


def test_prepare_flags_bad_slot_and_parent():
    w = W.small(seed=12)
    st = VerifyStep(w, fused=True)
    st.load(w)
    st.out_cache_loc[1] = w.num_slots + 3
    st.parents[2] = 7
    st.prepare(); torch.cuda.synchronize()
    s = int(st.status.item())
    assert s & abi.DEV_BAD_SLOT and s & abi.DEV_BAD_PARENT


@pytest.mark.parametrize("bits", [False, True], ids=["bytes", "bits"])
@pytest.mark.parametrize("layout", ["contiguous", "paged64"])
def test_kv_layouts_tc(layout, bits):
    """Pools whose slots come in runs: one contiguous run, or 64-slot pages."""
    w = W.config(2, layout)
    st = VerifyStep(w, path=abi.PATH_TC, mask_bits=bits); st.run(); torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    ref = OracleRun(w)
    out, lse = ref.attention()
    compare_attention(st.out, st.lse, out, lse)


def test_contiguous_run_to_pool_end():
    """A run ending at the last pool slot (the pool holds exactly the batch's
    rows): the last block's rows past the split end read as zeros."""
    w = W.make_workload("end", 8, [500, 300], "uniform", [16, 16], 832, seed=31, kv_layout="contiguous")
    assert int(w.pool_slots.max()) == 831
    for path in (abi.PATH_TC, abi.PATH_SIMT):
        st = VerifyStep(w, path=path, fused=True); st.run(); torch.cuda.synchronize()
        assert int(st.status.item()) == 0
        ref = OracleRun(w)
        out, lse = ref.attention()
        compare_attention(st.out, st.lse, out, lse)


def test_kv_layout_paged_long_prefix_sampled():
    w = W.config(4, "paged64")
    st = VerifyStep(w, path=abi.PATH_TC, fused=True); st.run(); torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    ref = OracleRun(w)
    rows = sample_rows(w, 8, seed=44)
    out, lse = ref.attention(rows=rows)
    compare_attention(st.out, st.lse, out, lse, rows=rows)
