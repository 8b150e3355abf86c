"""GPU parity through the C ABI against the fp64 oracle.

Marshaling (scatter, kv indices, mask) is compared bit for bit; attention
within the verify tolerances (out max-abs <= 1e-2 and mean-abs <= 1e-3,
lse |err| <= 1e-3 * max(1, |lse|)). Paths are forced so the warp-shuffle
and tensor-core kernels are each checked."""
import numpy as np
import pytest
import torch

import __graft_entry__
from speculative_decode_mla_tree_gb300 import abi, workloads as W
from speculative_decode_mla_tree_gb300.step import VerifyStep

from parity import OracleRun, bits, compare_attention, sample_rows

pytestmark = pytest.mark.gpu
PATHS = [pytest.param(abi.PATH_SIMT, id="simt"), pytest.param(abi.PATH_TC, id="tcgen05")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    __graft_entry__.build()


_cache = {}


def _oracle(key, w):
    if key not in _cache:
        _cache[key] = OracleRun(w)
    return _cache[key]


def _check_marshal(st, ref):
    w = st.w
    assert int(st.status.item()) == 0
    assert (st.kv_indices.cpu().numpy() == ref.kv_indices).all()
    assert (st.kv_indptr.cpu().numpy() == ref.kv_indptr).all()
    assert (st.mask_indptr.cpu().numpy() == ref.mask_indptr).all()
    assert (st.mask.cpu().numpy() == ref.mask).all()
    loc = w.out_cache_loc.numpy()
    assert (bits(st.pool[st.out_cache_loc.long()]) == ref.pool[loc]).all()


def _edge_workload():
    """Single node, pure chain of 64, star, random forest, empty prefix."""
    parents = [[-1], list(range(-1, 63)), [-1] + [0] * 15, [-1, -1, 0, 2, 1, -1, 5, 3, 3, -1],
               [-1, 0, 1]]
    return W.make_workload("edges", 8, [7, 100, 33, 500, 0], None, None, 8192, seed=77,
                           parents=parents)


@pytest.mark.parametrize("path", PATHS)
def test_small_ragged(path):
    w = W.small(seed=1)
    st = VerifyStep(w, path=path); st.run(); torch.cuda.synchronize()
    ref = _oracle("small", w)
    _check_marshal(st, ref)
    out, lse = ref.attention()
    compare_attention(st.out, st.lse, out, lse)


@pytest.mark.parametrize("path", PATHS)
def test_edge_trees(path):
    w = _edge_workload()
    st = VerifyStep(w, path=path); st.run(); torch.cuda.synchronize()
    ref = _oracle("edges", w)
    _check_marshal(st, ref)
    out, lse = ref.attention()
    compare_attention(st.out, st.lse, out, lse)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("cid", [1, 2])
def test_config_full(cid, path):
    w = W.config(cid)
    st = VerifyStep(w, path=path); st.run(); torch.cuda.synchronize()
    ref = _oracle(cid, w)
    _check_marshal(st, ref)
    out, lse = ref.attention()
    compare_attention(st.out, st.lse, out, lse)


@pytest.mark.parametrize("splits", [1, 7, 64, 256])
@pytest.mark.parametrize("path", PATHS)
def test_forced_splits(path, splits):
    w = W.make_workload("splits", 16, [3000, 20000], "uniform", [32, 8], 65536, seed=5)
    st = VerifyStep(w, path=path, max_splits=splits); st.run(); torch.cuda.synchronize()
    ref = _oracle("splits", w)
    rows = sample_rows(w, 12, seed=2)
    out, lse = ref.attention(rows=rows)
    compare_attention(st.out, st.lse, out, lse, rows=rows)


@pytest.mark.parametrize("path", PATHS)
def test_config4_long_prefix(path):
    w = W.config(4)
    for splits in (64, 256):
        st = VerifyStep(w, path=path, max_splits=splits); st.run(); torch.cuda.synchronize()
        ref = _oracle(4, w)
        _check_marshal(st, ref)
        rows = sample_rows(w, 16, seed=4)
        out, lse = ref.attention(rows=rows)
        compare_attention(st.out, st.lse, out, lse, rows=rows)
        del st


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("cid", [3, 5])
def test_config_sampled(cid, path):
    w = W.config(cid)
    st = VerifyStep(w, path=path); st.run(); torch.cuda.synchronize()
    ref = _oracle(cid, w)
    _check_marshal(st, ref)
    rows = sample_rows(w, 8 if cid == 3 else 4, seed=cid)
    out, lse = ref.attention(rows=rows)
    compare_attention(st.out, st.lse, out, lse, rows=rows)


def test_paths_agree_full_config3():
    """Every row of config 3: the two kernels agree within the tolerance."""
    w = W.config(3)
    a = VerifyStep(w, path=abi.PATH_SIMT); a.run()
    b = VerifyStep(w, path=abi.PATH_TC, pool=a.pool); b.run()
    torch.cuda.synchronize()
    d = (a.out.float() - b.out.float()).abs()
    assert float(d.max()) <= 1e-2 and float(d.mean()) <= 1e-3
    dl = (a.lse - b.lse).abs() / a.lse.abs().clamp(min=1.0)
    assert float(dl.max()) <= 1e-3


@pytest.mark.parametrize("path", PATHS)
def test_graph_capture_and_replay(path):
    """The whole step captured once, replayed on new contents of the same
    shapes; nothing is allocated while capturing."""
    w1 = W.make_workload("g", 8, [300, 1200, 77], "uniform", [16, 9, 30], 16384, seed=101)
    w2 = W.make_workload("g", 8, [300, 1200, 77], "uniform", [16, 9, 30], 16384, seed=202)
    st = VerifyStep(w1, path=path)
    st.run(); torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        before = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
        st.run()
        after = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    assert after == before
    for w in (w1, w2):
        st.pool.copy_(w.dense_pool("cuda"))
        st.load(w)
        g.replay(); torch.cuda.synchronize()
        ref = OracleRun(w)
        _check_marshal(st, ref)
        out, lse = ref.attention()
        compare_attention(st.out, st.lse, out, lse)


@pytest.mark.parametrize("bits", [False, True], ids=["bytes", "bits"])
def test_more_requests_than_one_launch_plans(bits):
    """300 requests of one 128-row tile each: the tensor-core path serves
    them in launches of at most 256 requests (no fall-back to the other
    kernel), split and unsplit, and agrees with the oracle on every row.
    With only 46..316 keys per request some outputs reach magnitudes of 2-4,
    where rounding the exact result to bf16 alone moves it by up to 0.0078,
    so the comparison adds that rounding (2^-9 |ref|) to the bounds."""
    import numpy as np
    rng = np.random.default_rng(300)
    prefix = [int(x) for x in rng.integers(30, 300, size=300)]
    w = W.make_workload("many", 8, prefix, "uniform", [16] * 300, 131072, seed=300)
    kv_len = sum(w.prefix_lens) + w.total_q
    assert abi.mla_tree_verify_launch_count(w.batch, w.total_q, w.heads, kv_len, 1, abi.PATH_AUTO) == 2
    assert abi.mla_tree_verify_launch_count(w.batch, w.total_q, w.heads, kv_len, 4, abi.PATH_TC) == 3
    ref = _oracle("many", w)
    out, lse = ref.attention()
    for splits in (1, 4):
        st = VerifyStep(w, path=abi.PATH_AUTO, max_splits=splits, mask_bits=bits)
        st.run()
        torch.cuda.synchronize()
        assert int(st.status.item()) == 0
        compare_attention(st.out, st.lse, out, lse, rounding_term=True)


def test_bad_slot_sets_status_and_skips():
    w = W.small(seed=8)
    st = VerifyStep(w, path=abi.PATH_SIMT)
    st.run(); torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    st.kv_indices[3] = w.num_slots + 5          # out of range, checked by the kernel
    st.verify(); torch.cuda.synchronize()
    assert int(st.status.item()) & abi.DEV_BAD_SLOT


def test_bad_parent_sets_status():
    w = W.small(seed=9)
    st = VerifyStep(w)
    st.parents[2] = 5                            # node 2's parent must be < 2
    st.run(); torch.cuda.synchronize()
    assert int(st.status.item()) & abi.DEV_BAD_PARENT


def test_mask_capacity_overflow_is_flagged():
    w = W.small(seed=10)
    st = VerifyStep(w)
    st.mask = st.mask[: st.mask.numel() // 2]
    st.run(); torch.cuda.synchronize()
    assert int(st.status.item()) & abi.DEV_BAD_INDPTR


def test_empty_batch_is_noop():
    q = torch.empty((0, 8, 576), dtype=torch.bfloat16, device="cuda")
    z32 = torch.zeros(1, dtype=torch.int32, device="cuda")
    z64 = torch.zeros(1, dtype=torch.int64, device="cuda")
    abi.mla_tree_verify(q, torch.zeros((4, 576), dtype=torch.bfloat16, device="cuda"),
                        torch.empty(0, dtype=torch.int32, device="cuda"), z32, z32,
                        torch.empty(0, dtype=torch.uint8, device="cuda"), z64, 0.1,
                        torch.empty((0, 8, 512), dtype=torch.bfloat16, device="cuda"),
                        torch.empty((0, 8), dtype=torch.float32, device="cuda"),
                        torch.empty(256, dtype=torch.uint8, device="cuda"))


def test_validate_mode_agrees_and_returns_tensor_core_result():
    """Validate mode: out/lse equal a plain tensor-core call bit for bit, the
    measured differences are within the verify tolerance, no mismatch bit;
    with tolerance 0 the two kernels' rounding differences set it."""
    w = W.config(2)
    st = VerifyStep(w, path=abi.PATH_TC); st.run(); torch.cuda.synchronize()
    nb = abi.mla_tree_verify_validate_workspace_bytes(w.batch, w.total_q, w.heads)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    diff = torch.full((2,), -1.0, dtype=torch.float32, device="cuda")
    out = torch.empty_like(st.out); lse = torch.empty_like(st.lse)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    abi.mla_tree_verify_validate(st.q, st.pool, st.kv_indices, st.kv_indptr, st.qo_indptr, st.mask,
                                 st.mask_indptr, st.sm_scale, out, lse, ws, diff, 1e-2, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out, st.out) and torch.equal(lse, st.lse)
    d = diff.cpu().tolist()
    assert 0.0 <= d[0] <= 1e-2 and 0.0 <= d[1] <= 1e-3
    abi.mla_tree_verify_validate(st.q, st.pool, st.kv_indices, st.kv_indptr, st.qo_indptr, st.mask,
                                 st.mask_indptr, st.sm_scale, out, lse, ws, diff, 0.0, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & abi.DEV_MISMATCH
    assert float(diff[0].item()) > 0.0
