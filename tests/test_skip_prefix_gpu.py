"""GPU parity of the prefix-skip switch (mla_tree_verify_masked with
MASK_SKIP_PREFIX): with every prefix entry of the mask cleared, the switch
must give the oracle's result for the tree mask, and the same outputs bit
for bit as the plain call on the intact mask, on both kernels and both mask
forms."""
import numpy as np
import pytest
import torch

import __graft_entry__
import oracle
from speculative_decode_mla_tree_gb300 import abi, workloads as W
from speculative_decode_mla_tree_gb300.step import VerifyStep

from parity import OracleRun, bits as raw_bits, compare_attention, sample_rows

pytestmark = pytest.mark.gpu
PATHS = [pytest.param(abi.PATH_SIMT, id="simt"), pytest.param(abi.PATH_TC, id="tcgen05")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    __graft_entry__.build()


def _clear_prefix(st, bits):
    """A copy of the step's mask with every prefix entry cleared: bytes
    j < P_b, or in the bit form every bit j < P_b."""
    qptr = st.qo_indptr.cpu().numpy().astype(np.int64)
    kptr = st.kv_indptr.cpu().numpy().astype(np.int64)
    if bits:
        m = st.mask_words.cpu().numpy().view(np.uint32).copy()
        mptr = st.mask_word_indptr.cpu().numpy()
    else:
        m = st.mask.cpu().numpy().copy()
        mptr = st.mask_indptr.cpu().numpy()
    for b in range(len(qptr) - 1):
        n, L = int(qptr[b + 1] - qptr[b]), int(kptr[b + 1] - kptr[b])
        P = L - n
        if bits:
            W_b = (L + 31) // 32
            for i in range(n):
                row = int(mptr[b]) + i * W_b
                m[row:row + P // 32] = 0
                if P % 32:
                    m[row + P // 32] &= np.uint32((0xFFFFFFFF << (P % 32)) & 0xFFFFFFFF)
        else:
            for i in range(n):
                m[int(mptr[b]) + i * L:int(mptr[b]) + i * L + P] = 0
    t = torch.from_numpy(m.view(np.int32) if bits else m).to(st.out.device)
    return t


def _oracle_skip(w, rows=None):
    """The oracle with the switch on, over the byte mask with every prefix
    byte cleared."""
    ref = OracleRun(w)
    m = ref.mask.copy()
    qptr = w.qo_indptr.numpy().astype(np.int64)
    for b in range(len(qptr) - 1):
        n = int(qptr[b + 1] - qptr[b])
        L = int(ref.kv_indptr[b + 1] - ref.kv_indptr[b])
        for i in range(n):
            m[ref.mask_indptr[b] + i * L:ref.mask_indptr[b] + i * L + L - n] = 0
    return oracle.verify_attention(raw_bits(w.q), ref.pool, ref.kv_indices, ref.kv_indptr,
                                   w.qo_indptr, m, ref.mask_indptr, w.heads, w.sm_scale, rows=rows,
                                   skip_prefix=True)


def _run_masked(st, mask, bits, flags):
    out = torch.empty_like(st.out)
    lse = torch.empty_like(st.lse)
    mptr = st.mask_word_indptr if bits else st.mask_indptr
    abi.mla_tree_verify_masked(st.q, st.pool, st.kv_indices, st.kv_indptr, st.qo_indptr, mask, mptr,
                               flags | (abi.MASK_BITS if bits else 0), st.sm_scale, out, lse,
                               st.workspace, st.max_splits, st.path, st.status)
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    return out, lse


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("bits", [False, True], ids=["bytes", "bits"])
def test_skip_prefix_ignores_prefix_entries(path, bits):
    w = W.config(2)
    st = VerifyStep(w, path=path, mask_bits=bits)
    st.run()
    torch.cuda.synchronize()
    cleared = _clear_prefix(st, bits)
    out, lse = _run_masked(st, cleared, bits, abi.MASK_SKIP_PREFIX)
    # the same visibility as the intact tree mask: the same bits
    assert torch.equal(out, st.out) and torch.equal(lse, st.lse)
    o_ref, l_ref = _oracle_skip(w)
    compare_attention(out, lse, o_ref, l_ref)
    # without the switch the cleared prefix really is gone
    o2, _ = _run_masked(st, cleared, bits, 0)
    assert not torch.equal(o2, st.out)


@pytest.mark.parametrize("bits", [False, True], ids=["bytes", "bits"])
def test_skip_prefix_long_prefix_tc(bits):
    """64 heads, 32 requests of prefix 8192: the kernel variant for long
    work, split over many items per cluster."""
    w = W.config(3)
    st = VerifyStep(w, path=abi.PATH_TC, mask_bits=bits)
    st.run()
    torch.cuda.synchronize()
    out, lse = _run_masked(st, _clear_prefix(st, bits), bits, abi.MASK_SKIP_PREFIX)
    assert torch.equal(out, st.out) and torch.equal(lse, st.lse)
    rows = sample_rows(w, 6, seed=33)
    o_ref, l_ref = _oracle_skip(w, rows=rows)
    compare_attention(out, lse, o_ref, l_ref, rows=rows)


@pytest.mark.parametrize("splits", [1, 7])
def test_skip_prefix_forced_splits(splits):
    """Split edges that fall inside and across the prefix boundary."""
    w = W.make_workload("skipsplit", 8, [37, 300, 1000], "uniform", [16, 20, 24], 4096, seed=5)
    st = VerifyStep(w, path=abi.PATH_TC, mask_bits=True, max_splits=splits)
    st.run()
    torch.cuda.synchronize()
    out, lse = _run_masked(st, _clear_prefix(st, True), True, abi.MASK_SKIP_PREFIX)
    assert torch.equal(out, st.out) and torch.equal(lse, st.lse)
    o_ref, l_ref = _oracle_skip(w)
    compare_attention(out, lse, o_ref, l_ref)
