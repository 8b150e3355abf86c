"""Failure detection of the tensor-core kernel without a GPU fault.

Every wait inside the kernel is bounded. The test shortens the bound to
1 ms and tells the kernel's copy engines to issue nothing from one work item
on, so the waits on that item's keys run out: the kernel must report
MT_DEV_TIMEOUT through the status word, drain what it has in flight and
exit, and the very next normal call on the same stream must be correct."""
import pytest
import torch

import __graft_entry__
from speculative_decode_mla_tree_gb300 import abi, workloads as W
from speculative_decode_mla_tree_gb300.step import VerifyStep

from parity import OracleRun, compare_attention, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    __graft_entry__.build()
    yield
    abi.mla_tree_test_wait_limits(-1, 0)


def _workload():
    # 4 requests x 32 tiles of 128 (node, head) rows: more work items than
    # clusters, so a cluster's second item can be dropped too
    return W.make_workload("timeout", 64, [700, 900, 400, 1100], "uniform", [64] * 4, 8192, seed=71)


_ref = {}


@pytest.mark.parametrize("drop", [0, 100], ids=["first_item", "second_round_item"])
def test_wait_gives_up_then_next_call_is_correct(drop):
    w = _workload()
    st = VerifyStep(w, path=abi.PATH_TC, max_splits=1, mask_bits=True)
    st.run()                                    # a normal call first
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    abi.mla_tree_test_wait_limits(drop, 1_000_000)
    try:
        st.verify()
        torch.cuda.synchronize()
    finally:
        abi.mla_tree_test_wait_limits(-1, 0)
    assert int(st.status.item()) & abi.DEV_TIMEOUT
    # the device is usable and the next call on the same stream is right
    st.status.zero_()
    st.out.zero_()
    st.verify()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    if "r" not in _ref:
        rows = sample_rows(w, 16, seed=7)
        _ref["r"] = (rows, OracleRun(w).attention(rows=rows))
    rows, (out, lse) = _ref["r"]
    compare_attention(st.out, st.lse, out, lse, rows=rows)


def test_hooks_reject_bad_arguments():
    with pytest.raises(abi.MlaTreeError):
        abi.mla_tree_test_wait_limits(-2, 0)
    with pytest.raises(abi.MlaTreeError):
        abi.mla_tree_test_wait_limits(-1, -5)
