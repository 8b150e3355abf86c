"""GPU parity over head counts that shape the (node, head) row tiles
differently: one head (a tile of 128 distinct draft nodes), head counts that
do not divide the 128-row tile (a node's heads straddle two tiles), and 128
heads (one node per tile). Both kernels, both mask forms, against the fp64
oracle."""
import pytest
import torch

import __graft_entry__
from speculative_decode_mla_tree_gb300 import abi, workloads as W
from speculative_decode_mla_tree_gb300.step import VerifyStep

from parity import OracleRun, compare_attention

pytestmark = pytest.mark.gpu
PATHS = [pytest.param(abi.PATH_SIMT, id="simt"), pytest.param(abi.PATH_TC, id="tcgen05")]

# heads -> (prefix lengths, tree sizes): at least 128 rows per request
SHAPES = {
    1: ([150, 431], [160, 200]),
    3: ([90, 700], [64, 50]),
    12: ([250, 33, 600], [20, 11, 24]),
    128: ([300, 120], [4, 3]),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    __graft_entry__.build()


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("bits", [False, True], ids=["bytes", "bits"])
@pytest.mark.parametrize("heads", sorted(SHAPES))
def test_head_counts(heads, bits, path):
    prefix, sizes = SHAPES[heads]
    w = W.make_workload("heads%d" % heads, heads, prefix, "uniform", sizes, 8192, seed=heads)
    st = VerifyStep(w, path=path, mask_bits=bits)
    st.run()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    out, lse = OracleRun(w).attention()
    compare_attention(st.out, st.lse, out, lse)


@pytest.mark.parametrize("heads", [3, 12])
def test_head_counts_forced_splits_tc(heads):
    """The same shapes cut into up to 5 splits per request, merged."""
    prefix, sizes = SHAPES[heads]
    w = W.make_workload("hsplit%d" % heads, heads, prefix, "uniform", sizes, 8192, seed=heads + 1)
    st = VerifyStep(w, path=abi.PATH_TC, mask_bits=True, max_splits=5)
    st.run()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    out, lse = OracleRun(w).attention()
    compare_attention(st.out, st.lse, out, lse)
