"""GPU parity at the edges of the arithmetic, and on the two largest
workloads the way a serving engine runs them, against the fp64 oracle.

* Stress inputs (workloads.stress): a peaked softmax (queries x8), latent
  half-dot-products that are large and cancel exactly, and values beyond the
  fp16 range. Every factor is a power of two, so the inputs are exact in
  bf16 and the oracle's expectations need no other reasoning. Both kernels,
  both mask forms, unsplit and split (the split partials and their merge are
  where a narrow intermediate format would overflow or round). These inputs push single
  outputs to magnitudes of 4-5, so the comparison adds the bf16 rounding of
  the output itself (2^-9 |ref|) to the stated bounds.
* The 64-request ragged workload (prefixes 128..131072, 8..64-node trees,
  64 heads, 2^22-slot pool), captured once as one CUDA graph of the whole
  step (fused marshaling + verify) and replayed on a second draw of the same
  shapes: >= 256 sampled rows covering every request, both draws.
* The 4-request, 200000-key workload in full (all 2048 rows) at 64 and 256
  splits."""
import numpy as np
import pytest
import torch

import __graft_entry__
from speculative_decode_mla_tree_gb300 import abi, workloads as W
from speculative_decode_mla_tree_gb300.step import VerifyStep

from parity import OracleRun, compare_attention, sample_rows

pytestmark = pytest.mark.gpu
PATHS = [pytest.param(abi.PATH_SIMT, id="simt"), pytest.param(abi.PATH_TC, id="tcgen05")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    __graft_entry__.build()


def _base():
    """Three requests of 512, 256 and 384 (node, head) rows: several 128-row
    tiles, ragged key counts."""
    return W.make_workload("stress", 16, [3000, 1500, 700], "uniform", [32, 16, 24], 16384, seed=61)


_refs = {}


def _ref(kind):
    if kind not in _refs:
        w = W.stress(_base(), kind)
        _refs[kind] = (w, OracleRun(w).attention())
    return _refs[kind]


@pytest.mark.parametrize("bits", [True, False], ids=["bits", "bytes"])
@pytest.mark.parametrize("splits", [0, 7], ids=["auto", "split7"])
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("kind", W.STRESS_KINDS)
def test_stress_inputs(kind, path, splits, bits):
    """Both mask forms: the tensor-core kernel applies the bit form in the
    softmax and the byte form in the score exchange (hidden columns sent as
    -inf), so each form meets the stress inputs on its own code."""
    w, (out, lse) = _ref(kind)
    st = VerifyStep(w, path=path, max_splits=splits, mask_bits=bits)
    st.run()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    if kind == "huge_v":
        # values are 2^17 times those of a normal draw: compare at that scale
        s = 2.0 ** 17
        assert torch.isfinite(st.out.float()).all()
        compare_attention(st.out.float() / s, st.lse, out / s, lse, rounding_term=True)
    else:
        compare_attention(st.out, st.lse, out, lse, rounding_term=True)


def test_config5_graph_replay_two_draws():
    """The whole step of the 64-request workload as one captured graph
    (nothing allocated while capturing), replayed on two draws of the same
    shapes; 4 rows of every request (256) compared per draw."""
    w1 = W.config(5)
    w2 = W.redraw(w1, 2005)
    st = VerifyStep(w1, fused=True)
    st.run()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        before = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
        st.run()
        after = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    assert after == before
    for k, w in enumerate((w2, w1)):
        st.pool.copy_(w.dense_pool("cuda"))
        st.load(w)
        st.status.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(st.status.item()) == 0
        rows = sample_rows(w, 4, seed=50 + k)
        assert len(rows) >= 256 and len({r[0] for r in rows}) >= w.batch
        out, lse = OracleRun(w).attention(rows=rows)
        compare_attention(st.out, st.lse, out, lse, rows=rows)


_c4 = {}


@pytest.mark.parametrize("splits", [64, 256])
@pytest.mark.parametrize("path", PATHS)
def test_config4_full(path, splits):
    """All 2048 rows of the 200000-key workload."""
    if "w" not in _c4:
        w = W.config(4)
        _c4["w"] = w
        _c4["ref"] = OracleRun(w).attention()
    w = _c4["w"]
    out, lse = _c4["ref"]
    st = VerifyStep(w, path=path, max_splits=splits, fused=True)
    st.run()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    assert np.isfinite(out).all()
    compare_attention(st.out, st.lse, out, lse)
