"""Shared helpers of the parity tests: oracle results for a workload and the
comparison rules (bit-exact for integers and bytes; for attention the
tolerances of the verify contract)."""
import numpy as np
import torch

import oracle

OUT_MAX_ABS = 1e-2
OUT_MEAN_ABS = 1e-3
LSE_REL = 1e-3


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class OracleRun:
    """Oracle scatter / indices / mask for a workload (attention on demand)."""

    def __init__(self, w):
        self.w = w
        self.pool = oracle.draft_kv_scatter(bits(w.dense_pool()), bits(w.draft_kv), w.out_cache_loc)
        self.kv_indices, self.kv_indptr = oracle.kv_indices_build(
            w.prefix_indices, w.prefix_indptr, w.out_cache_loc, w.qo_indptr)
        self.mask_indptr, self.mask = oracle.tree_mask_pack(w.parents, w.qo_indptr, self.kv_indptr)

    def attention(self, rows=None):
        return oracle.verify_attention(bits(self.w.q), self.pool, self.kv_indices, self.kv_indptr,
                                       self.w.qo_indptr, self.mask, self.mask_indptr, self.w.heads,
                                       self.w.sm_scale, rows=rows)


def sample_rows(w, per_request, seed=0):
    """(t, h) rows covering every request: its first and last token plus
    random ones, random heads."""
    rng = np.random.default_rng(seed)
    qo = w.qo_indptr.tolist()
    rows = []
    for b in range(w.batch):
        n = qo[b + 1] - qo[b]
        if n == 0:
            continue
        ts = {qo[b], qo[b + 1] - 1}
        while len(ts) < min(per_request, n):
            ts.add(qo[b] + int(rng.integers(0, n)))
        for t in sorted(ts):
            rows.append((t, int(rng.integers(0, w.heads))))
    return rows


# bf16 keeps 8 significant bits: rounding the output to the nearest bf16
# moves it by at most 2^-9 of its magnitude
BF16_HALF_ULP_REL = 2.0 ** -9


def compare_attention(out_gpu, lse_gpu, out_ref, lse_ref, rows=None, rounding_term=False):
    """Assert the verify tolerances; returns the stats.

    rounding_term: the absolute bounds (max 1e-2, mean 1e-3) hold for
    outputs below about 2.5 in magnitude, where the final rounding to bf16
    moves a value by less than 0.005. Inputs that drive single outputs
    further out (a peaked softmax returns single value entries of size 4-5,
    where half a bf16 ulp is 0.0156) add that unavoidable rounding, at most
    2^-9 |ref| per element, to both bounds."""
    o = out_gpu.detach().float().cpu().numpy().astype(np.float64)
    l = lse_gpu.detach().cpu().numpy().astype(np.float64)
    if rows is not None:
        ts = np.array([r[0] for r in rows]); hs = np.array([r[1] for r in rows])
        o, l, out_ref, lse_ref = o[ts, hs], l[ts, hs], out_ref[ts, hs], lse_ref[ts, hs]
    assert np.isfinite(out_ref).all()
    err = np.abs(o - out_ref)
    if rounding_term:
        err = np.maximum(err - BF16_HALF_ULP_REL * np.abs(out_ref), 0.0)
    finite = np.isfinite(lse_ref)
    assert (np.isneginf(l[~finite])).all(), "rows with nothing visible must give lse = -inf"
    lerr = np.abs(l[finite] - lse_ref[finite]) / np.maximum(1.0, np.abs(lse_ref[finite]))
    stats = {"max_abs": float(err.max()) if err.size else 0.0,
             "mean_abs": float(err.mean()) if err.size else 0.0,
             "lse_rel": float(lerr.max()) if lerr.size else 0.0}
    assert stats["max_abs"] <= OUT_MAX_ABS, stats
    assert stats["mean_abs"] <= OUT_MEAN_ABS, stats
    assert stats["lse_rel"] <= LSE_REL, stats
    return stats
