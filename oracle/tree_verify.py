"""The oracle proper: scatter, index marshaling, tree mask, masked attention,
split partials and their log-sum-exp merge, all on the CPU in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Notation per request b: n_b draft nodes (query tokens), P_b prefix slots,
L_b = P_b + n_b key/value positions, H heads. A pool row holds 576 bf16
values: 512 latent dims followed by 64 rope dims; the key is the whole row,
the value is its first 512 dims (absorbed MLA: the query carries 512
absorbed-latent dims and 64 rope dims -- "Pivot to Live Cutover" page,
section "Input Knowledge Required").
"""
from __future__ import annotations

import numpy as np

D_QK = 576
D_V = 512


def _as_np(x):
    """Accept numpy arrays or CPU torch tensors (bf16 tensors as raw bits)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            if x.dtype == torch.bfloat16:
                return x.contiguous().view(torch.int16).numpy().view(np.uint16)
            return x.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x)


def bf16_bits_to_f64(bits):
    """Widen raw bf16 bit patterns exactly to float64.

    A bf16 value is the upper half of an IEEE float32, so shifting its 16 bits
    into the high half of a 32-bit word gives that float32 exactly, and float32
    widens to float64 exactly.
    """
    b = _as_np(bits).astype(np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def draft_kv_scatter(pool_bits, src_bits, out_cache_loc):
    """Write each draft token's key/value row into the pool at its slot.

    "Flipping the Switch" page, section "The Long Road to Parity": in the
    extend path the draft tokens' KV does not come through ``kv_indices``; it
    arrives as separate k/v tensors and is stored at ``out_cache_loc``. The
    pool row at ``out_cache_loc[t]`` becomes ``src[t]`` bit for bit; every
    other row is unchanged. Returns a new array (raw bf16 bits).
    """
    pool = _as_np(pool_bits).astype(np.uint16).copy()
    src = _as_np(src_bits).astype(np.uint16)
    loc = _as_np(out_cache_loc).astype(np.int64)
    for t in range(loc.shape[0]):
        pool[loc[t], :] = src[t, :D_QK]
    return pool


def kv_indices_build(prefix_indices, prefix_indptr, out_cache_loc, qo_indptr):
    """Concatenate, per request, its prefix slots with its draft-token slots.

    "Flipping the Switch" page, section "The Long Road to Parity": the fix for
    the uncorrelated output was to rebuild the full KV index array by joining
    the prefix slots with the draft tokens' slot locations. Position j < P_b
    of request b is prefix slot j; position P_b + k is draft token k's slot.
    Returns (kv_indices int32 [sum L_b], kv_indptr int32 [B+1]).
    """
    pidx = _as_np(prefix_indices).astype(np.int64)
    pptr = _as_np(prefix_indptr).astype(np.int64)
    loc = _as_np(out_cache_loc).astype(np.int64)
    qptr = _as_np(qo_indptr).astype(np.int64)
    batch = len(qptr) - 1
    kv_indices = []
    kv_indptr = [0]
    for b in range(batch):
        row = np.concatenate([pidx[pptr[b]:pptr[b + 1]],     # prefix slots, in order
                              loc[qptr[b]:qptr[b + 1]]])     # then the draft slots
        kv_indices.append(row)
        kv_indptr.append(kv_indptr[-1] + len(row))
    flat = np.concatenate(kv_indices) if kv_indices else np.zeros(0, dtype=np.int64)
    return flat.astype(np.int32), np.array(kv_indptr, dtype=np.int32)


def ancestors_or_self(parents_local):
    """For each node of one draft tree, the set of nodes it may attend to.

    A draft node sees itself and every node on its path back to the prefix,
    found here by walking parent links one step at a time (brute force).
    ``parents_local[i]`` is -1 (hangs off the prefix) or an earlier node.
    The tree-mask meaning -- which speculative tokens a query may see -- is
    the "Pivot to Live Cutover" page, section "The Technical Investigation:
    Probing the Integration Surface".
    """
    par = [int(p) for p in parents_local]
    out = []
    for i in range(len(par)):
        seen = set()
        k = i
        while k != -1:
            if not (-1 <= par[k] < k):
                raise ValueError("parent of node %d is %d, not in [-1, %d]" % (k, par[k], k - 1))
            seen.add(k)
            k = par[k]
        out.append(seen)
    return out


def tree_mask_pack(parents, qo_indptr, kv_indptr):
    """Build the flat per-request visibility mask and its offsets.

    "Flipping the Switch" page, section "The Long Road to Parity": the mask
    row stride is the full sequence length, prefix plus draft (the logged
    ``mask=(270,)`` is 9 rows of 21 + 9 columns). "Pivot to Live Cutover"
    page, same investigation section: the mask is one flat buffer with a
    per-sequence offset ``mask_indptr``. One byte per (row, column), 1 =
    visible; prefix columns are all visible, draft column P_b + k is visible
    from row i when k is i or an ancestor of i.
    Returns (mask_indptr int64 [B+1], packed_mask uint8 [mask_indptr[B]]).
    """
    par = _as_np(parents).astype(np.int64)
    qptr = _as_np(qo_indptr).astype(np.int64)
    kptr = _as_np(kv_indptr).astype(np.int64)
    batch = len(qptr) - 1
    mask_indptr = [0]
    chunks = []
    for b in range(batch):
        n = qptr[b + 1] - qptr[b]
        L = kptr[b + 1] - kptr[b]
        P = L - n
        vis = ancestors_or_self(par[qptr[b]:qptr[b + 1]])
        m = np.zeros((n, L), dtype=np.uint8)
        m[:, :P] = 1                      # every prefix column is visible
        for i in range(n):
            for k in vis[i]:
                m[i, P + k] = 1
        chunks.append(m.reshape(-1))
        mask_indptr.append(mask_indptr[-1] + n * L)
    packed = np.concatenate(chunks) if chunks else np.zeros(0, dtype=np.uint8)
    return np.array(mask_indptr, dtype=np.int64), packed


def tree_mask_pack_bits(parents, qo_indptr, kv_indptr):
    """The same visibility as ``tree_mask_pack``, one bit per (row, column).

    "Pivot to Live Cutover" page, section "The Technical Investigation:
    Probing the Integration Surface", calls the custom mask a packed bitmask.
    This encoding keeps that literal reading next to the byte-per-element
    one: row i of request b holds its L_b visibility bits, column j in bit
    j % 32 of word j // 32 (least significant bit first), in
    W_b = ceil(L_b / 32) uint32 words; bits past L_b are zero. Rows follow
    each other, requests too: row i of request b starts at word
    mask_word_indptr[b] + i * W_b.
    Returns (mask_word_indptr int64 [B+1], mask_words uint32 [mask_word_indptr[B]]).
    """
    par = _as_np(parents).astype(np.int64)
    qptr = _as_np(qo_indptr).astype(np.int64)
    kptr = _as_np(kv_indptr).astype(np.int64)
    batch = len(qptr) - 1
    indptr = [0]
    chunks = []
    for b in range(batch):
        n = int(qptr[b + 1] - qptr[b])
        L = int(kptr[b + 1] - kptr[b])
        P = L - n
        W = (L + 31) // 32
        vis = ancestors_or_self(par[qptr[b]:qptr[b + 1]])
        words = np.zeros((n, W), dtype=np.uint64)
        for i in range(n):
            cols = list(range(P)) + [P + k for k in vis[i]]
            for j in cols:
                words[i, j // 32] |= np.uint64(1) << np.uint64(j % 32)
        chunks.append(words.astype(np.uint32).reshape(-1))
        indptr.append(indptr[-1] + n * W)
    packed = np.concatenate(chunks) if chunks else np.zeros(0, dtype=np.uint32)
    return np.array(indptr, dtype=np.int64), packed


def _request_rows(qptr, heads, rows):
    """Group requested (token, head) rows by request; None = all rows."""
    batch = len(qptr) - 1
    groups = {}
    if rows is None:
        for b in range(batch):
            for t in range(qptr[b], qptr[b + 1]):
                groups.setdefault(b, []).extend((t, h) for h in range(heads))
        return groups
    for t, h in rows:
        b = int(np.searchsorted(qptr, t, side="right") - 1)
        groups.setdefault(b, []).append((int(t), int(h)))
    return groups


def verify_attention(q_bits, kv_bits, kv_indices, kv_indptr, qo_indptr, packed_mask,
                     mask_indptr, heads, sm_scale, rows=None, kv_range=None, skip_prefix=False):
    """Exact masked scaled-dot-product attention of every draft row.

    What the verify kernel computes ("Flipping the Switch" page, section "The
    Long Road to Parity"; "Pivot to Live Cutover" page, sections "The
    Technical Investigation" and "Input Knowledge Required"): row (t, h) of
    request b scores every key position j of the request,
    s_j = sm_scale * <q[t, h, :576], kv[slot_j, :576]>, keeps the positions
    whose mask byte is nonzero, and returns
        lse = log sum_vis exp(s_j)                (natural log)
        out = sum_vis exp(s_j - lse) * kv[slot_j, :512].
    A row with no visible position gets out = 0 and lse = -inf.

    The max-shifted form below is the same quantity, written so that exp does
    not overflow. ``rows`` restricts the work to a list of (t, h) pairs;
    ``kv_range`` = (lo, hi) restricts every request to logical positions
    [lo_b, hi_b) (a list of pairs, one per request) for split partials.
    ``skip_prefix``: the switch that leaves the mask unread over the prefix
    ("Pivot to Live Cutover" page, section "The Technical Investigation"):
    the first P_b = L_b - n_b positions are visible to every row whatever
    their mask bytes hold.

    Returns (out float64 [T, H, 512], lse float64 [T, H]); rows not computed
    are NaN.
    """
    qf_bits = _as_np(q_bits)
    kvf_bits = _as_np(kv_bits)
    kidx = _as_np(kv_indices).astype(np.int64)
    kptr = _as_np(kv_indptr).astype(np.int64)
    qptr = _as_np(qo_indptr).astype(np.int64)
    mask = _as_np(packed_mask)
    mptr = _as_np(mask_indptr).astype(np.int64)
    T = int(qptr[-1])
    scale = np.float64(np.float32(sm_scale))
    out = np.full((T, heads, D_V), np.nan)
    lse = np.full((T, heads), np.nan)
    for b, pairs in _request_rows(qptr, heads, rows).items():
        n = qptr[b + 1] - qptr[b]
        L = kptr[b + 1] - kptr[b]
        lo, hi = (0, L) if kv_range is None else kv_range[b]
        slots = kidx[kptr[b] + lo:kptr[b] + hi]
        K = bf16_bits_to_f64(kvf_bits[slots, :D_QK])          # [Lr, 576]
        V = K[:, :D_V]                                        # [Lr, 512]
        vis_full = mask[mptr[b]:mptr[b] + n * L].reshape(n, L) != 0
        if skip_prefix:
            vis_full = vis_full.copy()
            vis_full[:, :L - n] = True
        vis_all = vis_full[:, lo:hi]
        ts = np.array([p[0] for p in pairs])
        hs = np.array([p[1] for p in pairs])
        Q = bf16_bits_to_f64(qf_bits[ts, hs, :D_QK])          # [R, 576]
        S = scale * (Q @ K.T)                                 # [R, Lr]
        vis = vis_all[ts - qptr[b]]                           # [R, Lr]
        S = np.where(vis, S, -np.inf)
        m = S.max(axis=1) if S.shape[1] else np.full(len(pairs), -np.inf)
        empty = ~np.isfinite(m)
        m_safe = np.where(empty, 0.0, m)
        e = np.where(vis, np.exp(S - m_safe[:, None]), 0.0)
        lsum = e.sum(axis=1)
        row_lse = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, lsum)))
        w = np.where(empty[:, None], 0.0, e / np.where(empty, 1.0, lsum)[:, None])
        O = w @ V
        out[ts, hs] = O
        lse[ts, hs] = row_lse
    return out, lse


def split_bounds(L, splits):
    """Cut logical positions [0, L) into ``splits`` contiguous pieces of near
    equal length (the first L % splits pieces one longer)."""
    base, extra = divmod(L, splits)
    bounds, lo = [], 0
    for s in range(splits):
        hi = lo + base + (1 if s < extra else 0)
        bounds.append((lo, hi))
        lo = hi
    return bounds


def verify_attention_split(q_bits, kv_bits, kv_indices, kv_indptr, qo_indptr, packed_mask,
                           mask_indptr, heads, sm_scale, splits, rows=None):
    """Split-KV partials: attention of each row over each piece of its
    request's key positions, each piece normalised on its own.

    The pages' kernel is a KV-split flash-decode design ("Flipping the Switch"
    page, section "The Broader Context": split count raised from 16 to 64).
    Piece s of request b yields o_s (its own softmax-weighted V average) and
    lse_s (its own log-sum-exp); an empty piece gives o_s = 0, lse_s = -inf.
    Returns a list of (o_s, lse_s), one per split index.
    """
    kptr = _as_np(kv_indptr).astype(np.int64)
    batch = len(kptr) - 1
    per_req = [split_bounds(int(kptr[b + 1] - kptr[b]), splits) for b in range(batch)]
    parts = []
    for s in range(splits):
        rng = [per_req[b][s] for b in range(batch)]
        parts.append(verify_attention(q_bits, kv_bits, kv_indices, kv_indptr, qo_indptr,
                                      packed_mask, mask_indptr, heads, sm_scale,
                                      rows=rows, kv_range=rng))
    return parts


def lse_merge(parts):
    """Combine split partials into the full result.

    For one row with pieces (o_s, lse_s):
        lse = log sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * o_s,
    which equals attention over the union of the pieces because each o_s is
    its piece's exp-weighted V sum divided by exp(lse_s). Empty pieces
    (lse_s = -inf) contribute nothing; all-empty rows give out 0, lse -inf.
    """
    lses = np.stack([p[1] for p in parts])                 # [S, T, H]
    outs = np.stack([p[0] for p in parts])                 # [S, T, H, 512]
    m = lses.max(axis=0)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    w = np.where(np.isfinite(lses), np.exp(lses - m_safe[None]), 0.0)
    tot = w.sum(axis=0)
    lse = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, tot)))
    coef = np.where(empty[None], 0.0, w / np.where(empty, 1.0, tot)[None])
    outs = np.where(np.isfinite(outs), outs, 0.0)
    out = (coef[..., None] * outs).sum(axis=0)
    return out, lse
