"""Seeded synthetic inputs for tree-verify MLA attention.

This module only draws random inputs (tree shapes, prefix lengths, pool
slots, bf16 query / latent-KV values). It holds none of the method's
arithmetic: no scatter, no index marshaling, no mask building, no attention.
Both the fp64 oracle (through the tests) and the CUDA library consume what it
produces, so it is the one module the two sides share.

Workload recipes follow the shapes the pages report for the live verify call
("Flipping the Switch" page, section "The Long Road to Parity": q of shape
(9, 8, 576), prefix 21, 9 draft tokens) and the five benchmark configurations
of the project description:

  c1  1 request, prefix 21, 9-node random tree, 8 heads, 4096-slot pool
  c2  8 requests, prefix U{1024..4096}, 16-node trees (branching <= 3),
      8 heads, 65536-slot pool
  c3  32 requests, prefix 8192, 64-node trees (branching <= 4, depth <= 8),
      64 heads, latent values N(0, 0.5^2), rope values N(0, 1), 300000 slots
  c4  4 requests, prefix 200000, 32-node random trees, 16 heads, 2^20 slots
  c5  64 requests, prefix floor(exp(U(ln 128, ln 131072))), tree sizes
      U{8..64}, even requests chains and odd requests random trees,
      64 heads, 2^22 slots

Every draw comes from one CPU ``torch.Generator`` seeded with
``1000 + config id`` in a fixed order, so a workload is reproducible on any
host. Values are drawn in float32 and rounded to bf16 by torch.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

D_QK = 576        # absorbed MLA query/key width: 512 latent + 64 rope dims
D_LATENT = 512    # latent dims; V is this leading slice of each pool row
D_ROPE = 64
D_V = 512


@dataclass
class Workload:
    """One batch of tree-verify inputs (all tensors on the CPU).

    Token order: requests are concatenated; request b owns query tokens
    ``qo_indptr[b] .. qo_indptr[b+1]-1`` (its draft-tree nodes in node order).
    ``parents`` holds, per token, the local index of its parent node inside
    its own request, or -1 for a node that hangs directly off the prefix.
    ``pool_slots``/``pool_rows`` give the pool contents before the draft rows
    are scattered: every slot the batch touches (prefix and draft slots) holds
    a drawn row; all other slots are zero and are never read.
    """

    name: str
    heads: int
    num_slots: int
    sm_scale: float
    prefix_lens: list
    tree_sizes: list
    parents: torch.Tensor          # int32 [T]
    qo_indptr: torch.Tensor        # int32 [B+1]
    prefix_indptr: torch.Tensor    # int32 [B+1]
    prefix_indices: torch.Tensor   # int32 [sum P]
    out_cache_loc: torch.Tensor    # int32 [T]
    q: torch.Tensor                # bf16 [T, H, 576]
    draft_kv: torch.Tensor         # bf16 [T, 576] rows to scatter
    pool_slots: torch.Tensor       # int64 [R] slots holding drawn rows
    pool_rows: torch.Tensor        # bf16 [R, 576]
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return len(self.prefix_lens)

    @property
    def total_q(self) -> int:
        return int(self.qo_indptr[-1])

    def dense_pool(self, device="cpu") -> torch.Tensor:
        """The whole pool [num_slots, 576] bf16 before the draft scatter."""
        pool = torch.zeros((self.num_slots, D_QK), dtype=torch.bfloat16, device=device)
        pool.index_copy_(0, self.pool_slots.to(device), self.pool_rows.to(device))
        return pool

    def kv_bytes(self) -> int:
        """Latent-KV bytes one verify call must read (each row once)."""
        return sum(p + n for p, n in zip(self.prefix_lens, self.tree_sizes)) * D_QK * 2


# ---------------------------------------------------------------- tree shapes

def _parents_uniform(n, g):
    """parent[i] uniform in {-1, ..., i-1}: a random forest in topological order."""
    out = []
    for i in range(n):
        out.append(int(torch.randint(-1, i, (1,), generator=g)))
    return out


def _parents_chain(n, g=None):
    return [i - 1 for i in range(n)]


def _parents_bounded(n, g, max_children, max_depth=None):
    """Node 0 is the root under the prefix; node i>0 picks its parent uniformly
    among earlier nodes that still have fewer than ``max_children`` children
    and (if given) depth below ``max_depth`` (the root has depth 1)."""
    parents = [-1]
    children = [0]
    depth = [1]
    for i in range(1, n):
        cands = [k for k in range(i)
                 if children[k] < max_children and (max_depth is None or depth[k] < max_depth)]
        if not cands:
            raise ValueError("tree constraints cannot place node %d" % i)
        k = cands[int(torch.randint(0, len(cands), (1,), generator=g))]
        parents.append(k)
        children[k] += 1
        children.append(0)
        depth.append(depth[k] + 1)
    return parents


def tree_parents(rule, n, g):
    if rule == "uniform":
        return _parents_uniform(n, g)
    if rule == "chain":
        return _parents_chain(n)
    if rule.startswith("branch"):
        # "branch3" or "branch4d8"
        spec = rule[len("branch"):]
        if "d" in spec:
            k, d = spec.split("d")
            return _parents_bounded(n, g, int(k), int(d))
        return _parents_bounded(n, g, int(spec))
    raise ValueError(rule)


# ---------------------------------------------------------------- values

def _draw_rows(count, g, latent_std=1.0, rope_std=1.0):
    x = torch.randn((count, D_QK), generator=g, dtype=torch.float32)
    if latent_std != 1.0:
        x[:, :D_LATENT] *= latent_std
    if rope_std != 1.0:
        x[:, D_LATENT:] *= rope_std
    return x.to(torch.bfloat16)


def _draw_slots(total, num_slots, g, kv_layout):
    """Distinct pool slots for ``total`` tokens.

    shuffled:   a random permutation prefix of the pool (no two neighbours
                adjacent in general);
    contiguous: one run of consecutive slots at a random offset (a freshly
                allocated or defragmented pool);
    paged64:    random distinct pages of 64 consecutive slots, in random
                order (a paged pool with 64-slot pages).
    """
    if kv_layout == "shuffled":
        return torch.randperm(num_slots, generator=g)[:total].to(torch.int64)
    if kv_layout == "contiguous":
        off = int(torch.randint(0, num_slots - total + 1, (1,), generator=g))
        return torch.arange(off, off + total, dtype=torch.int64)
    if kv_layout == "paged64":
        pages = (total + 63) // 64
        pick = torch.randperm(num_slots // 64, generator=g)[:pages].to(torch.int64)
        return (pick[:, None] * 64 + torch.arange(64)[None, :]).reshape(-1)[:total]
    raise ValueError(kv_layout)


def make_workload(name, heads, prefix_lens, tree_rules, tree_sizes, num_slots, seed,
                  latent_std=1.0, rope_std=1.0, sm_scale=None, parents=None, g=None,
                  kv_layout="shuffled"):
    """Draw one workload.

    ``tree_rules`` is one rule name or a per-request list; ``parents`` may be
    given explicitly (list of per-request local parent lists) to build edge
    cases. Slots for all prefix and draft tokens are distinct, drawn by
    ``kv_layout`` (see ``_draw_slots``; default a random permutation prefix
    of the pool) and handed out request by request: the first P_b to the
    prefix, the next n_b to the draft tokens.
    """
    if g is None:
        g = torch.Generator().manual_seed(seed)
    batch = len(prefix_lens)
    if isinstance(tree_rules, str):
        tree_rules = [tree_rules] * batch
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(192.0)
    if parents is None:
        parents = [tree_parents(tree_rules[b], tree_sizes[b], g) for b in range(batch)]
    tree_sizes = [len(p) for p in parents]
    total_slots = sum(prefix_lens) + sum(tree_sizes)
    if total_slots > num_slots:
        raise ValueError("pool of %d slots cannot hold %d distinct rows" % (num_slots, total_slots))
    if kv_layout == "paged64" and (total_slots + 63) // 64 > num_slots // 64:
        raise ValueError("pool of %d slots cannot hold %d slots in 64-slot pages" % (num_slots, total_slots))
    slots = _draw_slots(total_slots, num_slots, g, kv_layout)

    prefix_indices, out_cache_loc = [], []
    off = 0
    for b in range(batch):
        prefix_indices.append(slots[off:off + prefix_lens[b]])
        off += prefix_lens[b]
        out_cache_loc.append(slots[off:off + tree_sizes[b]])
        off += tree_sizes[b]
    T = sum(tree_sizes)
    q = _draw_rows(T * heads, g, latent_std, rope_std).view(T, heads, D_QK)
    pool_rows = _draw_rows(total_slots, g, latent_std, rope_std)
    draft_kv = _draw_rows(T, g, latent_std, rope_std)

    def indptr(sizes):
        v = [0]
        for s in sizes:
            v.append(v[-1] + s)
        return torch.tensor(v, dtype=torch.int32)

    return Workload(
        name=name, heads=heads, num_slots=num_slots, sm_scale=float(sm_scale),
        prefix_lens=list(prefix_lens), tree_sizes=list(tree_sizes),
        parents=torch.tensor([p for ps in parents for p in ps], dtype=torch.int32),
        qo_indptr=indptr(tree_sizes), prefix_indptr=indptr(prefix_lens),
        prefix_indices=torch.cat(prefix_indices).to(torch.int32) if batch else torch.zeros(0, dtype=torch.int32),
        out_cache_loc=torch.cat(out_cache_loc).to(torch.int32) if batch else torch.zeros(0, dtype=torch.int32),
        q=q, draft_kv=draft_kv, pool_slots=slots, pool_rows=pool_rows,
        meta={"seed": seed, "rules": list(tree_rules) if tree_rules else None, "kv_layout": kv_layout,
              "latent_std": latent_std, "rope_std": rope_std},
    )


CONFIG_NAMES = {
    1: "c1: 1 req, prefix 21 + 9-node tree, 8 heads",
    2: "c2: 8 req, prefix U[1024,4096] + 16-node trees (branching<=3), 8 heads",
    3: "c3: 32 req, prefix 8192 + 64-node trees (branching<=4, depth<=8), 64 heads",
    4: "c4: 4 req, prefix 200000 + 32-node trees, 16 heads, split-KV",
    5: "c5: 64 req, prefix loguniform[128,131072] + 8..64-node trees, 64 heads, graph",
}


def config(cid: int, kv_layout: str = "shuffled") -> Workload:
    """The five benchmark configurations, seeded with 1000 + cid. ``kv_layout``
    varies only how pool slots are handed out (see ``_draw_slots``)."""
    g = torch.Generator().manual_seed(1000 + cid)
    seed = 1000 + cid
    kw = {"g": g, "kv_layout": kv_layout}
    if cid == 1:
        return make_workload("c1", 8, [21], "uniform", [9], 4096, seed, **kw)
    if cid == 2:
        P = [int(torch.randint(1024, 4097, (1,), generator=g)) for _ in range(8)]
        return make_workload("c2", 8, P, "branch3", [16] * 8, 65536, seed, **kw)
    if cid == 3:
        return make_workload("c3", 64, [8192] * 32, "branch4d8", [64] * 32, 300000, seed,
                             latent_std=0.5, rope_std=1.0, **kw)
    if cid == 4:
        return make_workload("c4", 16, [200000] * 4, "uniform", [32] * 4, 1 << 20, seed, **kw)
    if cid == 5:
        lo, hi = math.log(128.0), math.log(131072.0)
        P = [int(math.floor(math.exp(lo + (hi - lo) * float(torch.rand((1,), generator=g)))))
             for _ in range(64)]
        n = [int(torch.randint(8, 65, (1,), generator=g)) for _ in range(64)]
        rules = ["chain" if b % 2 == 0 else "uniform" for b in range(64)]
        return make_workload("c5", 64, P, rules, n, 1 << 22, seed, **kw)
    raise ValueError(cid)


def redraw(w: Workload, seed: int) -> Workload:
    """New contents with the shapes of ``w``: the same batch, heads, pool
    size, prefix lengths and tree sizes (so a CUDA graph captured on ``w``'s
    buffers replays on it), with new tree parents drawn by the same rules,
    new slots and new values, from ``seed``."""
    m = w.meta
    return make_workload(w.name, w.heads, w.prefix_lens, m["rules"], w.tree_sizes, w.num_slots,
                         seed, latent_std=m.get("latent_std", 1.0), rope_std=m.get("rope_std", 1.0),
                         sm_scale=w.sm_scale, kv_layout=m.get("kv_layout", "shuffled"))


def _map_rows(w: Workload, q_fn, row_fn) -> Workload:
    """A copy of ``w`` whose q, pool rows and draft rows are replaced by
    q_fn(q) and row_fn(rows), computed in float32 and rounded to bf16."""
    import dataclasses
    q = q_fn(w.q.float()).to(torch.bfloat16)
    return dataclasses.replace(w, q=q, pool_rows=row_fn(w.pool_rows.float()).to(torch.bfloat16),
                               draft_kv=row_fn(w.draft_kv.float()).to(torch.bfloat16),
                               meta=dict(w.meta))


STRESS_KINDS = ("peaked", "cancel", "huge_v")


def stress(w: Workload, kind: str) -> Workload:
    """Input transforms that push the arithmetic of a verify kernel to the
    edges of what bf16 inputs allow. Every factor is a power of two, so the
    transformed values are exact in bf16.

    peaked  every query value x8: scaled scores spread over tens of log2
            units, so the softmax is dominated by a few keys per row.
    cancel  key latent dims 256..511 copy dims 0..255; query dims 0..255
            x64 and dims 256..511 their negation; query rope dims x4. The
            latent dot product is exactly zero, but its two halves are
            large (hundreds of log2 units once scaled) and of opposite
            sign, so any kernel that rounds per-half partial scores loses
            the (rope-only, moderately peaked) score.
    huge_v  key latent dims x2^17 and query latent dims x2^-17: the scores
            are those of ``w``, while the values (latent dims) reach
            several times 2^17, beyond the largest finite fp16 number.
    """
    if kind == "peaked":
        return _map_rows(w, lambda q: q * 8.0, lambda r: r)

    if kind == "cancel":
        def qf(q):
            q = q.clone()
            q[..., :256] *= 64.0
            q[..., 256:512] = -q[..., :256]
            q[..., D_LATENT:] *= 4.0
            return q

        def rf(r):
            r = r.clone()
            r[:, 256:512] = r[:, :256]
            return r
        return _map_rows(w, qf, rf)

    if kind == "huge_v":
        def qf(q):
            q = q.clone()
            q[..., :D_LATENT] *= 2.0 ** -17
            return q

        def rf(r):
            r = r.clone()
            r[:, :D_LATENT] *= 2.0 ** 17
            return r
        return _map_rows(w, qf, rf)
    raise ValueError(kind)


def small(seed=0, heads=8, batch=3, prefix=(5, 40, 130), tree=(4, 9, 17), rule="uniform",
          num_slots=2048, **kw) -> Workload:
    """A small ragged workload for quick parity cases."""
    return make_workload("small", heads, list(prefix[:batch]), rule, list(tree[:batch]),
                         num_slots, seed, **kw)
