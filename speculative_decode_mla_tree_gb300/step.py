"""Device buffers for one batch shape and the four library calls of one
verify step: draft-KV scatter, KV index marshaling, tree-mask packing and
tree-verify attention. Buffers are allocated once, so a step can be
replayed or captured into a CUDA graph; refilling the input buffers in place
(``load``) gives a new step of the same shape."""
from __future__ import annotations

import torch

from . import abi


class VerifyStep:
    def __init__(self, w, device="cuda", max_splits=0, path=abi.PATH_AUTO, pool=None,
                 mask_bits=False, fused=False):
        """mask_bits: pack the tree mask in its bit form; fused (implies
        mask_bits): scatter, index marshaling and mask packing as one launch
        (mla_tree_prepare)."""
        dev = torch.device(device)
        self.device = dev
        self.w = w
        self.heads = w.heads
        self.sm_scale = w.sm_scale
        self.max_splits = max_splits
        self.path = path
        self.fused = fused
        self.mask_bits = mask_bits or fused
        B, T = w.batch, w.total_q
        L = [p + n for p, n in zip(w.prefix_lens, w.tree_sizes)]
        # resident latent-KV pool (before the draft rows are scattered in)
        self.pool = w.dense_pool(dev) if pool is None else pool
        # per-step inputs
        self.q = torch.empty_like(w.q, device=dev)
        self.draft_kv = torch.empty_like(w.draft_kv, device=dev)
        self.out_cache_loc = torch.empty_like(w.out_cache_loc, device=dev)
        self.prefix_indices = torch.empty_like(w.prefix_indices, device=dev)
        self.prefix_indptr = torch.empty_like(w.prefix_indptr, device=dev)
        self.qo_indptr = torch.empty_like(w.qo_indptr, device=dev)
        self.parents = torch.empty_like(w.parents, device=dev)
        # intermediates and outputs
        self.kv_indices = torch.empty(sum(L), dtype=torch.int32, device=dev)
        self.kv_indptr = torch.empty(B + 1, dtype=torch.int32, device=dev)
        self.mask_indptr = torch.empty(B + 1, dtype=torch.int64, device=dev)
        self.mask = torch.empty(sum(n * l for n, l in zip(w.tree_sizes, L)), dtype=torch.uint8, device=dev)
        # the bit form of the mask (rows of ceil(L/32) uint32 words, held as int32)
        self.mask_word_indptr = torch.empty(B + 1, dtype=torch.int64, device=dev)
        self.mask_words = torch.empty(sum(n * ((l + 31) // 32) for n, l in zip(w.tree_sizes, L)),
                                      dtype=torch.int32, device=dev)
        self.out = torch.empty((T, w.heads, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((T, w.heads), dtype=torch.float32, device=dev)
        nbytes = abi.mla_tree_verify_workspace_bytes(B, T, w.heads, max_splits)
        self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.load(w)

    def inputs(self):
        """(device buffer, host tensor) pairs of the per-step inputs."""
        w = self.w
        return [(self.q, w.q), (self.draft_kv, w.draft_kv), (self.out_cache_loc, w.out_cache_loc),
                (self.prefix_indices, w.prefix_indices), (self.prefix_indptr, w.prefix_indptr),
                (self.qo_indptr, w.qo_indptr), (self.parents, w.parents)]

    def load(self, w=None):
        if w is not None:
            self.w = w
        for d, h in self.inputs():
            d.copy_(h, non_blocking=False)

    def run(self, stream=None):
        if self.fused:
            self.prepare(stream)
            self.verify(stream)
            return
        abi.mla_tree_draft_kv_scatter(self.draft_kv, self.out_cache_loc, self.pool, self.status, stream)
        abi.mla_tree_kv_indices_build(self.prefix_indices, self.prefix_indptr, self.out_cache_loc,
                                      self.qo_indptr, self.kv_indices, self.kv_indptr, self.status, stream)
        self.pack_mask(stream)
        self.verify(stream)

    def prepare(self, stream=None):
        abi.mla_tree_prepare(self.draft_kv, self.out_cache_loc, self.prefix_indices, self.prefix_indptr,
                             self.qo_indptr, self.parents, self.pool, self.kv_indices, self.kv_indptr,
                             self.mask_word_indptr, self.mask_words, self.status, stream)

    def pack_mask(self, stream=None):
        if self.mask_bits:
            abi.tree_mask_pack_bits(self.parents, self.qo_indptr, self.kv_indptr, self.mask_word_indptr,
                                    self.mask_words, self.status, stream)
        else:
            abi.tree_mask_pack(self.parents, self.qo_indptr, self.kv_indptr, self.mask_indptr,
                               self.mask, self.status, stream)

    def verify(self, stream=None):
        if self.mask_bits:
            abi.mla_tree_verify_bits(self.q, self.pool, self.kv_indices, self.kv_indptr, self.qo_indptr,
                                     self.mask_words, self.mask_word_indptr, self.sm_scale, self.out,
                                     self.lse, self.workspace, self.max_splits, self.path, self.status,
                                     stream)
            return
        abi.mla_tree_verify(self.q, self.pool, self.kv_indices, self.kv_indptr, self.qo_indptr,
                            self.mask, self.mask_indptr, self.sm_scale, self.out, self.lse,
                            self.workspace, self.max_splits, self.path, self.status, stream)
