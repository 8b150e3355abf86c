"""Device buffers for one batch shape and the four library calls of one
verify step: draft-KV scatter, KV index marshaling, tree-mask packing and
tree-verify attention. Buffers are allocated once, so a step can be
replayed or captured into a CUDA graph; refilling the input buffers in place
(``load``) gives a new step of the same shape."""
from __future__ import annotations

import torch

from . import abi


def _carve(dev, specs, buf=None):
    """One uint8 buffer holding tensors of the given (shape, dtype), each at a
    256-byte aligned offset; returns (buffer, views)."""
    offs, off = [], 0
    for shape, dtype in specs:
        n = 1
        for d in shape:
            n *= int(d)
        offs.append((off, n, shape, dtype))
        off += -(-n * torch.empty((), dtype=dtype).element_size() // 256) * 256
    if buf is None:
        buf = torch.empty(max(off, 256), dtype=torch.uint8, device=dev)
    views = []
    for o, n, shape, dtype in offs:
        es = torch.empty((), dtype=dtype).element_size()
        views.append(buf[o:o + n * es].view(dtype).view(shape))
    return buf, views


class VerifyStep:
    def __init__(self, w, device="cuda", max_splits=0, path=abi.PATH_AUTO, pool=None,
                 mask_bits=False, fused=False, skip_prefix=False):
        """mask_bits: pack the tree mask in its bit form; fused (implies
        mask_bits): scatter, index marshaling and mask packing as one launch
        (mla_tree_prepare); skip_prefix: verify with the prefix-skip switch
        (the prefix columns of the mask are not read)."""
        self.skip_prefix = bool(skip_prefix)
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
        # per-step inputs: views into one device buffer, so that a step's
        # inputs arrive with one host-to-device copy (see packed_inputs)
        self._in_spec = [("q", w.q), ("draft_kv", w.draft_kv), ("out_cache_loc", w.out_cache_loc),
                         ("prefix_indices", w.prefix_indices), ("prefix_indptr", w.prefix_indptr),
                         ("qo_indptr", w.qo_indptr), ("parents", w.parents)]
        self.inbuf, views = _carve(dev, [(h.shape, h.dtype) for _, h in self._in_spec])
        for (name, _), v in zip(self._in_spec, views):
            setattr(self, name, v)
        # intermediates and outputs
        self.kv_indices = torch.empty(sum(L), dtype=torch.int32, device=dev)
        self.kv_indptr = torch.empty(B + 1, dtype=torch.int32, device=dev)
        self.mask_indptr = torch.empty(B + 1, dtype=torch.int64, device=dev)
        self.mask = torch.empty(sum(n * l for n, l in zip(w.tree_sizes, L)), dtype=torch.uint8, device=dev)
        # the bit form of the mask (rows of ceil(L/32) uint32 words, held as int32)
        self.mask_word_indptr = torch.empty(B + 1, dtype=torch.int64, device=dev)
        self.mask_words = torch.empty(sum(n * ((l + 31) // 32) for n, l in zip(w.tree_sizes, L)),
                                      dtype=torch.int32, device=dev)
        # outputs: views into one device buffer (one device-to-host copy)
        self.outbuf, (self.out, self.lse) = _carve(dev, [((T, w.heads, 512), torch.bfloat16),
                                                         ((T, w.heads), torch.float32)])
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

    def packed_inputs(self, pin=True):
        """The per-step inputs packed in host memory with the layout of
        ``inbuf``: ``inbuf.copy_(packed, non_blocking=True)`` loads a step."""
        host = torch.zeros(self.inbuf.numel(), dtype=torch.uint8)
        _, views = _carve(torch.device("cpu"), [(h.shape, h.dtype) for _, h in self._in_spec], host)
        for v, (_, h) in zip(views, self._in_spec):
            v.copy_(h)
        return host.pin_memory() if pin else host

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
        if self.skip_prefix:
            flags = abi.MASK_SKIP_PREFIX | (abi.MASK_BITS if self.mask_bits else 0)
            mask, mptr = ((self.mask_words, self.mask_word_indptr) if self.mask_bits
                          else (self.mask, self.mask_indptr))
            abi.mla_tree_verify_masked(self.q, self.pool, self.kv_indices, self.kv_indptr,
                                       self.qo_indptr, mask, mptr, flags, self.sm_scale, self.out,
                                       self.lse, self.workspace, self.max_splits, self.path,
                                       self.status, stream)
            return
        if self.mask_bits:
            abi.mla_tree_verify_bits(self.q, self.pool, self.kv_indices, self.kv_indptr, self.qo_indptr,
                                     self.mask_words, self.mask_word_indptr, self.sm_scale, self.out,
                                     self.lse, self.workspace, self.max_splits, self.path, self.status,
                                     stream)
            return
        abi.mla_tree_verify(self.q, self.pool, self.kv_indices, self.kv_indptr, self.qo_indptr,
                            self.mask, self.mask_indptr, self.sm_scale, self.out, self.lse,
                            self.workspace, self.max_splits, self.path, self.status, stream)
