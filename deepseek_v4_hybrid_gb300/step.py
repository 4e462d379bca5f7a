"""Device-resident decode step: owns the device tensors of one workload and issues the four
library calls (insert -> compress -> indexer/top-k -> attention) on one stream.

Memory comes from torch; every computation is a libdsv4 kernel.  The per-call parameter structs
are built once, so a step is four C calls with no host synchronisation (graph-capturable).
"""
from __future__ import annotations

import numpy as np
import torch

from . import (BF16, F32, dsv4_compress_update, dsv4_indexer_topk, dsv4_indexer_topk_workspace_bytes,
               dsv4_kv_insert, dsv4_padded_num_q_heads, dsv4_qnorm_rope_kv_insert, dsv4_sparse_mla_decode,
               dsv4_sparse_mla_decode_workspace_bytes, indexer_topk_params, sparse_mla_params, _abi)

PAGE = 64
WINDOW = 128


def to_device(a, device):
    """numpy array -> device tensor with the same bytes (uint16 bf16 bits become torch.bfloat16)."""
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def _ws(nbytes, device):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


class DeviceStep:
    # per-step inputs (copied host -> device every step in the end-to-end measurement)
    STEP_INPUTS = ("q", "kv_new", "slot_mapping", "positions", "kv_score", "q_idx", "w_idx")

    # caches, block tables and weights: what the steps of one prefill share (see PrefillRunner)
    SHARED = ("swa_cache", "swa_bt", "cos_sin", "q_norm_w", "state", "ape", "norm_w", "main_cache", "main_bt",
              "wk", "ik_norm_w", "idx_cache", "idx_bt")

    def __init__(self, st, device="cuda", topk_override=None, shared=None):
        """shared: device tensors (by the names in SHARED) to use instead of uploading st's."""
        cfg = st.cfg
        self.cfg, self.device = cfg, device
        dev = lambda a: to_device(a, device)  # noqa: E731
        shared = shared or {}
        keep = lambda name, a: shared[name] if name in shared else dev(a)  # noqa: E731
        self.positions = dev(st.positions.astype(np.int32))
        self.kv_new = dev(st.kv_new)
        self.slot_mapping = dev(st.slot_mapping.astype(np.int64))
        self.swa_cache = keep("swa_cache", st.swa_cache)
        self.swa_bt = keep("swa_bt", st.swa_bt)
        self.max_context = int(st.ctx_len.max())
        T, H = cfg.T, cfg.H
        # with query preparation, the fused insert turns the raw queries q_in [T, H, 576] into the
        # attention's q [T, H_pad, 576]; the sink of the padding heads is -inf
        self.q_prep = bool(getattr(cfg, "q_prep", False))
        self.H_pad = dsv4_padded_num_q_heads(H, cfg.cache_dtype) if self.q_prep else H
        self.cos_sin = keep("cos_sin", st.cos_sin)
        if self.q_prep:
            self.q_in = dev(st.q)
            self.q = torch.empty((T, self.H_pad, 576), dtype=self.q_in.dtype, device=device)
            self.q_norm_w = keep("q_norm_w", st.q_norm_w)
            sink = np.full(self.H_pad, -np.inf, np.float32)
            sink[:H] = st.sink
            self.sink = dev(sink)
        else:
            self.q = dev(st.q)
            self.sink = dev(st.sink)
        odt = torch.float32 if cfg.out_dtype == F32 else torch.bfloat16
        self.out = torch.empty((T, self.H_pad, 512), dtype=odt, device=device)
        self.lse = torch.empty((T, self.H_pad), dtype=torch.float32, device=device)
        self.has_compress = cfg.ratio > 0
        self.has_indexer = cfg.ratio > 0 and cfg.topk > 0
        self.kv_score = self.state = self.ape = self.norm_w = None
        self.main_cache = self.main_bt = None
        self.q_idx = self.w_idx = None
        if self.has_compress:
            self.kv_score = dev(st.kv_score)
            self.state = keep("state", st.state)
            self.ape = keep("ape", st.ape)
            self.norm_w = keep("norm_w", st.norm_w)
            self.main_cache = keep("main_cache", st.main_cache)
            self.main_bt = keep("main_bt", st.main_bt)
        self.topk_idx = None
        self.ik_store = self.has_indexer and bool(getattr(cfg, "ik_store", False)) and st.wk is not None
        if self.ik_store:
            self.wk = keep("wk", st.wk)
            self.ik_norm_w = keep("ik_norm_w", st.ik_norm_w)
        if self.has_indexer:
            self.idx_cache = keep("idx_cache", st.idx_cache)
            self.idx_bt = keep("idx_bt", st.idx_bt)
            self.q_idx = dev(st.q_idx)
            self.w_idx = dev(st.w_idx)
            self.topk_idx = torch.empty((T, cfg.topk), dtype=torch.int32, device=device)
            self.topk_score = torch.empty((T, cfg.topk), dtype=torch.float32, device=device)
            # two-level candidate filtering: a consumer reads another layer's blocks, the source writes its own
            self.cand_blocks = None
            self.cand_write = bool(getattr(cfg, "cand_write", False))
            if getattr(cfg, "cand_block", 0):
                if self.cand_write:
                    self.cand_blocks = torch.full((T, cfg.cand_topk), -7, dtype=torch.int32, device=device)
                else:
                    self.cand_blocks = dev(st.cand_in.astype(np.int32))
            self.ix_params = indexer_topk_params(self.q_idx, cfg.act_dtype, self.w_idx, self.idx_cache,
                                                 cfg.idx_dtype, self.idx_bt, self.positions, cfg.q_per_seq,
                                                 cfg.ratio, cfg.topk, PAGE, self.max_context, self.topk_idx,
                                                 self.topk_score, cand_blocks=self.cand_blocks,
                                                 cand_block_size=getattr(cfg, "cand_block", 0),
                                                 cand_write=self.cand_write)
            # zero-filled once: every call leaves its histograms and counters cleared, so no call needs a memset
            self.ix_ws = torch.zeros(max(int(dsv4_indexer_topk_workspace_bytes(self.ix_params)), 256),
                                     dtype=torch.uint8, device=device)
            self.ix_params.workspace = self.ix_ws.data_ptr()
            self.ix_params.workspace_bytes = self.ix_ws.numel()
            self.ix_params.workspace_zeroed = 1
        attn_topk = self.topk_idx
        if topk_override is not None:
            self.given_topk = dev(topk_override.astype(np.int32))
            attn_topk = self.given_topk
        self.at_params = sparse_mla_params(self.q, cfg.act_dtype, self.positions, cfg.q_per_seq, self.swa_cache,
                                           self.swa_bt, self.main_cache, self.main_bt, cfg.cache_dtype, PAGE,
                                           cfg.ratio, WINDOW, attn_topk if cfg.topk > 0 else None, self.sink,
                                           st.softmax_scale, self.out, cfg.out_dtype, self.lse, self.max_context)
        self.at_ws = _ws(dsv4_sparse_mla_decode_workspace_bytes(self.at_params), device)
        self.at_params.workspace = self.at_ws.data_ptr()
        self.at_params.workspace_bytes = self.at_ws.numel()
        self.eps = st.eps

    def insert(self, stream=None, after_independent=False):
        if self.q_prep:
            dsv4_qnorm_rope_kv_insert(self.q_in, self.q, self.cfg.act_dtype, self.kv_new, self.slot_mapping,
                                      self.swa_cache, self.cfg.cache_dtype, PAGE, self.positions, self.cos_sin,
                                      q_norm_weight=self.q_norm_w, eps=self.eps, stream=stream,
                                      after_independent=after_independent)
        else:
            dsv4_kv_insert(self.kv_new, self.cfg.act_dtype, self.slot_mapping, self.swa_cache, self.cfg.cache_dtype,
                           PAGE, stream=stream, after_independent=after_independent)

    def compress(self, stream=None, after_independent=False):
        if self.has_compress:
            cfg = self.cfg
            ik = {}
            if self.ik_store:
                ik = dict(wk=self.wk, ik_norm_weight=self.ik_norm_w, ik_eps=self.eps, ik_cache=self.idx_cache,
                          ik_dtype=cfg.idx_dtype, ik_block_table=self.idx_bt)
            dsv4_compress_update(self.kv_score, self.positions, cfg.q_per_seq, cfg.ratio, cfg.coff, self.state,
                                 self.ape, self.norm_w, self.eps, self.cos_sin, self.main_cache, cfg.cache_dtype,
                                 self.main_bt, PAGE, stream=stream, after_independent=after_independent, **ik)

    def indexer(self, stream=None):
        if self.has_indexer:
            dsv4_indexer_topk(self.ix_params, stream=stream)

    def attention(self, stream=None):
        dsv4_sparse_mla_decode(self.at_params, stream=stream)

    def run(self, stream=None):
        """One decode step.
        With an indexer whose keys the compressor writes: compress (fold + index keys) -> indexer +
        top-k (scores the keys written just before) -> insert -> attention.  The indexer reads none of
        what insert writes and insert reads none of its outputs, so insert starts at once beside the
        indexer and waits for it only before exiting; attention waits for insert, whose completion
        implies the others'.
        With an indexer over given keys: indexer -> insert -> compress -> attention, insert and
        compress both starting at once beside the indexer.
        Without an indexer: compress -> insert -> attention, the insert (which touches nothing the
        compressor reads or writes) starting at once beside the compressor."""
        if self.ik_store:
            self.compress(stream)
            self.indexer(stream)
            self.insert(stream, after_independent=True)
        elif self.has_indexer:
            self.indexer(stream)
            self.insert(stream, after_independent=True)
            self.compress(stream, after_independent=True)
        elif self.has_compress:
            self.compress(stream)
            self.insert(stream, after_independent=True)
        else:
            self.insert(stream)
        self.attention(stream)

    def step_input_tensors(self):
        """The tensors a caller fills every step (the raw queries under the name "q")."""
        d = {k: getattr(self, k) for k in self.STEP_INPUTS if getattr(self, k, None) is not None}
        if self.q_prep:
            d["q"] = self.q_in
        if getattr(self, "cand_blocks", None) is not None and not self.cand_write:
            d["cand_blocks"] = self.cand_blocks  # the blocks an earlier layer published this step
        return d


class PrefillRunner:
    """Chunked prefill on the device: the decode chain over consecutive chunks of `chunk` positions of
    every sequence, from position 0 ("DeepSeek-V4 Inference on Ascend", §8 "The prefill path";
    "vllm.models.deepseek_v41.attention", DeepseekV4Attention.PREFILL_CHUNK_SIZE = 4).  One DeviceStep
    a chunk, all over one set of device caches, state ring and weights: what a chunk writes, the next
    one reads.  run() issues the chunks in order on one stream (graph-capturable)."""

    def __init__(self, pf, chunk=4, device="cuda"):
        self.spans = pf.spans(chunk)
        first = DeviceStep(pf.chunk(*self.spans[0]), device)
        shared = {k: getattr(first, k) for k in DeviceStep.SHARED if getattr(first, k, None) is not None}
        self.steps = [first] + [DeviceStep(pf.chunk(p0, n), device, shared=shared) for p0, n in self.spans[1:]]
        self.shared = shared

    def run(self, stream=None):
        for s in self.steps:
            s.run(stream)
