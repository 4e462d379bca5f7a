"""DeepSeek-V4 hybrid compressed-attention decode step on one GB300 (sm_103a).

Thin Python binding of libdsv4.so (include/dsv4.h).  The functions below take torch CUDA tensors,
fill the C parameter structs and call the library on the current torch stream; every step of the
decode path runs in the library's CUDA kernels.  There is no CPU fallback: the import fails if
the library is not built.
"""
from __future__ import annotations

import torch

from . import _abi
from ._abi import BF16, F32, FP8_DS_MLA, I8_ROWSCALE, MXFP4, Dsv4Error  # noqa: F401

_lib = _abi.load()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def dsv4_kv_insert(kv_new, kv_dtype, slot_mapping, cache, cache_dtype, page_size, positions=None, cos_sin=None,
                   stream=None, after_independent=False):
    """Writes kv_new[T, 576] into the paged SWA cache at slot_mapping[T] (int64, -1 skips).
    after_independent: see include/dsv4.h (the kernel before it on the stream touches nothing this call does)."""
    T = slot_mapping.shape[0]
    p = _abi.make(_abi.KvInsertParams, kv_new=_ptr(kv_new), kv_dtype=kv_dtype, slot_mapping=_ptr(slot_mapping),
                  cache=_ptr(cache), cache_dtype=cache_dtype, T=T, page_size=page_size,
                  num_pages=cache.shape[0], positions=_ptr(positions), cos_sin=_ptr(cos_sin),
                  max_pos=0 if cos_sin is None else cos_sin.shape[0], after_independent=int(after_independent))
    _abi.check("dsv4_kv_insert", _lib.dsv4_kv_insert(p, _stream(stream)))


def dsv4_qnorm_rope_kv_insert(q, q_out, act_dtype, kv_new, slot_mapping, cache, cache_dtype, page_size, positions,
                              cos_sin, q_norm_weight=None, eps=1e-6, apply_q_norm=True, apply_q_rope=True,
                              apply_kv_rope=True, stream=None, after_independent=False):
    """Per-head RMSNorm + GPT-J RoPE of q[T, H, 576] into q_out[T, H_pad, 576] (heads >= H zero) and the
    kv rows' RoPE + store into the paged SWA cache, in one launch (see include/dsv4.h)."""
    T, H, _ = q.shape
    p = _abi.make(_abi.QnormRopeKvInsertParams, q=_ptr(q), q_out=_ptr(q_out), H=H, H_pad=q_out.shape[1],
                  q_norm_weight=_ptr(q_norm_weight), apply_q_norm=int(apply_q_norm), apply_q_rope=int(apply_q_rope),
                  eps=eps, kv_new=_ptr(kv_new), slot_mapping=_ptr(slot_mapping), cache=_ptr(cache),
                  cache_dtype=cache_dtype, page_size=page_size, num_pages=cache.shape[0],
                  apply_kv_rope=int(apply_kv_rope), act_dtype=act_dtype, T=T, positions=_ptr(positions),
                  cos_sin=_ptr(cos_sin), max_pos=0 if cos_sin is None else cos_sin.shape[0],
                  after_independent=int(after_independent))
    _abi.check("dsv4_qnorm_rope_kv_insert", _lib.dsv4_qnorm_rope_kv_insert(p, _stream(stream)))


def dsv4_padded_num_q_heads(H, cache_dtype) -> int:
    """Query heads the attention's q and output buffers hold for H heads with this cache dtype."""
    n = int(_lib.dsv4_padded_num_q_heads(int(H), int(cache_dtype)))
    if n < 0:
        raise ValueError(f"no padded head count for H={H}, cache dtype {cache_dtype}")
    return n


def dsv4_compress_update(kv_score, positions, q_per_seq, ratio, coff, state, ape, norm_weight, eps, cos_sin,
                         main_cache, cache_dtype, block_table, page_size, stream=None, after_independent=False,
                         wk=None, ik_norm_weight=None, ik_eps=1e-6, ik_cache=None, ik_dtype=BF16,
                         ik_block_table=None):
    """Compressor state store + fold of the new tokens, and (with wk) the index key of every new entry
    into the indexer cache (see include/dsv4.h)."""
    T = positions.shape[0]
    p = _abi.make(_abi.CompressUpdateParams, kv_score=_ptr(kv_score), positions=_ptr(positions), T=T,
                  B=T // q_per_seq, q_per_seq=q_per_seq, ratio=ratio, coff=coff, state=_ptr(state), ape=_ptr(ape),
                  norm_weight=_ptr(norm_weight), eps=eps, cos_sin=_ptr(cos_sin), max_pos=cos_sin.shape[0],
                  main_cache=_ptr(main_cache), cache_dtype=cache_dtype, page_size=page_size,
                  num_pages=main_cache.shape[0], block_table=_ptr(block_table),
                  max_pages_per_seq=block_table.shape[1], after_independent=int(after_independent))
    if wk is not None:
        p.wk, p.ik_norm_weight, p.ik_eps, p.ik_dim = _ptr(wk), _ptr(ik_norm_weight), ik_eps, wk.shape[0]
        p.ik_cache, p.ik_dtype, p.ik_num_pages = _ptr(ik_cache), ik_dtype, ik_cache.shape[0]
        p.ik_block_table, p.ik_max_pages = _ptr(ik_block_table), ik_block_table.shape[1]
    _abi.check("dsv4_compress_update", _lib.dsv4_compress_update(p, _stream(stream)))


def indexer_topk_params(q, q_dtype, weights, k_cache, k_dtype, block_table, positions, q_per_seq, ratio, topk,
                        page_size, max_context, topk_idx=None, topk_score=None, workspace=None, cand_blocks=None,
                        cand_block_size=0, cand_write=False):
    """Parameter struct of dsv4_indexer_topk.  cand_blocks ([T, cand_topk] int32) with cand_block_size > 0
    turns on two-level candidate filtering: read by a consumer, written by the source (cand_write)."""
    T, n_heads, head_dim = q.shape
    return _abi.make(_abi.IndexerTopkParams, q=_ptr(q), q_dtype=q_dtype, weights=_ptr(weights),
                     k_cache=_ptr(k_cache), k_dtype=k_dtype, num_pages=k_cache.shape[0],
                     block_table=_ptr(block_table), max_pages_per_seq=block_table.shape[1],
                     positions=_ptr(positions), T=T, B=T // q_per_seq, q_per_seq=q_per_seq, ratio=ratio,
                     n_heads=n_heads, head_dim=head_dim, topk=topk, page_size=page_size, max_context=max_context,
                     topk_idx=_ptr(topk_idx), topk_score=_ptr(topk_score), workspace=_ptr(workspace),
                     workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size(),
                     cand_blocks=_ptr(cand_blocks), cand_block_size=cand_block_size if cand_blocks is not None else 0,
                     cand_topk=0 if cand_blocks is None else cand_blocks.shape[1], cand_write=int(cand_write))


def dsv4_indexer_topk_workspace_bytes(params) -> int:
    return int(_lib.dsv4_indexer_topk_workspace_bytes(params))


def dsv4_indexer_topk(params, stream=None):
    """Lightning-Indexer scores + per-query top-k into params.topk_idx (see include/dsv4.h)."""
    _abi.check("dsv4_indexer_topk", _lib.dsv4_indexer_topk(params, _stream(stream)))


def sparse_mla_params(q, q_dtype, positions, q_per_seq, swa_cache, swa_block_table, main_cache, main_block_table,
                      cache_dtype, page_size, ratio, window, topk_idx, sink, softmax_scale, out, out_dtype, lse,
                      max_context, workspace=None):
    T, H, _ = q.shape
    return _abi.make(_abi.SparseMlaDecodeParams, q=_ptr(q), q_dtype=q_dtype, T=T, B=T // q_per_seq,
                     q_per_seq=q_per_seq, H=H, positions=_ptr(positions), swa_cache=_ptr(swa_cache),
                     swa_block_table=_ptr(swa_block_table), swa_max_pages=swa_block_table.shape[1],
                     swa_num_pages=swa_cache.shape[0], main_cache=_ptr(main_cache),
                     main_block_table=_ptr(main_block_table),
                     main_max_pages=0 if main_block_table is None else main_block_table.shape[1],
                     main_num_pages=0 if main_cache is None else main_cache.shape[0], cache_dtype=cache_dtype,
                     page_size=page_size, ratio=ratio, window=window, topk_idx=_ptr(topk_idx),
                     topk=0 if topk_idx is None else topk_idx.shape[1], sink=_ptr(sink),
                     softmax_scale=softmax_scale, out=_ptr(out), out_dtype=out_dtype, lse=_ptr(lse),
                     max_context=max_context, workspace=_ptr(workspace),
                     workspace_bytes=0 if workspace is None else workspace.numel() * workspace.element_size())


def dsv4_sparse_mla_decode_workspace_bytes(params) -> int:
    return int(_lib.dsv4_sparse_mla_decode_workspace_bytes(params))


def dsv4_sparse_mla_decode(params, stream=None):
    """Shared-KV sparse MLA decode attention into params.out (see include/dsv4.h)."""
    _abi.check("dsv4_sparse_mla_decode", _lib.dsv4_sparse_mla_decode(params, _stream(stream)))


def dsv4_kernel_launches() -> int:
    """Kernels the library has enqueued (or recorded into a graph) since it was loaded."""
    return int(_lib.dsv4_kernel_launches())


def dsv4_read_device_flags() -> int:
    """Synchronises and returns (and clears) the kernels' range-check flags."""
    f = _abi.u32(0)
    st = _lib.dsv4_read_device_flags(f)
    if st not in (_abi.OK, _abi.ERR_BOUNDS, _abi.ERR_TIMEOUT):
        _abi.check("dsv4_read_device_flags", st)
    return int(f.value)
