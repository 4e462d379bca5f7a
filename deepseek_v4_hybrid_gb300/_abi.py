"""ctypes mirror of include/dsv4.h and the loader of the in-tree libdsv4.so.

Argument marshalling only: every step of the decode path runs in the library's CUDA kernels.
Importing this module fails loudly if the library has not been built.
"""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libdsv4.so")

F32, BF16, FP8_DS_MLA, I8_ROWSCALE, MXFP4 = 0, 1, 2, 3, 4
OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_BOUNDS, ERR_TIMEOUT = 0, -1, -2, -3, -4, -5
LATENT_DIM, VALUE_DIM, ROPE_DIM, FP8_DS_MLA_BYTES = 576, 512, 64, 656
ABI_VERSION = 3

vp, i32, i64, u32, f32 = C.c_void_p, C.c_int32, C.c_int64, C.c_uint32, C.c_float


class KvInsertParams(C.Structure):
    _fields_ = [("struct_size", u32), ("kv_new", vp), ("kv_dtype", i32), ("slot_mapping", vp), ("cache", vp),
                ("cache_dtype", i32), ("T", i32), ("page_size", i32), ("num_pages", i64), ("positions", vp),
                ("cos_sin", vp), ("max_pos", i32), ("after_independent", i32)]


class QnormRopeKvInsertParams(C.Structure):
    _fields_ = [("struct_size", u32), ("q", vp), ("q_out", vp), ("H", i32), ("H_pad", i32), ("q_norm_weight", vp),
                ("apply_q_norm", i32), ("apply_q_rope", i32), ("eps", f32), ("kv_new", vp), ("slot_mapping", vp),
                ("cache", vp), ("cache_dtype", i32), ("page_size", i32), ("num_pages", i64),
                ("apply_kv_rope", i32), ("act_dtype", i32), ("T", i32), ("positions", vp), ("cos_sin", vp),
                ("max_pos", i32), ("after_independent", i32)]


class CompressUpdateParams(C.Structure):
    _fields_ = [("struct_size", u32), ("kv_score", vp), ("positions", vp), ("T", i32), ("B", i32),
                ("q_per_seq", i32), ("ratio", i32), ("coff", i32), ("state", vp), ("ape", vp),
                ("norm_weight", vp), ("eps", f32), ("cos_sin", vp), ("max_pos", i32), ("main_cache", vp),
                ("cache_dtype", i32), ("page_size", i32), ("num_pages", i64), ("block_table", vp),
                ("max_pages_per_seq", i32), ("after_independent", i32), ("wk", vp), ("ik_norm_weight", vp),
                ("ik_eps", f32), ("ik_dim", i32), ("ik_cache", vp), ("ik_dtype", i32), ("ik_num_pages", i64),
                ("ik_block_table", vp), ("ik_max_pages", i32)]


class IndexerTopkParams(C.Structure):
    _fields_ = [("struct_size", u32), ("q", vp), ("q_dtype", i32), ("weights", vp), ("k_cache", vp),
                ("k_dtype", i32), ("num_pages", i64), ("block_table", vp), ("max_pages_per_seq", i32),
                ("positions", vp), ("T", i32), ("B", i32), ("q_per_seq", i32), ("ratio", i32),
                ("n_heads", i32), ("head_dim", i32), ("topk", i32), ("page_size", i32), ("max_context", i32),
                ("topk_idx", vp), ("topk_score", vp), ("workspace", vp), ("workspace_bytes", C.c_size_t),
                ("workspace_zeroed", i32), ("cand_blocks", vp), ("cand_block_size", i32), ("cand_topk", i32),
                ("cand_write", i32)]


class SparseMlaDecodeParams(C.Structure):
    _fields_ = [("struct_size", u32), ("q", vp), ("q_dtype", i32), ("T", i32), ("B", i32), ("q_per_seq", i32),
                ("H", i32), ("positions", vp), ("swa_cache", vp), ("swa_block_table", vp), ("swa_max_pages", i32),
                ("swa_num_pages", i64), ("main_cache", vp), ("main_block_table", vp), ("main_max_pages", i32),
                ("main_num_pages", i64), ("cache_dtype", i32), ("page_size", i32), ("ratio", i32),
                ("window", i32), ("topk_idx", vp), ("topk", i32), ("sink", vp), ("softmax_scale", f32),
                ("out", vp), ("out_dtype", i32), ("lse", vp), ("max_context", i32), ("workspace", vp),
                ("workspace_bytes", C.c_size_t)]


EXPORTS = ["dsv4_kv_insert", "dsv4_compress_update", "dsv4_indexer_topk_workspace_bytes", "dsv4_indexer_topk",
           "dsv4_sparse_mla_decode_workspace_bytes", "dsv4_sparse_mla_decode", "dsv4_abi_version",
           "dsv4_status_string", "dsv4_last_cuda_error", "dsv4_read_device_flags", "dsv4_indexer_topk_noalloc",
           "dsv4_qnorm_rope_kv_insert", "dsv4_padded_num_q_heads", "dsv4_kernel_launches"]

# bytes of the scratch array built into the library for dsv4_indexer_topk_noalloc
NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024

_lib = None


def load(path: str = LIB_PATH) -> C.CDLL:
    """Loads libdsv4.so (raises if it is missing: there is no fallback path)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libdsv4.so is not built ({path}); run __graft_entry__.build() or "
                           "python -m deepseek_v4_hybrid_gb300.build")
    lib = C.CDLL(path)
    for name, st in (("dsv4_kv_insert", KvInsertParams), ("dsv4_compress_update", CompressUpdateParams),
                     ("dsv4_qnorm_rope_kv_insert", QnormRopeKvInsertParams),
                     ("dsv4_indexer_topk", IndexerTopkParams), ("dsv4_sparse_mla_decode", SparseMlaDecodeParams),
                     ("dsv4_indexer_topk_noalloc", IndexerTopkParams)):
        fn = getattr(lib, name)
        fn.argtypes = [C.POINTER(st), vp]
        fn.restype = C.c_int
    for name, st in (("dsv4_indexer_topk_workspace_bytes", IndexerTopkParams),
                     ("dsv4_sparse_mla_decode_workspace_bytes", SparseMlaDecodeParams)):
        fn = getattr(lib, name)
        fn.argtypes = [C.POINTER(st)]
        fn.restype = C.c_size_t
    lib.dsv4_padded_num_q_heads.argtypes = [C.c_int, C.c_int]
    lib.dsv4_padded_num_q_heads.restype = C.c_int
    lib.dsv4_abi_version.restype = C.c_int
    lib.dsv4_status_string.argtypes = [C.c_int]
    lib.dsv4_status_string.restype = C.c_char_p
    lib.dsv4_last_cuda_error.restype = C.c_int
    lib.dsv4_kernel_launches.argtypes = []
    lib.dsv4_kernel_launches.restype = C.c_uint64
    lib.dsv4_read_device_flags.argtypes = [C.POINTER(u32)]
    lib.dsv4_read_device_flags.restype = C.c_int
    if lib.dsv4_abi_version() != ABI_VERSION:
        raise RuntimeError("libdsv4.so ABI version mismatch")
    _lib = lib
    return lib


def make(struct_type, **fields):
    s = struct_type()
    s.struct_size = C.sizeof(struct_type)
    for k, v in fields.items():
        setattr(s, k, v)
    return s


class Dsv4Error(RuntimeError):
    def __init__(self, call: str, status: int):
        lib = load()
        msg = lib.dsv4_status_string(status).decode()
        if status == ERR_CUDA:
            msg += f" (cudaError {lib.dsv4_last_cuda_error()})"
        super().__init__(f"{call}: {msg}")
        self.status = status


def check(call: str, status: int) -> None:
    if status != OK:
        raise Dsv4Error(call, status)
