"""The C-ABI library loads, exports every symbol include/dsv4.h declares, its struct layouts match
the ctypes mirror, and host-side validation rejects bad arguments without touching a GPU."""
import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsv4.h")


@pytest.fixture(scope="module")
def abi():
    import __graft_entry__
    lib_path = os.path.join(ROOT, "deepseek_v4_hybrid_gb300", "_lib", "libdsv4.so")
    if not os.path.exists(lib_path):
        __graft_entry__._build_module().build()
    from deepseek_v4_hybrid_gb300 import _abi
    _abi.load()
    return _abi


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|uint64_t|const char\*)\s+(dsv4_\w+)\s*\(", text, re.M)))


def test_exports_every_declared_symbol(abi):
    names = declared_functions()
    assert len(names) == 14
    out = subprocess.run(["nm", "-D", "--defined-only", abi.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (dsv4_\w+)", out))
    assert set(names) <= exported, set(names) - exported
    assert set(abi.EXPORTS) == set(names)


def test_struct_layout_matches_header(abi, tmp_path):
    """Compile a C program that prints sizeof/offsetof of every field and compare with ctypes."""
    structs = {"dsv4_kv_insert_params": abi.KvInsertParams, "dsv4_compress_update_params": abi.CompressUpdateParams,
               "dsv4_qnorm_rope_kv_insert_params": abi.QnormRopeKvInsertParams,
               "dsv4_indexer_topk_params": abi.IndexerTopkParams,
               "dsv4_sparse_mla_decode_params": abi.SparseMlaDecodeParams}
    lines = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{HEADER}"', 'int main(void){']
    for cname, st in structs.items():
        lines.append(f'printf("{cname} %zu\\n", sizeof({cname}));')
        for f, _ in st._fields_:
            lines.append(f'printf("{cname}.{f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0;}")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", str(src), "-o", str(exe)], check=True)
    got = dict(l.rsplit(" ", 1) for l in subprocess.run([str(exe)], capture_output=True, text=True,
                                                          check=True).stdout.split("\n") if l)
    for cname, st in structs.items():
        assert int(got[cname]) == C.sizeof(st), cname
        for f, _ in st._fields_:
            assert int(got[f"{cname}.{f}"]) == getattr(st, f).offset, (cname, f)


def test_host_validation_rejects_bad_arguments(abi):
    lib = abi.load()
    p = abi.make(abi.KvInsertParams, T=1, page_size=64, kv_dtype=abi.BF16, cache_dtype=abi.BF16)
    assert lib.dsv4_kv_insert(p, None) == abi.ERR_INVALID             # null pointers
    p.struct_size = 4
    assert lib.dsv4_kv_insert(p, None) == abi.ERR_INVALID             # wrong struct size
    p = abi.make(abi.KvInsertParams, T=0, page_size=64, kv_dtype=abi.BF16, cache_dtype=abi.BF16)
    assert lib.dsv4_kv_insert(p, None) == abi.OK                      # empty batch: no-op
    p = abi.make(abi.KvInsertParams, T=1, page_size=64, kv_dtype=abi.FP8_DS_MLA, cache_dtype=abi.BF16)
    assert lib.dsv4_kv_insert(p, None) == abi.ERR_UNSUPPORTED
    p = abi.make(abi.KvInsertParams, T=2, page_size=64, kv_dtype=abi.BF16, cache_dtype=abi.BF16, kv_new=0x1001,
                 slot_mapping=0x1000, cache=0x1000)
    assert lib.dsv4_kv_insert(p, None) == abi.ERR_INVALID             # misaligned kv_new

    qp = abi.make(abi.QnormRopeKvInsertParams, T=2, H=64, H_pad=64, page_size=64, act_dtype=abi.BF16,
                  cache_dtype=abi.BF16)
    assert lib.dsv4_qnorm_rope_kv_insert(qp, None) == abi.ERR_INVALID   # null pointers
    for k in ("q", "kv_new", "slot_mapping", "cache"):
        setattr(qp, k, 0x100000)
    qp.q_out = 0x100000 + 64 * 576 * 2                                  # overlaps q, different layout
    assert lib.dsv4_qnorm_rope_kv_insert(qp, None) == abi.ERR_INVALID
    qp.H_pad = 32
    assert lib.dsv4_qnorm_rope_kv_insert(qp, None) == abi.ERR_INVALID   # H_pad < H
    qp.H_pad, qp.q_out, qp.apply_q_rope = 64, 0x100000, 1
    assert lib.dsv4_qnorm_rope_kv_insert(qp, None) == abi.ERR_INVALID   # RoPE without a table
    qp.apply_q_rope, qp.act_dtype = 0, abi.FP8_DS_MLA
    assert lib.dsv4_qnorm_rope_kv_insert(qp, None) == abi.ERR_UNSUPPORTED
    assert lib.dsv4_padded_num_q_heads(32, abi.BF16) == 64
    assert lib.dsv4_padded_num_q_heads(64, abi.FP8_DS_MLA) == 64
    assert lib.dsv4_padded_num_q_heads(16, abi.F32) == 16
    assert lib.dsv4_padded_num_q_heads(0, abi.BF16) == -1
    assert lib.dsv4_abi_version() == abi.ABI_VERSION == 3

    c = abi.make(abi.CompressUpdateParams, T=2, B=1, q_per_seq=2, ratio=8, coff=1, page_size=64,
                 max_pages_per_seq=1, max_pos=10, cache_dtype=abi.BF16)
    assert lib.dsv4_compress_update(c, None) == abi.ERR_UNSUPPORTED   # ratio must be 4 or 128
    c.ratio, c.coff, c.T = 128, 1, 3
    assert lib.dsv4_compress_update(c, None) == abi.ERR_INVALID       # T != B * q_per_seq

    ix = abi.make(abi.IndexerTopkParams, T=1, B=1, q_per_seq=1, ratio=4, n_heads=64, head_dim=128, topk=512,
                  page_size=64, max_pages_per_seq=4, max_context=1000, q_dtype=abi.BF16, k_dtype=abi.BF16)
    need = lib.dsv4_indexer_topk_workspace_bytes(ix)
    assert need >= 4 * (1000 // 4)
    for k in ("q", "weights", "k_cache", "block_table", "positions", "topk_idx", "workspace"):
        setattr(ix, k, 0x10000)
    ix.workspace_bytes = need - 1
    assert lib.dsv4_indexer_topk(ix, None) == abi.ERR_INVALID         # workspace too small
    ix.workspace_bytes, ix.k_dtype = need, abi.FP8_DS_MLA
    assert lib.dsv4_indexer_topk(ix, None) == abi.ERR_UNSUPPORTED     # fp8 record is not an indexer key dtype
    ix.k_dtype, ix.head_dim = abi.BF16, 100
    assert lib.dsv4_indexer_topk(ix, None) == abi.ERR_UNSUPPORTED
    ix.head_dim, ix.cand_block_size, ix.cand_topk = 128, 1000, 8
    assert lib.dsv4_indexer_topk(ix, None) == abi.ERR_INVALID         # candidate block not a power of two
    ix.cand_block_size = 64
    assert lib.dsv4_indexer_topk(ix, None) == abi.ERR_INVALID         # below one 128-entry tile
    ix.cand_block_size, ix.cand_topk = 1024, 65
    assert lib.dsv4_indexer_topk(ix, None) == abi.ERR_INVALID         # more than 64 blocks a token
    ix.cand_topk = 8
    assert lib.dsv4_indexer_topk(ix, None) == abi.ERR_INVALID         # no candidate list
    ix.cand_blocks, ix.cand_write = 0x10002, 0
    assert lib.dsv4_indexer_topk(ix, None) == abi.ERR_INVALID         # misaligned list

    at = abi.make(abi.SparseMlaDecodeParams, T=1, B=1, q_per_seq=1, H=256, page_size=64, window=128, ratio=4,
                  swa_max_pages=1, max_context=100, q_dtype=abi.BF16, out_dtype=abi.BF16, cache_dtype=abi.BF16)
    assert lib.dsv4_sparse_mla_decode(at, None) == abi.ERR_UNSUPPORTED  # more than 128 heads
    at.H = 64
    assert lib.dsv4_sparse_mla_decode(at, None) == abi.ERR_INVALID      # null pointers
    assert lib.dsv4_sparse_mla_decode_workspace_bytes(at) > 0
    assert lib.dsv4_status_string(abi.ERR_BOUNDS).decode().startswith("a kernel skipped")
    n0 = lib.dsv4_kernel_launches()
    assert lib.dsv4_indexer_topk(ix, None) != abi.OK and lib.dsv4_kernel_launches() == n0  # refused: nothing launched
