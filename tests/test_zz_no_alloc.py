"""dsv4_indexer_topk_noalloc: the indexer + top-k call for callers that cannot allocate device memory
(for instance a plugin inside a host runtime that owns every device allocation).  Instead of a
caller-provided workspace it uses a fixed-size scratch array built into the library.

This file is named to run last: it checks the added entry point through the C ABI against the
regular dsv4_indexer_topk on the same inputs, on two calls in a row (the array keeps the previous
call's contents, which must not leak into the next result), and that a problem too large for the
array is refused before anything is launched.
"""
import numpy as np
import pytest
import torch

import dsv4_inputs as I

pytestmark = pytest.mark.gpu


def _regular_and_noalloc(name, cfg=None):
    import deepseek_v4_hybrid_gb300 as M
    from deepseek_v4_hybrid_gb300 import _abi
    from deepseek_v4_hybrid_gb300.step import DeviceStep
    st = I.make_step(cfg if cfg is not None else I.ALL_CONFIGS[name])
    ds = DeviceStep(st)
    ds.indexer()                                  # regular entry point, caller-owned workspace
    torch.cuda.synchronize()
    want_idx, want_score = ds.topk_idx.cpu().numpy(), ds.topk_score.cpu().numpy()

    got_idx = torch.full_like(ds.topk_idx, -7)
    got_score = torch.full_like(ds.topk_score, 7.0)
    p = _abi.make(_abi.IndexerTopkParams, **{f: getattr(ds.ix_params, f) for f, _ in _abi.IndexerTopkParams._fields_
                                           if f != "struct_size"})
    p.topk_idx, p.topk_score = got_idx.data_ptr(), got_score.data_ptr()
    p.workspace, p.workspace_bytes = None, 0     # ignored by the no-allocation variant
    lib = _abi.load()
    rc = lib.dsv4_indexer_topk_noalloc(p, torch.cuda.current_stream().cuda_stream)
    assert rc == _abi.OK, lib.dsv4_status_string(rc)
    torch.cuda.synchronize()
    assert M.dsv4_read_device_flags() == 0
    return want_idx, want_score, got_idx.cpu().numpy(), got_score.cpu().numpy(), p


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _near_limit_config():
    """A bf16-key c4 workload of 32 sequences (one long, the rest short) whose indexer workspace is just
    under the array's size (the workspace grows with tokens x the longest context)."""
    import dataclasses
    from deepseek_v4_hybrid_gb300 import _abi
    lib = _abi.load()
    base = I.CONFIGS["csa_c4_bf16"]
    best = None
    for ctx in range(4096, 1 << 22, 4096):
        p = _abi.make(_abi.IndexerTopkParams, T=32, B=32, q_per_seq=1, ratio=4, n_heads=64, head_dim=128, topk=512,
                      page_size=64, max_pages_per_seq=1, max_context=ctx, q_dtype=_abi.BF16, k_dtype=_abi.BF16)
        if lib.dsv4_indexer_topk_workspace_bytes(p) > _abi.NOALLOC_SCRATCH_BYTES:
            break
        best = ctx
    assert best is not None
    return dataclasses.replace(base, name="noalloc_near_limit", B=32, explicit_lens=(best,) + (3000,) * 31), best


def _check_same(name, want_idx, want_score, got_idx, got_score):
    assert np.array_equal(got_idx, want_idx), name
    valid = want_idx >= 0
    assert np.array_equal(got_score[valid], want_score[valid]), name
    assert np.all(got_score[~valid] == -np.inf)


def test_noalloc_matches_regular_entry_point_on_two_calls(cuda):
    # bf16, int8 row-scale and MXFP4 keys, larger problems first, then smaller ones: every call
    # must be unaffected by what the previous one left in the array
    for name in ("small_c4_h128", "small_c4_bf16", "small_c4_fp8", "small_c4_mxfp4"):
        _check_same(name, *_regular_and_noalloc(name)[:4])


def test_noalloc_just_under_its_limit(cuda):
    from deepseek_v4_hybrid_gb300 import _abi
    cfg, ctx = _near_limit_config()
    want_idx, want_score, got_idx, got_score, p = _regular_and_noalloc(cfg.name, cfg)
    lib = _abi.load()
    need = lib.dsv4_indexer_topk_workspace_bytes(p)
    assert _abi.NOALLOC_SCRATCH_BYTES - 2 * 1024 * 1024 < need <= _abi.NOALLOC_SCRATCH_BYTES, need
    _check_same(cfg.name, want_idx, want_score, got_idx, got_score)


def test_noalloc_rejects_problems_larger_than_its_scratch(cuda):
    """Refused before any launch: the outputs keep what they held."""
    from deepseek_v4_hybrid_gb300 import _abi
    _, _, _, _, p = _regular_and_noalloc("small_c4_bf16")
    lib = _abi.load()
    idx = torch.full((p.T, p.topk), -7, dtype=torch.int32, device="cuda")
    score = torch.full((p.T, p.topk), 7.0, dtype=torch.float32, device="cuda")
    p.topk_idx, p.topk_score = idx.data_ptr(), score.data_ptr()
    p.max_context = 1 << 30                       # needs far more scratch than the array holds
    assert lib.dsv4_indexer_topk_workspace_bytes(p) > _abi.NOALLOC_SCRATCH_BYTES
    assert lib.dsv4_indexer_topk_noalloc(p, torch.cuda.current_stream().cuda_stream) == _abi.ERR_INVALID
    torch.cuda.synchronize()
    assert torch.all(idx == -7) and torch.all(score == 7.0)
