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


def _regular_and_noalloc(name):
    import deepseek_v4_hybrid_gb300 as M
    from deepseek_v4_hybrid_gb300 import _abi
    from deepseek_v4_hybrid_gb300.step import DeviceStep
    st = I.make_step(I.ALL_CONFIGS[name])
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


def test_noalloc_matches_regular_entry_point_on_two_calls(cuda):
    for name in ("small_c4_h128", "small_c4_bf16"):   # larger problem first, then a smaller one
        want_idx, want_score, got_idx, got_score, _ = _regular_and_noalloc(name)
        assert np.array_equal(got_idx, want_idx), name
        valid = want_idx >= 0
        assert np.array_equal(got_score[valid], want_score[valid]), name
        assert np.all(got_score[~valid] == -np.inf)


def test_noalloc_rejects_problems_larger_than_its_scratch(cuda):
    from deepseek_v4_hybrid_gb300 import _abi
    _, _, _, _, p = _regular_and_noalloc("small_c4_bf16")
    lib = _abi.load()
    p.max_context = 1 << 30                       # needs far more scratch than the array holds
    assert lib.dsv4_indexer_topk_workspace_bytes(p) > _abi.NOALLOC_SCRATCH_BYTES
    assert lib.dsv4_indexer_topk_noalloc(p, torch.cuda.current_stream().cuda_stream) == _abi.ERR_INVALID
