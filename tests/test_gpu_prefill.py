"""GPU parity of the chunked prefill: the device runs the chain over consecutive 4-position chunks of
every sequence from position 0 on one set of caches; before each chunk the oracle takes the device's
caches as they are and computes that chunk's step, which must match everything the device wrote and
returned for it (so each chunk is checked on exactly the rows the earlier chunks left)."""
import numpy as np
import pytest
import torch

import dsv4_inputs as I
from oracle import compare as CMP
from oracle import dsv4_oracle as O

from test_gpu_parity import gpu_results, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import deepseek_v4_hybrid_gb300 as M
    return M


@pytest.mark.parametrize("name", ["prefill_c4_small", "prefill_c4_f32", "prefill_c128_small"])
def test_prefill_chunk_by_chunk_parity(lib, name):
    from deepseek_v4_hybrid_gb300.step import PrefillRunner
    cfg, P = I.PREFILL_CONFIGS[name]
    pf = I.make_prefill(cfg, P)
    runner = PrefillRunner(pf, chunk=4)
    assert runner.spans[-1][1] == (P % 4 or 4)
    sh = runner.shared
    for (p0, n), ds in zip(runner.spans, runner.steps):
        st = pf.chunk(p0, n)
        for f in ("swa_cache", "state", "main_cache", "idx_cache"):
            if f in sh:
                setattr(st, f, to_host(sh[f]).copy())
        ds.run()
        torch.cuda.synchronize()
        assert lib.dsv4_read_device_flags() == 0
        res = O.decode_step(st)
        rep = CMP.check_step(st, res, gpu_results(ds), where=f"{name} positions {p0}..{p0 + n - 1}")
        assert rep["tokens"] == cfg.B * n


def test_prefill_graph_replay_matches_eager(lib):
    """The whole prefill captured as one CUDA graph and replayed gives the eager run's outputs."""
    from deepseek_v4_hybrid_gb300.step import PrefillRunner
    cfg, P = I.PREFILL_CONFIGS["prefill_c4_small"]
    runner = PrefillRunner(I.make_prefill(cfg, 97), chunk=4)
    runner.run()
    torch.cuda.synchronize()
    eager = [(s.out.clone(), s.topk_idx.clone()) for s in runner.steps]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        runner.run()
    g.replay()
    torch.cuda.synchronize()
    assert lib.dsv4_read_device_flags() == 0
    for (o, k), s in zip(eager, runner.steps):
        assert torch.equal(o, s.out) and torch.equal(k, s.topk_idx)
