"""The oracle's whole-step run on the small workloads: shapes, counts and internal consistency."""
import numpy as np
import pytest

import dsv4_inputs as I
from oracle import dsv4_oracle as O


@pytest.mark.parametrize("name", sorted(I.SMALL_CONFIGS))
def test_oracle_step_runs_and_is_consistent(name):
    st = I.make_step(I.SMALL_CONFIGS[name])
    cfg = st.cfg
    res = O.decode_step(st)
    for t in res["tokens"]:
        out, lse = res["out"][t], res["lse"][t]
        assert out.shape == (cfg.H, 512) and np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
        if cfg.topk:
            p = int(st.positions[t])
            nc = O.n_compressed(p, cfg.ratio)
            sel = res["topk"][t]
            avail = nc
            if cfg.cand_block and not cfg.cand_write and nc > cfg.topk:
                # a candidate consumer: only entries of its listed blocks
                listed = set(O.listed_blocks(st.cand_in[t]))
                avail = sum(1 for j in range(nc) if j // cfg.cand_block in listed)
                assert all(j // cfg.cand_block in listed for j in sel[sel >= 0])
            assert np.sum(sel >= 0) == min(avail, cfg.topk)
            assert np.all(sel[sel >= 0] < nc)
            if cfg.cand_block and cfg.cand_write:
                cb = res["cand_out"][t]
                nblk = -(-nc // cfg.cand_block)
                assert np.sum(cb >= 0) == min(nblk, cfg.cand_topk) and np.all(np.diff(cb[cb >= 0]) > 0)
    # every emitting token wrote exactly one main-cache row at j = p // ratio
    if cfg.ratio:
        emit = [(t // cfg.q_per_seq, int(st.positions[t]) // cfg.ratio) for t in range(cfg.T)
                if O.emits(int(st.positions[t]), cfg.ratio)]
        assert sorted(res["entries"]) == sorted(emit)
    assert len(res["swa_written"]) == cfg.T


def test_attention_only_override_matches_given_selection():
    st = I.make_step(I.SMALL_CONFIGS["small_c4_bf16"])
    a = O.decode_step(st, topk_override=st.given_topk)
    b = O.decode_step(st)
    t = 0
    assert not np.array_equal(a["out"][t], b["out"][t])
