"""The parity checks' own helpers for candidate filtering accept the oracle's answers and reject
planted mistakes (test infrastructure checked on the CPU)."""
import numpy as np

from oracle import compare as CMP
from oracle import dsv4_oracle as O


def _scores(n, seed):
    return np.random.default_rng(seed).standard_normal(n).astype(np.float32)


def test_masked_topk_match_accepts_the_oracle_and_rejects_mistakes():
    s = _scores(3000, 1)
    cand = np.array([0, 2, 5, -1], np.int32)
    inc = CMP.included_entries(cand, 3000, 512)
    assert inc[-1] == 2999 and len(inc) == 512 + 512 + (3000 - 2560)
    sel = np.sort(O.masked_topk(s, 200, cand, 512))
    assert CMP.masked_topk_match(sel, s, 200, inc) == (True, True)
    bad = sel.copy()
    bad[0] = 600                                  # an entry of block 1, which the list does not name
    assert not CMP.masked_topk_match(np.sort(bad), s, 200, inc)[0]
    order = inc[np.argsort(-s[inc].astype(np.float64), kind="stable")]
    swap = sel.copy()
    swap[np.searchsorted(sel, order[0])] = order[600]   # the best entry replaced by a far worse one
    assert not CMP.masked_topk_match(np.sort(swap), s, 200, inc)[0]
    few = np.full(200, -1, np.int32)
    few[:100] = sel[:100]                          # too few entries
    assert not CMP.masked_topk_match(few, s, 200, inc)[0]


def test_cand_blocks_match_accepts_the_oracle_and_rejects_mistakes():
    s = _scores(5000, 2)
    got = O.candidate_blocks(s, 256, 6)
    assert CMP.cand_blocks_match(got, s, 256, 6)
    bmax = np.array([s[b * 256:(b + 1) * 256].max() for b in range(20)])
    worst = int(np.argmin(bmax))
    bad = got.copy()
    bad[0] = worst
    assert not CMP.cand_blocks_match(np.sort(bad), s, 256, 6)    # a low block instead of a best one
    assert not CMP.cand_blocks_match(got[::-1], s, 256, 6)       # not increasing
    short = s[:700]                                                # 3 blocks <= 6: all of them, then -1
    assert CMP.cand_blocks_match(np.array([0, 1, 2, -1, -1, -1]), short, 256, 6)
    assert not CMP.cand_blocks_match(np.array([0, 1, -1, -1, -1, -1]), short, 256, 6)
