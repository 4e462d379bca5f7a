"""Comparison of a device decode step's results with the oracle's (test infrastructure only).

Tolerances: integer work (slots, state rows, top-k sets) must match exactly, except top-k
entries whose oracle score lies within 1e-5 of the k-th best (near-ties may rank either way).
Attention outputs: max |gpu - oracle| <= 2e-2 * max |oracle| per token for bf16/fp8 caches and
<= 1e-4 * max |oracle| for fp32.  Compressed entries written by the fold: within one unit in the
last place of their storage format (plus 1e-5 of the row max for the fp32 arithmetic).
"""
from __future__ import annotations

import numpy as np

from . import dsv4_oracle as O

TIE_EPS = 1e-5


def attention_tolerance(cache_dtype: int) -> float:
    return 1e-4 if cache_dtype == O.F32 else 2e-2


def _e4m3_ulp(v):
    v = np.abs(v)
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -6)))
    return np.exp2(e - 3)


def entry_error_ok(stored_gpu, value, dtype):
    """Is a stored compressed entry within one storage ulp of the oracle's (unencoded) value?"""
    dec = O.decode_rows(stored_gpu, dtype)
    value = np.asarray(value, np.float64)
    amax = np.max(np.abs(value))
    if dtype == O.F32:
        return np.max(np.abs(dec - value)) <= 1e-5 * amax, dec
    if dtype == O.BF16:
        bound = np.abs(value) * 2.0 ** -7 + 1e-5 * amax
        return bool(np.all(np.abs(dec - value) <= bound)), dec
    # fp8_ds_mla: per 64-dim block, one e4m3 ulp at the block's scale; rope dims as bf16
    ok = True
    for blk in range(8):
        seg = slice(64 * blk, 64 * blk + 64)
        eb = O.ue8m0_exponent(np.max(np.abs(value[seg])))
        bound = _e4m3_ulp(value[seg] / 2.0 ** eb) * 2.0 ** eb + 1e-5 * amax
        ok &= bool(np.all(np.abs(dec[seg] - value[seg]) <= bound))
    ok &= bool(np.all(np.abs(dec[512:] - value[512:]) <= np.abs(value[512:]) * 2.0 ** -7 + 1e-5 * amax))
    return ok, dec


KEY_ABS = 1e-4  # of the key row's largest element: each element is a 576-term fp32 dot product (the
                # device sums in another order than the oracle's fp64) of RMS-normalised values


def key_ulps(stored, dtype):
    """Per-element bound on how far the device's encoding of a key may lie from the oracle's `stored`
    one: one unit in the last place of the format (bf16 element, int8 code step), plus KEY_ABS of the
    row's largest element for the fp32 arithmetic before the rounding."""
    v = O.decode_rows(stored, dtype)
    slack = KEY_ABS * np.max(np.abs(v))
    if dtype == O.F32:
        return np.zeros(v.shape) + slack
    if dtype == O.BF16:
        a = np.maximum(np.abs(v), 2.0 ** -126)
        return np.exp2(np.floor(np.log2(a)) - 7) + slack
    st = np.asarray(stored, np.uint8)
    if dtype == O.MXFP4:
        # two E2M1 steps (0.5 below 2, 1 in [2, 4), 2 above) at the block's scale: a neighbouring code, or
        # the next block exponent when the block's max sits at the exponent's boundary
        d = v.shape[-1]
        scale = np.repeat(np.exp2(st[d // 2:].astype(np.float64) - 127.0), O.MXFP4_BLOCK)
        a = np.abs(v) / scale
        step = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
        return 2.0 * step * scale + slack
    scale = float(np.ascontiguousarray(st[-4:]).view(np.float32)[0])
    return np.full(v.shape, scale * 1.001) + slack


def key_ok(stored_gpu, stored_oracle, dtype):
    """An index key written by the device within one storage unit of the oracle's."""
    g = O.decode_rows(stored_gpu, dtype)
    o = O.decode_rows(stored_oracle, dtype)
    return bool(np.all(np.abs(g - o) <= key_ulps(stored_oracle, dtype) * 1.0001))


def new_key_score_bound(q_t, w_t, stored_key, dtype):
    """How far the score of an entry whose key was written this step may move when the key changes by
    at most one storage unit per element: |sum_h w_h (ReLU(q_h.k') - ReLU(q_h.k))| <= sum_h |w_h|
    sum_d |q_hd| u_d (ReLU is 1-Lipschitz)."""
    u = key_ulps(stored_key, dtype)
    return float(np.sum(np.abs(np.asarray(w_t, np.float64)) * (np.abs(np.asarray(q_t, np.float64)) @ u)))


def topk_sets_match(gpu_idx, oracle_scores, k, slack=0.0):
    """GPU list vs the oracle's scores: same set except near-ties at the k-th score (within TIE_EPS,
    plus `slack` when this step wrote keys the scores depend on); returns (ok, exact) where exact
    says the two sets are identical."""
    s = np.asarray(oracle_scores, np.float32)
    n = s.shape[0]
    g = np.asarray(gpu_idx)
    m = min(n, k)
    valid = g[g >= 0]
    if len(valid) != m or np.any(g[m:] != -1) or len(set(valid.tolist())) != m or np.any(valid >= n):
        return False, False
    want = set(O.topk_select(s, k)[:m].tolist())
    got = set(valid.tolist())
    if got == want:
        return True, True
    if m == 0:
        return True, True
    kth = np.sort(s)[::-1][m - 1]
    diff = got ^ want
    return bool(all(abs(float(s[j]) - float(kth)) <= TIE_EPS + slack for j in diff)), False


def included_entries(cand_row, nc, block):
    """Entries j < nc of the blocks a consumer's list names, increasing."""
    listed = O.listed_blocks(cand_row)
    return np.array([j for b in listed for j in range(b * block, min((b + 1) * block, nc))], np.int64)


def masked_topk_match(gpu_idx, oracle_scores, k, inc, slack=0.0):
    """topk_sets_match for a candidate consumer: every selected entry lies in `inc` (the included
    entries, increasing), and the selection matches the oracle's top-k among them."""
    g = np.asarray(gpu_idx)
    valid = g[g >= 0]
    if not np.all(np.isin(valid, inc)):
        return False, False
    sub = np.where(g >= 0, np.searchsorted(inc, np.maximum(g, 0)), -1)  # positions within inc
    return topk_sets_match(sub, np.asarray(oracle_scores, np.float32)[inc], k, slack)


def cand_blocks_match(gpu_row, oracle_scores, block, m, slack=0.0):
    """The source's published blocks vs the oracle's scores: every block when there are at most m;
    else m distinct increasing blocks whose set differs from the oracle's only in blocks whose block
    score lies within TIE_EPS (+ slack) of the oracle's m-th best block score."""
    s = np.asarray(oracle_scores, np.float32)
    n = s.shape[0]
    nblk = -(-n // block)
    g = np.asarray(gpu_row)
    if nblk <= m:
        return bool(np.array_equal(g, np.concatenate([np.arange(nblk), np.full(m - nblk, -1)])))
    if np.any(g < 0) or np.any(g >= nblk) or np.any(np.diff(g) <= 0):
        return False
    want = O.candidate_blocks(s, block, m)
    diff = set(g.tolist()) ^ set(want.tolist())
    if not diff:
        return True
    bmax = np.array([np.max(s[b * block:(b + 1) * block]) for b in range(nblk)], np.float64)
    mth = np.sort(bmax)[::-1][m - 1]
    return bool(all(abs(bmax[b] - mth) <= TIE_EPS + slack for b in diff))


def q_out_ok(stored_gpu, stored_oracle, act_dtype):
    """Prepared query heads: padding heads exactly zero; the others within one unit in the last place
    of the activation format (the device normalises in fp32, the oracle in fp64) plus 1e-6 of the
    head's largest value."""
    g = O.decode_rows(stored_gpu, act_dtype)
    o = O.decode_rows(stored_oracle, act_dtype)
    rel = 2.0 ** -7 if act_dtype == O.BF16 else 1e-5
    amax = np.max(np.abs(o), axis=-1, keepdims=True)
    return bool(np.all(np.abs(g - o) <= rel * np.abs(o) + 1e-6 * amax))


def check_step(st, res, gpu, where=""):
    """Asserts parity of every device result in `gpu` (numpy arrays) with the oracle's `res`.
    Returns a small report dict."""
    cfg = st.cfg
    rep = {"tokens": len(res["tokens"]), "max_rel_err": 0.0, "tie_tokens": 0}
    # a1: inserted SWA rows (rotated in fp32 when the insert applies RoPE: within one storage ulp of the
    # oracle's row, else bit-exact)
    rotated = bool(getattr(cfg, "q_prep", False))
    for (page, off), row in res["swa_written"].items():
        if rotated:
            ok, _ = entry_error_ok(gpu["swa_cache"][page, off], O.decode_rows(row, cfg.cache_dtype), cfg.cache_dtype)
            assert ok, f"{where} SWA row {(page, off)}"
        else:
            assert np.array_equal(gpu["swa_cache"][page, off], row), f"{where} SWA row {(page, off)}"
    # the prepared queries
    for t, qo in res.get("q_out", {}).items():
        if "q_out" in gpu:
            H = cfg.H
            assert np.all(O.decode_rows(gpu["q_out"][t][H:], cfg.act_dtype) == 0.0), f"{where} padded heads of {t}"
            assert q_out_ok(gpu["q_out"][t][:H], qo[:H], cfg.act_dtype), f"{where} prepared query of token {t}"
    if cfg.ratio:
        # a2: fp32 state ring, bit-exact; emitted entries within one storage ulp
        for b, stb in res["state"].items():
            assert np.array_equal(gpu["state"][b], stb), f"{where} state of seq {b}"
        for (b, j), e in res["entries"].items():
            page = st.main_bt[b][j // O.PAGE]
            ok, _ = entry_error_ok(gpu["main_cache"][page, j % O.PAGE], e, cfg.cache_dtype)
            assert ok, f"{where} compressed entry {(b, j)}"
    # index keys written by the compressor: within one storage unit of the oracle's
    for (page, off), row in res.get("idx_written", {}).items():
        assert key_ok(gpu["idx_cache"][page, off], row, cfg.idx_dtype), f"{where} index key row {(page, off)}"
    new_keys = {}
    for (b, j) in res.get("keys", {}):
        new_keys.setdefault(b, []).append(j)
    same_sel = {}
    if cfg.ratio and cfg.topk:
        for t in res["tokens"]:
            b = t // cfg.q_per_seq
            bounds = {}
            for j in new_keys.get(b, []):
                if j < len(res["scores"][t]):
                    row = res["idx_written"][(int(st.idx_bt[b][j // O.PAGE]), j % O.PAGE)]
                    bounds[j] = new_key_score_bound(O.decode_rows(st.q_idx[t], cfg.act_dtype), st.w_idx[t], row,
                                                    cfg.idx_dtype)
            slack = 2.0 * max(bounds.values(), default=0.0)
            nc = len(res["scores"][t])
            cb = getattr(cfg, "cand_block", 0)
            if cb and not getattr(cfg, "cand_write", False) and nc > cfg.topk:
                inc = included_entries(st.cand_in[t], nc, cb)
                ok, exact = masked_topk_match(gpu["topk_idx"][t], res["scores"][t], cfg.topk, inc, slack)
            else:
                ok, exact = topk_sets_match(gpu["topk_idx"][t], res["scores"][t], cfg.topk, slack)
            assert ok, f"{where} top-k of token {t}"
            if cb and getattr(cfg, "cand_write", False) and "cand_out" in gpu:
                assert cand_blocks_match(gpu["cand_out"][t], res["scores"][t], cb, cfg.cand_topk, slack), \
                    f"{where} published candidate blocks of token {t}"
            same_sel[t] = exact
            rep["tie_tokens"] += int(not exact)
            if "topk_score" in gpu and exact:
                sel = gpu["topk_idx"][t]
                valid = sel[sel >= 0]
                sv = gpu["topk_score"][t][sel >= 0]
                ref = res["scores"][t][valid]
                extra = np.array([bounds.get(int(j), 0.0) for j in valid])
                scale = max(1e-30, float(np.max(np.abs(res["scores"][t]))) if len(res["scores"][t]) else 1.0)
                assert np.all(np.abs(sv - ref) <= 1e-5 * scale + 1e-7 + extra), f"{where} top-k scores of token {t}"
    tol = attention_tolerance(cfg.cache_dtype)
    for t in res["tokens"]:
        if same_sel.get(t, True) is False:
            continue  # a near-tie changed the selected rows: attention is checked on given selections
        ref = res["out"][t]
        out = gpu["out"][t][:ref.shape[0]].astype(np.float64)  # the padding heads are not compared
        amax = float(np.max(np.abs(ref)))
        err = float(np.max(np.abs(out - ref)))
        rep["max_rel_err"] = max(rep["max_rel_err"], err / amax)
        assert err <= tol * amax, f"{where} attention of token {t}: err {err:.3e} vs {tol} * {amax:.3e}"
        if "lse" in gpu:
            lerr = float(np.max(np.abs(gpu["lse"][t][:ref.shape[0]] - res["lse"][t])))
            assert lerr <= (1e-5 if cfg.cache_dtype == O.F32 else 2e-3), f"{where} lse of token {t}: {lerr:.3e}"
    return rep
