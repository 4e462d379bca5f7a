"""Pins of the oracle's compositions (no GPU needed): the value of one compressed entry, and which
rows one decode step's attention sees.

Both are recomputed here element by element with Python scalars (math.fsum, math.exp, math.sqrt)
in the order "DeepSeek V4 Attention: Code Reading Map", "How Does Compression Actually Work?"
gives the steps: softmax of the gate scores over the group's tokens per channel, the weighted sum
of kv, RMSNorm times its weight, then GPT-J RoPE of dims 512..575 at the group's position.  The
rotary table is built here from math.cos / math.sin, not taken from the input generator.  The
decode-step pin assembles the attended rows by hand (the window including this step's new row,
the selected compressed rows including the entry folded this step) and applies
scipy.special.softmax / logsumexp to them.
"""
import dataclasses
import math

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import dsv4_inputs as I
from oracle import dsv4_oracle as O

D, DV = 576, 512


def rotary_table(max_pos, theta=10000.0):
    """[max_pos, 64]: cos of the 32 pair angles then their sin; pair i turns by pos * theta^(-2i/64)."""
    t = np.zeros((max_pos, 64))
    for pos in range(max_pos):
        for i in range(32):
            a = pos * theta ** (-2.0 * i / 64.0)
            t[pos, i] = math.cos(a)
            t[pos, 32 + i] = math.sin(a)
    return t


def scalar_entry(state_b, j, ratio, coff, gamma, eps, table):
    """Compressed entry j of one sequence from its fp32 state ring, one channel at a time."""
    nslots = coff * ratio
    members = []  # (slot, kv column offset, score column offset) of every row in the group
    for pos in range(j * ratio, (j + 1) * ratio):
        members.append((pos % nslots, 0, coff * D))
    if coff == 2 and j >= 1:  # overlapping series B: the previous block's tokens
        for pos in range((j - 1) * ratio, j * ratio):
            members.append((pos % nslots, D, coff * D + D))
    e = [0.0] * D
    for c in range(D):
        scores = [float(state_b[s][so + c]) for s, _, so in members]
        kvs = [float(state_b[s][ko + c]) for s, ko, _ in members]
        top = max(scores)
        w = [math.exp(x - top) for x in scores]
        z = math.fsum(w)
        e[c] = math.fsum(wi * kv for wi, kv in zip(w, kvs)) / z
    inv = 1.0 / math.sqrt(math.fsum(x * x for x in e) / D + eps)
    n = [e[c] * inv * float(gamma[c]) for c in range(D)]
    row = table[j * ratio]
    for i in range(32):
        a, b = n[512 + 2 * i], n[512 + 2 * i + 1]
        cs, sn = float(row[i]), float(row[32 + i])
        n[512 + 2 * i] = a * cs - b * sn
        n[512 + 2 * i + 1] = a * sn + b * cs
    return np.array(n)


@pytest.mark.parametrize("ratio,coff,j", [(4, 2, 5), (4, 2, 1), (4, 2, 0), (128, 1, 3)])
def test_compressed_entry_matches_scalar_recomputation(ratio, coff, j):
    rng = np.random.default_rng(100 + ratio + j)
    nslots = coff * ratio
    state_b = rng.standard_normal((nslots, 2 * coff * D)).astype(np.float32)
    gamma = (1.0 + 0.5 * rng.standard_normal(D)).astype(np.float32)   # far from 1 on purpose
    table = rotary_table((j + 1) * ratio + 1)
    want = scalar_entry(state_b, j, ratio, coff, gamma, 1e-6, table)
    got = O.compressed_entry(state_b, j, ratio, coff, gamma, 1e-6, table)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_compressed_entry_rope_uses_group_position_row():
    """Entry j takes the rotary row j * ratio: swapping in row j changes the rope dims only."""
    ratio, coff, j = 4, 2, 6
    rng = np.random.default_rng(7)
    state_b = rng.standard_normal((coff * ratio, 2 * coff * D)).astype(np.float32)
    gamma = (1.0 + 0.5 * rng.standard_normal(D)).astype(np.float32)
    table = rotary_table(64)
    got = O.compressed_entry(state_b, j, ratio, coff, gamma, 1e-6, table)
    shifted = table.copy()
    shifted[j * ratio] = table[j]
    other = O.compressed_entry(state_b, j, ratio, coff, gamma, 1e-6, shifted)
    assert np.array_equal(got[:512], other[:512])
    assert np.max(np.abs(got[512:] - other[512:])) > 1e-3


def scalar_rotate(y, p, table):
    """GPT-J RoPE of dims 512..575 of a list of values as complex multiplication, in place."""
    for k in range(32):
        z = complex(y[512 + 2 * k], y[513 + 2 * k]) * complex(float(table[p][k]), float(table[p][32 + k]))
        y[512 + 2 * k], y[513 + 2 * k] = z.real, z.imag
    return y


def _emitting_step(ctx, topk_sel, q_prep):
    cfg = dataclasses.replace(I.CONFIGS["tiny_c4_f32"], name="pin_emit", B=1, H=4, topk=8,
                              explicit_lens=(ctx,), q_prep=q_prep)
    st = I.make_step(cfg)
    st.cos_sin = rotary_table(ctx + 1).astype(np.float32)
    sel = np.full((1, cfg.topk), -1, np.int32)
    sel[0, :len(topk_sel)] = topk_sel
    return cfg, st, sel


@pytest.mark.parametrize("q_prep", [False, True])
@pytest.mark.parametrize("ctx,sel", [(300, [3, 10, 50, 74]), (256, [0, 63, 12]), (300, [74])])
def test_decode_step_attends_this_steps_row_and_entry(ctx, sel, q_prep):
    """One sequence whose new token completes a group: the attention of decode_step must equal a
    softmax over rows put together by hand -- the window ending at this step's own new row, then
    the selected entries, where the entry folded this step comes from the updated state ring.  With
    the query preparation on, the new row is rotated at its position and every query head is
    RMS-normed (times its weight), rotated and stored as fp32 before the attention reads it."""
    cfg, st, given = _emitting_step(ctx, sel, q_prep)
    p = ctx - 1
    assert (p + 1) % cfg.ratio == 0
    j_new = p // cfg.ratio
    res = O.decode_step(st, topk_override=given)

    # the state ring after this step's store: the new token's row, with APE on the score half (fp32)
    ring = np.array(st.state[0], np.float32, copy=True)
    new_row = np.array(st.kv_score[0], np.float32, copy=True)
    coff = cfg.coff
    new_row[coff * D:] = (new_row[coff * D:] + st.ape[p % cfg.ratio]).astype(np.float32)
    ring[p % (coff * cfg.ratio)] = new_row

    rows = []
    for pos in range(max(0, p - 127), p + 1):
        if pos == p:                                                     # inserted this step
            row = [float(x) for x in st.kv_new[0]]
            if q_prep:
                row = scalar_rotate(row, p, st.cos_sin)
            rows.append(np.asarray(row, np.float32).astype(np.float64))  # stored as fp32
        else:
            page = st.swa_bt[0][pos // 64]
            rows.append(np.asarray(st.swa_cache[page, pos % 64], np.float64))
    for j in given[0]:
        if j < 0 or j >= (p + 1) // cfg.ratio:
            continue
        if j == j_new:                                                   # folded this step
            e = scalar_entry(ring, j, cfg.ratio, coff, st.norm_w, st.eps, st.cos_sin)
            rows.append(e.astype(np.float32).astype(np.float64))        # stored as fp32
        else:
            page = st.main_bt[0][j // 64]
            rows.append(np.asarray(st.main_cache[page, j % 64], np.float64))
    R = np.stack(rows)
    if j_new in given[0]:
        assert R.shape[0] == min(p + 1, 128) + len(sel)

    q = np.asarray(st.q[0], np.float64)
    if q_prep:
        for h in range(cfg.H):
            inv = 1.0 / math.sqrt(math.fsum(x * x for x in q[h]) / D + st.eps)
            y = scalar_rotate([q[h][c] * inv * float(st.q_norm_w[c]) for c in range(D)], p, st.cos_sin)
            q[h] = np.asarray(y, np.float32)                             # stored as fp32
        np.testing.assert_allclose(np.asarray(res["q_out"][0])[:cfg.H].astype(np.float64), q, rtol=2.0 ** -23, atol=0)
    for h in range(cfg.H):
        z = st.softmax_scale * (R @ q[h])
        logits = np.concatenate([z, [float(st.sink[h])]])
        w = softmax(logits)[:-1]
        want = (w[:, None] * R[:, :DV]).sum(axis=0)
        np.testing.assert_allclose(res["out"][0][h], want, rtol=1e-9, atol=1e-12)
        assert abs(res["lse"][0][h] - logsumexp(logits)) <= 1e-10 * max(1.0, abs(logsumexp(logits)))


# ------------------------------------------------------------------------------------------------
# query preparation: per-head RMSNorm, GPT-J RoPE of dims 512..575, zero padding
# ------------------------------------------------------------------------------------------------

def test_qnorm_rope_against_scalar_recomputation():
    """Every head: RMSNorm over its 576 dims (weight far from 1), then each GPT-J pair of the rope
    dims turned as the complex number x_2k + i x_2k+1 times e^(i p theta^(-2k/64)), the angle taken
    from math.cos / math.sin here; heads past H are zero."""
    rng = np.random.default_rng(11)
    H, h_pad, p = 5, 8, 777
    q = rng.standard_normal((H, D)) * 0.3
    w = 1.0 + 0.5 * rng.standard_normal(D)
    table = rotary_table(p + 1)
    got = O.qnorm_rope(q, p, table, w, 1e-6, True, True, h_pad)
    for h in range(H):
        inv = 1.0 / math.sqrt(math.fsum(x * x for x in q[h]) / D + 1e-6)
        y = [q[h][c] * inv * w[c] for c in range(D)]
        for k in range(32):
            ang = p * 10000.0 ** (-2.0 * k / 64.0)
            z = complex(y[512 + 2 * k], y[513 + 2 * k]) * complex(math.cos(ang), math.sin(ang))
            y[512 + 2 * k], y[513 + 2 * k] = z.real, z.imag
        np.testing.assert_allclose(got[h], y, rtol=1e-12, atol=1e-12)
    assert np.all(got[H:] == 0.0)


def test_qnorm_invariants_and_switches():
    rng = np.random.default_rng(12)
    q = rng.standard_normal((3, D))
    table = rotary_table(40)
    # unit weight, no rope: every head's mean square is ms / (ms + eps); a head scaled by c > 0 maps
    # to (nearly) the same output
    y = O.qnorm_rope(q, 30, table, None, 1e-6, True, False, 3)
    for h in range(3):
        ms = np.mean(q[h] ** 2)
        assert abs(np.mean(y[h] ** 2) - ms / (ms + 1e-6)) < 1e-12
    y2 = O.qnorm_rope(q * 7.5, 30, table, None, 1e-6, True, False, 3)
    np.testing.assert_allclose(y2, y, rtol=1e-6)
    # rope only: the no-pe dims are untouched, each rope pair keeps its length, position 0 is the identity
    r = O.qnorm_rope(q, 30, table, None, 1e-6, False, True, 3)
    assert np.array_equal(r[:, :512], q[:, :512])
    np.testing.assert_allclose(np.hypot(r[:, 512::2], r[:, 513::2]), np.hypot(q[:, 512::2], q[:, 513::2]), rtol=1e-12)
    assert np.array_equal(O.qnorm_rope(q, 0, table, None, 1e-6, False, True, 3), q)
    # neither switch: a copy, zero padded
    z = O.qnorm_rope(q, 5, table, None, 1e-6, False, False, 6)
    assert np.array_equal(z[:3], q) and np.all(z[3:] == 0.0)


# ------------------------------------------------------------------------------------------------
# index keys written by the compressor
# ------------------------------------------------------------------------------------------------

def scalar_index_key(latent, wk, kn_w, eps, table, pos):
    """k = wk latent (fsum dot products), RMSNorm over its dims times kn_w, then its last 64 dims
    turned pairwise as complex numbers by the rotary row of `pos`."""
    d = len(wk)
    k = [math.fsum(float(wk[o][c]) * float(latent[c]) for c in range(len(latent))) for o in range(d)]
    inv = 1.0 / math.sqrt(math.fsum(x * x for x in k) / d + eps)
    k = [k[o] * inv * float(kn_w[o]) for o in range(d)]
    base = d - 64
    for i in range(32):
        z = complex(k[base + 2 * i], k[base + 2 * i + 1]) * complex(float(table[pos][i]), float(table[pos][32 + i]))
        k[base + 2 * i], k[base + 2 * i + 1] = z.real, z.imag
    return np.array(k)


def scalar_latent(state_b, j, ratio, coff, gamma, eps):
    """scalar_entry without its RoPE step: the fold, then RMSNorm times gamma."""
    no_rope = np.zeros((j * ratio + 1, 64))
    no_rope[:, :32] = 1.0                                   # cos 1, sin 0 at every position: identity
    return scalar_entry(state_b, j, ratio, coff, gamma, eps, no_rope)


@pytest.mark.parametrize("d", [128, 64])
def test_index_key_matches_scalar_recomputation(d):
    rng = np.random.default_rng(40 + d)
    ratio, coff, j = 4, 2, 9
    state_b = rng.standard_normal((coff * ratio, 2 * coff * D)).astype(np.float32)
    gamma = (1.0 + 0.5 * rng.standard_normal(D)).astype(np.float32)
    wk = rng.standard_normal((d, D)) * 0.05
    kn_w = 1.0 + 0.5 * rng.standard_normal(d)
    table = rotary_table(j * ratio + 1)
    lat = scalar_latent(state_b, j, ratio, coff, gamma, 1e-6)
    np.testing.assert_allclose(O.entry_latent(state_b, j, ratio, coff, gamma, 1e-6), lat, rtol=1e-12, atol=1e-12)
    want = scalar_index_key(lat, wk, kn_w, 1e-6, table, j * ratio)
    got = O.index_key(O.entry_latent(state_b, j, ratio, coff, gamma, 1e-6), wk, kn_w, 1e-6, table, j * ratio)
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("ctx", [300, 1024])
def test_decode_step_scores_the_key_written_this_step(ctx):
    """The indexer of the step sees the index key the compressor stored this step: the score of the
    new entry j = p / 4 equals sum_h w_h ReLU(q_h . k) with k assembled by hand from the updated
    state ring and stored as fp32 (the config's key dtype)."""
    cfg = dataclasses.replace(I.CONFIGS["tiny_c4_f32"], name="pin_key", B=1, explicit_lens=(ctx,))
    st = I.make_step(cfg)
    st.cos_sin = rotary_table(ctx + 1).astype(np.float32)
    p = ctx - 1
    j_new = p // cfg.ratio
    res = O.decode_step(st)
    ring = np.array(st.state[0], np.float32, copy=True)
    new_row = np.array(st.kv_score[0], np.float32, copy=True)
    new_row[cfg.coff * D:] = (new_row[cfg.coff * D:] + st.ape[p % cfg.ratio]).astype(np.float32)
    ring[p % (cfg.coff * cfg.ratio)] = new_row
    lat = scalar_latent(ring, j_new, cfg.ratio, cfg.coff, st.norm_w, st.eps)
    k = scalar_index_key(lat, O.bf16_decode(st.wk), st.ik_norm_w, st.eps, st.cos_sin, j_new * cfg.ratio)
    k = k.astype(np.float32).astype(np.float64)
    q = np.asarray(st.q_idx[0], np.float64)
    want = math.fsum(float(st.w_idx[0][h]) * max(0.0, math.fsum(q[h] * k)) for h in range(cfg.I_h))
    got = float(res["scores"][0][j_new])
    assert abs(got - want) <= 1e-6 * max(1.0, abs(want))
    assert np.array_equal(res["idx_written"][(st.idx_bt[0][j_new // 64], j_new % 64)], k.astype(np.float32))


# ------------------------------------------------------------------------------------------------
# chunked prefill: the chain over consecutive chunks from position 0
# ------------------------------------------------------------------------------------------------

def _prefill(name, P, chunk, **kw):
    cfg, _ = I.PREFILL_CONFIGS[name]
    pf = I.make_prefill(dataclasses.replace(cfg, **kw), P)
    toks = O.prefill(pf.chunk(p0, n) for p0, n in pf.spans(chunk))
    return pf, toks


@pytest.mark.parametrize("name,P", [("prefill_c4_f32", 70), ("prefill_c128_small", 260)])
def test_prefill_does_not_depend_on_the_chunk_size(name, P):
    """Each token reads only rows written at its own or earlier positions, so chunks of 4, 1 and 3
    positions give the same results and the same caches, bit for bit."""
    kw = {"B": 1, "H": 8} if name == "prefill_c128_small" else {}
    ref_pf, ref = _prefill(name, P, 4, **kw)
    for c in (1, 3):
        pf, got = _prefill(name, P, c, **kw)
        assert got.keys() == ref.keys()
        for k, v in ref.items():
            assert np.array_equal(got[k]["out"], v["out"]) and np.array_equal(got[k]["lse"], v["lse"]), (c, k)
            assert (v["topk"] is None) == (got[k]["topk"] is None)
            if v["topk"] is not None:
                assert np.array_equal(got[k]["topk"], v["topk"]), (c, k)
        for f in ("swa_cache", "state", "main_cache", "idx_cache"):
            a, b = getattr(ref_pf.base, f), getattr(pf.base, f)
            assert (a is None) == (b is None) and (a is None or np.array_equal(a, b)), (c, f)


def test_prefill_of_100_tokens_gives_25_entries_and_attends_them_all():
    """"DeepSeek-V4 Inference on Ascend", §8 "The prefill path": a 100-token prefill through a c4 layer
    leaves 25 compressed entries, the indexer's top-k of those 25 is all of them, and the attention of
    the last token scores the window plus the chosen entries.  Rebuilt here from the inputs alone: the
    window rows are the tokens' kv rotated at their positions, entry j is the scalar fold of the state
    rows of positions 4j - 4 .. 4j + 3."""
    cfg, _ = I.PREFILL_CONFIGS["prefill_c4_f32"]
    cfg = dataclasses.replace(cfg, B=1, H=4, topk=64)
    pf = I.make_prefill(cfg, 100)
    st = pf.base
    st.cos_sin = rotary_table(101).astype(np.float32)
    main_before = st.main_cache.copy()
    toks = O.prefill(pf.chunk(p0, n) for p0, n in pf.spans(4))
    ratio, coff = cfg.ratio, cfg.coff
    # the 25 entries, and nothing past them
    ents = []
    for j in range(25):
        ring = np.zeros((coff * ratio, 2 * coff * D), np.float32)
        for pos in range(max(0, 4 * j - 4), 4 * j + 4):
            r = np.array(st.kv_score[pos], np.float32, copy=True)
            r[coff * D:] = (r[coff * D:] + st.ape[pos % ratio]).astype(np.float32)
            ring[pos % (coff * ratio)] = r
        e = scalar_entry(ring, j, ratio, coff, st.norm_w, st.eps, st.cos_sin).astype(np.float32)
        got = st.main_cache[st.main_bt[0][j // 64], j % 64]
        np.testing.assert_allclose(got.astype(np.float64), e.astype(np.float64), rtol=1e-6, atol=1e-7)
        ents.append(got.astype(np.float64))
    for j in range(25, st.main_cache.shape[0] * 64):
        pg = st.main_bt[0][j // 64] if j // 64 < st.main_bt.shape[1] else -1
        if pg >= 0:
            assert np.array_equal(st.main_cache[pg, j % 64], main_before[pg, j % 64])
    last = toks[(0, 99)]
    assert sorted(last["topk"][:25].tolist()) == list(range(25)) and np.all(last["topk"][25:] == -1)
    rows = [np.asarray(scalar_rotate([float(x) for x in st.kv_new[pos]], pos, st.cos_sin), np.float32)
            .astype(np.float64) for pos in range(100)]
    R = np.stack(rows + ents)
    assert R.shape[0] == 100 + 25
    q = np.asarray(st.q[99], np.float64)
    for h in range(cfg.H):
        inv = 1.0 / math.sqrt(math.fsum(x * x for x in q[h]) / D + st.eps)
        qh = np.asarray(scalar_rotate([q[h][c] * inv * float(st.q_norm_w[c]) for c in range(D)], 99, st.cos_sin),
                        np.float32).astype(np.float64)
        logits = np.concatenate([st.softmax_scale * (R @ qh), [float(st.sink[h])]])
        want = (softmax(logits)[:-1, None] * R[:, :DV]).sum(axis=0)
        np.testing.assert_allclose(last["out"][h], want, rtol=1e-6, atol=1e-9)
