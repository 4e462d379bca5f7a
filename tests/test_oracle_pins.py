"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test checks the oracle against something it does not compute itself: a library routine
(torch's bf16 / float8_e4m3fn conversions, scipy's softmax), brute force on tiny inputs, a closed
form, an invariant, or a number the pages print (tests/golden/worked_numbers.json).
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

import dsv4_inputs as I
from oracle import dsv4_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_numbers.json")


def golden(case_id):
    with open(GOLDEN) as f:
        return {c["id"]: c for c in json.load(f)["cases"]}[case_id]


# ------------------------------------------------------------------------------------------------
# codecs against torch's conversions
# ------------------------------------------------------------------------------------------------

def test_bf16_codec_matches_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 20000),
                        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, 1e-40, -1e-41], np.float32)]).astype(np.float32)
    # exact ties between two bf16 neighbours (the low 16 bits = 0x8000)
    ties = ((rng.integers(0x3F000000, 0x41000000, 2000, dtype=np.uint32) & np.uint32(0xFFFF0000)) | np.uint32(0x8000))
    x = np.concatenate([x, ties.view(np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.bf16_encode(x.astype(np.float64))
    assert np.array_equal(got, want)
    back = torch.from_numpy(want.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(O.bf16_decode(want), back)


def test_e4m3_decode_all_codes_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = O.e4m3_decode(codes)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert set(codes[nan].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(got[~nan], want[~nan])
    assert got[0x7E] == 448.0


def test_e4m3_encode_matches_torch_rne():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(50000) * 50.0, rng.standard_normal(20000) * 0.01,
                        rng.uniform(-448, 448, 20000)]).astype(np.float32)
    # midpoints between neighbouring e4m3 values: round-half-even decides
    vals = O.e4m3_decode(np.arange(0, 0x7E, dtype=np.uint8))
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids, np.array([0.0, -0.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -10], np.float32)])
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_encode(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_e4m3_encode_saturates():
    assert O.e4m3_encode(np.array([1e6, -1e6, 464.0, 470.0])).tolist() == [0x7E, 0xFE, 0x7E, 0x7E]


@pytest.mark.parametrize("amax,e", [(448.0, 0), (448.0001, 1), (1.0, -8), (1.75, -8), (1.7500001, -7),
                                    (0.0, 0), (2.0 ** -140, -127)])
def test_ue8m0_exponent_cases(amax, e):
    assert O.ue8m0_exponent(amax) == e


def test_ue8m0_exponent_is_minimal_power_covering_amax():
    rng = np.random.default_rng(3)
    for amax in np.abs(rng.standard_normal(2000) * 10.0 ** rng.integers(-8, 8, 2000)):
        e = O.ue8m0_exponent(amax)
        assert 448.0 * 2.0 ** e >= amax and 448.0 * 2.0 ** (e - 1) < amax


def test_fp8_ds_mla_round_trip_exact_on_representable_values():
    """e4m3-representable values times a power-of-two block scale survive encode/decode bit-exactly."""
    rng = np.random.default_rng(4)
    repr_vals = O.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    row = np.zeros(576)
    for blk in range(8):
        e = int(rng.integers(-20, 5))
        seg = rng.choice(repr_vals, 64) * rng.choice([-1.0, 1.0], 64)
        seg[rng.integers(64)] = 448.0           # block amax fixes the exponent at e
        row[blk * 64:(blk + 1) * 64] = seg * 2.0 ** e
    row[512:] = O.bf16_decode(O.bf16_encode(rng.standard_normal(64)))
    rec = O.fp8_ds_mla_encode(row)
    assert rec.shape == (656,) and np.all(rec[648:] == 0)
    assert np.array_equal(O.fp8_ds_mla_decode(rec), row)


def test_fp8_ds_mla_error_bound():
    """A general row decodes within half an e4m3 ulp (relative 2^-4) of each element's block scale."""
    rng = np.random.default_rng(5)
    row = rng.standard_normal(576) * 0.1
    dec = O.fp8_ds_mla_decode(O.fp8_ds_mla_encode(row))
    for blk in range(8):
        seg = slice(blk * 64, (blk + 1) * 64)
        e = O.ue8m0_exponent(np.abs(row[seg]).max())
        # e4m3 spacing at magnitude a is <= a * 2^-3 (normal) or 2^-9 (subnormal)
        tol = np.maximum(np.abs(row[seg]) * 2.0 ** -4, 2.0 ** -10 * 2.0 ** e) * (1 + 1e-12)
        assert np.all(np.abs(dec[seg] - row[seg]) <= tol)
    assert np.allclose(dec[512:], row[512:], rtol=2 ** -8, atol=0)


def test_i8_rowscale_exact_for_scale_multiples():
    """A row of integer multiples of its own scale gets its integers back as codes."""
    q = np.concatenate([np.arange(-127, 1), np.arange(1, 128)[::-1][:1]])[:128].astype(np.float32)
    q[5] = 127
    for s in (0.003, 1.7e-5, 2.5):
        row = (q * np.float32(s)).astype(np.float32)
        rec = O.i8_rowscale_encode(row)
        assert rec.shape == (132,)
        assert np.array_equal(rec[:128].view(np.int8).astype(np.float32), q)
        scale = rec[128:].view(np.float32)[0]
        assert np.array_equal(O.i8_rowscale_decode(rec), q.astype(np.float64) * np.float64(scale))
    assert np.all(O.i8_rowscale_encode(np.zeros(128, np.float32))[:128] == 0)
    g = golden("indexer_fp8_row_bytes")
    assert O.i8_rowscale_encode(np.ones(g["head_dim"], np.float32)).shape[0] == g["bytes"]


# ------------------------------------------------------------------------------------------------
# counts and worked numbers from the pages
# ------------------------------------------------------------------------------------------------

def test_worked_prefill_count():
    g = golden("prefill_100_tokens_c4")
    assert O.n_compressed(g["tokens"] - 1, g["ratio"]) == g["entries"]


def test_worked_token_500000():
    g = golden("token_500000_block_position")
    assert g["position"] // g["ratio"] == g["block_position"]
    assert O.n_compressed(g["position"], g["ratio"]) == g["block_position"]
    g = golden("token_500000_rows_attended")
    w = O.window_positions(g["position"], g["window"])
    assert len(w) == g["window_rows"] and w[-1] == g["position"]
    assert len(w) + min(g["topk"], O.n_compressed(g["position"], g["ratio"])) == g["rows"]


def test_worked_swa_only_and_decode_101():
    g = golden("swa_only_layer")
    assert len(O.window_positions(g["position"], g["window"])) == g["rows"]
    assert O.n_compressed(g["position"], 0) == 0
    g = golden("decode_token_101")
    assert O.n_compressed(g["tokens"] - 1, g["ratio"]) == g["entries"] != g["page_claim"]


def test_counts_are_floor_len_over_ratio():
    for r in (4, 128):
        for length in range(1, 1000):
            assert O.n_compressed(length - 1, r) == math.floor(length / r)
            assert O.emits(length - 1, r) == (length % r == 0)
    assert list(O.window_positions(5)) == list(range(6))


# ------------------------------------------------------------------------------------------------
# indexer and top-k
# ------------------------------------------------------------------------------------------------

def test_indexer_score_brute_force_tiny():
    rng = np.random.default_rng(6)
    Ih, d, n = 3, 5, 7
    q, w, k = rng.standard_normal((Ih, d)), rng.standard_normal(Ih), rng.standard_normal((n, d))
    got = O.indexer_scores(q, w, k)
    for j in range(n):
        s = math.fsum(w[h] * max(0.0, math.fsum(q[h, i] * k[j, i] for i in range(d))) for h in range(Ih))
        assert got[j] == np.float32(s)


def test_indexer_single_head_unit_weight_is_relu_dot():
    rng = np.random.default_rng(7)
    q, k = rng.standard_normal((1, 16)), rng.standard_normal((40, 16))
    got = O.indexer_scores(q, np.ones(1), k).astype(np.float64)
    dots = np.array([float(np.dot(q[0], kj)) for kj in k])
    assert np.allclose(got, np.where(dots > 0, dots, 0.0), rtol=1e-7, atol=0)
    assert np.all(got[dots <= 0] == 0)


def test_indexer_negative_weight_lowers_scores_and_permutes():
    rng = np.random.default_rng(8)
    q, w, k = rng.standard_normal((4, 8)), rng.standard_normal(4), rng.standard_normal((30, 8))
    w[0] = -0.5
    s0 = O.indexer_scores(q, w, k)
    w2 = w.copy()
    w2[0] = -1.5
    assert np.all(O.indexer_scores(q, w2, k) <= s0)
    perm = rng.permutation(30)
    assert np.array_equal(O.indexer_scores(q, w, k[perm]), s0[perm])


def test_indexer_int8_keys_equal_decoded_keys():
    rng = np.random.default_rng(9)
    recs = np.stack([O.i8_rowscale_encode(rng.standard_normal(128).astype(np.float32) * 0.1) for _ in range(20)])
    keys = O.decode_rows(recs, O.I8_ROWSCALE)
    q, w = rng.standard_normal((2, 128)), rng.standard_normal(2)
    q8 = np.ascontiguousarray(recs[:, :128]).view(np.int8).astype(np.float64)
    sc = np.ascontiguousarray(recs[:, 128:]).view(np.float32)[:, 0].astype(np.float64)
    direct = np.array([sum(w[h] * max(0.0, float(q[h] @ q8[j]) * sc[j]) for h in range(2)) for j in range(20)])
    assert np.allclose(O.indexer_scores(q, w, keys), direct, rtol=1e-6, atol=0)


def test_topk_is_best_k_by_score_then_index_brute_force():
    rng = np.random.default_rng(10)
    for trial in range(200):
        n = int(rng.integers(0, 12))
        k = int(rng.integers(1, 8))
        s = rng.integers(-3, 4, n).astype(np.float32)        # many exact ties
        out = O.topk_select(s, k)
        m = min(n, k)
        chosen = out[:m]
        assert np.all(out[m:] == -1) and len(set(chosen.tolist())) == m
        rest = [j for j in range(n) if j not in set(chosen.tolist())]
        for c in chosen:
            for r in rest:
                assert s[c] > s[r] or (s[c] == s[r] and c < r)


def test_topk_short_context_selects_everything():
    s = np.random.default_rng(11).standard_normal(10).astype(np.float32)
    out = O.topk_select(s, 16)
    assert sorted(out[:10].tolist()) == list(range(10)) and np.all(out[10:] == -1)
    assert np.all(O.topk_select(np.zeros(0, np.float32), 4) == -1)


# ------------------------------------------------------------------------------------------------
# attention
# ------------------------------------------------------------------------------------------------

def _paged_setup(rng, rows, dtype=O.F32, shuffle=True):
    """Scatter explicit rows into a paged cache through a (shuffled) block table."""
    n = rows.shape[0]
    npg = (n + 63) // 64
    perm = rng.permutation(npg) if shuffle else np.arange(npg)
    cache = np.zeros((npg, 64, 576), np.float32)
    for j in range(n):
        cache[perm[j // 64], j % 64] = rows[j]
    return cache, perm.astype(np.int32)


def _brute_attention(q, rows, sink, scale):
    z = scale * (q @ rows.T)
    if sink is not None:
        z = np.concatenate([z, np.asarray(sink)[:, None]], axis=1)
        v = np.concatenate([rows[:, :512], np.zeros((1, 512))], axis=0)
    else:
        v = rows[:, :512]
    return softmax(z, axis=1) @ v, logsumexp(z, axis=1)


@pytest.mark.parametrize("sparse", [False, True])
def test_attention_equals_brute_force_over_concatenated_rows(sparse):
    rng = np.random.default_rng(12)
    H, ratio, p = 8, 128, 128 * 9 + 40            # n_c = 9
    swa_src = rng.standard_normal((p + 1, 576)).astype(np.float32) * 0.3
    main_src = rng.standard_normal((9, 576)).astype(np.float32) * 0.3
    swa_cache, swa_bt = _paged_setup(rng, swa_src)
    main_cache, main_bt = _paged_setup(rng, main_src)
    topk = np.array([7, 2, 5, -1, -1], np.int32) if sparse else None
    rows = O.attention_rows(p, 0, O.Paged(swa_cache), [swa_bt], O.F32, O.Paged(main_cache), [main_bt], ratio,
                            topk)
    sel = [7, 2, 5] if sparse else list(range(9))
    explicit = np.concatenate([swa_src[p - 127:p + 1], main_src[sel]]).astype(np.float64)
    assert np.array_equal(rows, explicit)
    q = rng.standard_normal((H, 576))
    sink = rng.standard_normal(H)
    out, lse = O.mqa_decode(q, rows, sink, 576 ** -0.5)
    bo, bl = _brute_attention(q, explicit, sink, 576 ** -0.5)
    assert np.allclose(out, bo, rtol=1e-12, atol=1e-14) and np.allclose(lse, bl, rtol=1e-12)


def test_sparse_with_k_at_least_nc_equals_dense():
    rng = np.random.default_rng(13)
    p, ratio = 4 * 37 + 3, 4
    nc = O.n_compressed(p, ratio)
    swa_cache, swa_bt = _paged_setup(rng, rng.standard_normal((p + 1, 576)).astype(np.float32))
    main_cache, main_bt = _paged_setup(rng, rng.standard_normal((nc, 576)).astype(np.float32))
    args = (p, 0, O.Paged(swa_cache), [swa_bt], O.F32, O.Paged(main_cache), [main_bt], ratio)
    scores = rng.standard_normal(nc).astype(np.float32)
    topk = np.sort(O.topk_select(scores, nc + 20)[:nc])
    topk = np.concatenate([topk, -np.ones(20, np.int32)])
    q = rng.standard_normal((4, 576))
    d = O.mqa_decode(q, O.attention_rows(*args, None), None, 0.05)
    s = O.mqa_decode(q, O.attention_rows(*args, topk), None, 0.05)
    assert np.array_equal(d[0], s[0]) and np.array_equal(d[1], s[1])


def test_sink_minus_inf_is_no_sink_and_closed_form():
    rng = np.random.default_rng(14)
    q, rows = rng.standard_normal((6, 576)), rng.standard_normal((50, 576))
    o0, l0 = O.mqa_decode(q, rows, None, 0.04)
    oi, li = O.mqa_decode(q, rows, np.full(6, -np.inf), 0.04)
    assert np.array_equal(o0, oi) and np.array_equal(l0, li)
    sink = rng.standard_normal(6) * 3
    o1, l1 = O.mqa_decode(q, rows, sink, 0.04)
    # the sink only enlarges the denominator: o_sink = o / (1 + e^(sink - lse)), lse_sink = logaddexp
    assert np.allclose(o1, o0 / (1.0 + np.exp(sink - l0))[:, None], rtol=1e-12)
    assert np.allclose(l1, np.logaddexp(l0, sink), rtol=1e-13)


def test_single_row_returns_its_value_half():
    rng = np.random.default_rng(15)
    row = rng.standard_normal((1, 576))
    out, lse = O.mqa_decode(rng.standard_normal((3, 576)), row, None, 0.1)
    assert np.allclose(out, np.repeat(row[:, :512], 3, 0), rtol=1e-15)


def test_block_table_permutation_leaves_output_bit_identical():
    rng = np.random.default_rng(16)
    p = 300
    src = rng.standard_normal((p + 1, 576)).astype(np.float32)
    c1, bt1 = _paged_setup(np.random.default_rng(1), src)
    c2, bt2 = _paged_setup(np.random.default_rng(2), src)
    assert not np.array_equal(bt1, bt2)
    q = rng.standard_normal((4, 576))
    r1 = O.attention_rows(p, 0, O.Paged(c1), [bt1], O.F32, None, None, 0)
    r2 = O.attention_rows(p, 0, O.Paged(c2), [bt2], O.F32, None, None, 0)
    assert np.array_equal(O.mqa_decode(q, r1, None, 0.1)[0], O.mqa_decode(q, r2, None, 0.1)[0])


def test_split_merge_equals_unsplit():
    rng = np.random.default_rng(17)
    q, rows, sink = rng.standard_normal((5, 576)), rng.standard_normal((300, 576)), rng.standard_normal(5)
    full_o, full_l = O.mqa_decode(q, rows, sink, 0.05)
    for cuts in ([0, 300], [0, 64, 128, 300], [0, 1, 2, 299, 300], list(range(0, 301, 37)) + [300]):
        cuts = sorted(set(cuts))
        parts = [O.mqa_partial(q, rows[a:b], 0.05) for a, b in zip(cuts[:-1], cuts[1:])]
        o, l = O.merge_partials([x[0] for x in parts], [x[1] for x in parts], sink)
        assert np.allclose(o, full_o, rtol=1e-12, atol=1e-15) and np.allclose(l, full_l, rtol=1e-13)


# ------------------------------------------------------------------------------------------------
# compressor
# ------------------------------------------------------------------------------------------------

def _state_from_rows(kv_rows, sc_rows, ratio, coff, series):
    """State ring with rows at given positions: {pos: (kv, score)} written into `series`."""
    st = np.zeros((coff * ratio, 2 * coff * 576), np.float32)
    for pos in kv_rows:
        s = pos % (coff * ratio)
        st[s, series[pos] * 576:(series[pos] + 1) * 576] = kv_rows[pos]
        st[s, coff * 576 + series[pos] * 576:coff * 576 + (series[pos] + 1) * 576] = sc_rows[pos]
    return st


@pytest.mark.parametrize("ratio,coff", [(128, 1), (4, 2)])
def test_fold_equal_scores_is_mean(ratio, coff):
    rng = np.random.default_rng(18)
    st = rng.standard_normal((coff * ratio, 2 * coff * 576)).astype(np.float32)
    st[:, coff * 576:] = 0.7                               # every gate score equal
    j = 5
    e = O.fold_entry(*O.fold_group(st, j, ratio, coff))
    cur = [st[q % (coff * ratio), :576] for q in range(j * ratio, (j + 1) * ratio)]
    prev = [st[q % (coff * ratio), 576:1152] for q in range((j - 1) * ratio, j * ratio)] if coff == 2 else []
    assert np.allclose(e, np.mean(np.array(cur + prev, np.float64), axis=0), rtol=1e-12, atol=1e-15)
    if coff == 2:
        e0 = O.fold_entry(*O.fold_group(st, 0, ratio, coff))
        assert np.allclose(e0, np.mean(np.array([st[q, :576] for q in range(4)], np.float64), 0), rtol=1e-12)


@pytest.mark.parametrize("ratio,coff", [(128, 1), (4, 2)])
def test_fold_dominant_score_selects_that_row_per_channel(ratio, coff):
    rng = np.random.default_rng(19)
    j = 3
    st = rng.standard_normal((coff * ratio, 2 * coff * 576)).astype(np.float32)
    kv, sc = O.fold_group(st, j, ratio, coff)
    n = kv.shape[0]
    pick = rng.integers(0, n, 576)
    # plant +1e4 in channel c at group row pick[c] (rows: series A current block, then series B previous)
    for c in range(576):
        i = pick[c]
        pos = j * ratio + i if i < ratio else (j - 1) * ratio + (i - ratio)
        col = coff * 576 + c + (576 if i >= ratio else 0)
        st[pos % (coff * ratio), col] = 1e4
    kv, sc = O.fold_group(st, j, ratio, coff)
    e = O.fold_entry(kv, sc)
    assert np.allclose(e, kv[pick, np.arange(576)], rtol=1e-12, atol=1e-12)


def test_c4_overlap_uses_series_b_of_previous_block():
    ratio, coff = 4, 2
    st = np.zeros((8, 4 * 576), np.float32)
    j = 6
    for q in range(j * 4, j * 4 + 4):
        st[q % 8, :576] = 1.0          # series A of the current block
        st[q % 8, 576:1152] = 99.0     # series B of the current block: not part of entry j
    for q in range((j - 1) * 4, j * 4):
        st[q % 8, :576] = -50.0        # series A of the previous block: not part of entry j
        st[q % 8, 576:1152] = 2.0      # series B of the previous block
    e = O.fold_entry(*O.fold_group(st, j, ratio, coff))
    assert np.allclose(e, 1.5)


def test_state_row_adds_ape_to_score_half_only():
    rng = np.random.default_rng(20)
    ks = rng.standard_normal(4 * 576).astype(np.float32)
    ape = rng.standard_normal((4, 2 * 576)).astype(np.float32)
    row = O.state_row(ks, 4 * 9 + 2, 4, 2, ape)
    assert np.array_equal(row[:1152], ks[:1152])
    assert np.array_equal(row[1152:], (ks[1152:] + ape[2]).astype(np.float32))


def test_rms_norm_invariants():
    rng = np.random.default_rng(21)
    x = rng.standard_normal(576) * 3
    y = O.rms_norm(x, np.ones(576), 0.0)
    assert abs(np.sqrt(np.mean(y * y)) - 1.0) < 1e-12
    assert np.allclose(O.rms_norm(7.5 * x, np.ones(576), 0.0), y, rtol=1e-12)
    w = rng.standard_normal(576)
    assert np.allclose(O.rms_norm(x, w, 0.0), y * w, rtol=1e-12)
    # eps enters under the root: tiny vectors are damped, not blown up
    assert np.all(np.abs(O.rms_norm(1e-6 * x, np.ones(576), 1e-6)) < np.abs(y))


def test_rope_matches_complex_rotation_and_identity_at_zero():
    from dsv4_inputs import rope_table
    tab = rope_table(5000)
    rng = np.random.default_rng(22)
    x = rng.standard_normal(64)
    assert np.array_equal(O.rope_gptj(x, tab[0, :32].astype(np.float64), tab[0, 32:].astype(np.float64)), x)
    for pos in (1, 17, 4096, 4999):
        c, s = tab[pos, :32].astype(np.float64), tab[pos, 32:].astype(np.float64)
        z = (x[0::2] + 1j * x[1::2]) * (c + 1j * s)
        y = O.rope_gptj(x, c, s)
        assert np.allclose(y[0::2], z.real, rtol=1e-14, atol=1e-15) and np.allclose(y[1::2], z.imag, rtol=1e-14,
                                                                                       atol=1e-15)
        assert np.allclose(np.hypot(y[0::2], y[1::2]), np.hypot(x[0::2], x[1::2]), rtol=1e-6)


def test_compress_update_emits_exactly_at_group_ends():
    rng = np.random.default_rng(23)
    ratio, coff, B = 4, 2, 1
    state = np.zeros((B, 8, 4 * 576), np.float32)
    main = O.Paged(np.zeros((2, 64, 576), np.float32))
    bt = np.array([[1, 0]], np.int32)
    from dsv4_inputs import rope_table
    tab = rope_table(200)
    emitted, keyed = [], []
    idx = O.Paged(np.zeros((2, 64, 132), np.uint8))
    ik = {"wk": rng.standard_normal((128, 576)) * 0.05, "kn_w": np.ones(128), "eps": 1e-6, "cache": idx,
          "bt": np.array([[0, 1]], np.int32), "dtype": O.I8_ROWSCALE}
    for p in range(0, 23):
        ks = rng.standard_normal((1, 4 * 576)).astype(np.float32)
        new_state, ent, keys = O.compress_update(state, ks, np.array([p], np.int32), 1, ratio, coff, None,
                                                 np.ones(576, np.float32), 1e-6, tab, main, bt, O.F32, ik=ik)
        state = new_state[0][None]
        emitted += list(ent.keys())
        keyed += list(keys.keys())
    assert [j for (_, j) in emitted] == list(range(O.n_compressed(22, ratio)))
    assert set(main.written.keys()) == {(1, j) for j in range(5)}
    assert keyed == emitted                                  # one index key per emitted entry
    assert set(idx.written.keys()) == {(0, j) for j in range(5)}


def test_kv_insert_slot_mapping_and_skip():
    rng = np.random.default_rng(24)
    cache = np.zeros((3, 64, 576), np.float32)
    sw = O.Paged(cache)
    kv = rng.standard_normal((3, 576)).astype(np.float32)
    O.kv_insert(sw, kv, O.F32, np.array([130, -1, 5]), O.F32)
    assert set(sw.written) == {(2, 2), (0, 5)}
    assert np.array_equal(sw.written[(2, 2)], kv[0]) and np.array_equal(sw.written[(0, 5)], kv[2])


# ------------------------------------------------------------------------------------------------
# MXFP4 index keys: E2M1 elements, one UE8M0 exponent per 32
# ------------------------------------------------------------------------------------------------

E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]   # the format's eight magnitudes (sign bit 3)


def test_e2m1_decode_all_codes():
    got = O.e2m1_decode(np.arange(16))
    want = np.array(E2M1_TABLE + [-v for v in E2M1_TABLE])
    assert np.array_equal(got, want)


def test_e2m1_encode_nearest_ties_to_even_brute_force():
    rng = np.random.default_rng(31)
    mids = [(a + b) / 2 for a, b in zip(E2M1_TABLE[:-1], E2M1_TABLE[1:])]
    x = np.concatenate([rng.uniform(-6.5, 6.5, 20000), mids, [-m for m in mids], [0.0, 6.0, -6.0, 100.0, -100.0]])
    got = O.e2m1_decode(O.e2m1_encode(x))
    for v, g in zip(x, got):
        a = min(abs(v), 6.0)
        d = [abs(a - t) for t in E2M1_TABLE]
        best = min(d)
        cands = [k for k in range(8) if d[k] == best]
        k = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]   # tie: even code
        assert g == (E2M1_TABLE[k] if v >= 0 else -E2M1_TABLE[k]), v


@pytest.mark.parametrize("amax,e", [(6.0, 0), (6.0001, 1), (3.0, -1), (1.0, -2), (0.75, -3), (0.0, 0)])
def test_mxfp4_exponent_cases(amax, e):
    assert O.mxfp4_exponent(amax) == e


def test_mxfp4_record_layout_round_trip_and_bound():
    rng = np.random.default_rng(32)
    # representable rows: E2M1 values times one power of two per 32-element block round-trip exactly
    codes = rng.integers(0, 16, 128)
    exps = rng.integers(-10, 10, 4)
    x = O.e2m1_decode(codes) * np.repeat(np.exp2(exps.astype(np.float64)), 32)
    rec = O.mxfp4_encode(x)
    assert rec.shape == (68,)                       # 128 / 2 + 128 / 32 bytes
    assert np.array_equal(O.mxfp4_decode(rec), x)
    # element 2i in the low nibble of byte i, block exponents after the codes
    y = np.zeros(128)
    y[0], y[1] = 1.5 * 2.0 ** -2, -6.0 * 2.0 ** -2  # block 0: max 1.5 -> e = -2, codes 3 and 15
    rec = O.mxfp4_encode(y)
    assert rec[0] == 0x03 | (0x0F << 4) and rec[64] == 125 and rec[65] == 127
    # any row: within half an E2M1 step (0.5 below 2, 1 in [2, 4), 2 in [4, 6]) at its block's scale
    z = rng.standard_normal(128) * 3.0
    dec = O.mxfp4_decode(O.mxfp4_encode(z))
    for blk in range(4):
        seg = slice(32 * blk, 32 * blk + 32)
        s = 2.0 ** O.mxfp4_exponent(np.max(np.abs(z[seg])))
        a = np.abs(z[seg]) / s
        step = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
        assert np.all(np.abs(dec[seg] - z[seg]) <= step / 2 * s + 1e-12)


def test_mxfp4_index_key_recall_against_fp32_keys():
    """Top-k over MXFP4-quantised keys against top-k over the fp32 keys they came from: the set the
    quantised cache selects, measured as recall (the pages report 0.3% of entries missed on real
    keys; these are Gaussian keys and queries, 64 heads x 128 dims, k = 512 of 16384)."""
    rng = np.random.default_rng(33)
    n, k, heads, d = 16384, 512, 64, 128
    keys = (rng.standard_normal((n, d)) * 0.1).astype(np.float32)
    q = (rng.standard_normal((heads, d)) * 0.1).astype(np.float32)
    w = (rng.standard_normal(heads) * 0.1).astype(np.float32)
    ref = set(O.topk_select(O.indexer_scores(q, w, keys), k).tolist())
    quant = O.decode_rows(np.stack([O.mxfp4_encode(r) for r in keys]), O.MXFP4)
    got = set(O.topk_select(O.indexer_scores(q, w, quant), k).tolist())
    recall = len(ref & got) / k
    assert recall >= 0.85, recall


# ------------------------------------------------------------------------------------------------
# two-level candidate filtering
# ------------------------------------------------------------------------------------------------

def test_candidate_blocks_brute_force():
    rng = np.random.default_rng(41)
    for n, block, m in [(1000, 64, 5), (4096, 512, 3), (300, 128, 8), (130, 128, 1)]:
        s = rng.integers(-5, 6, n).astype(np.float32)           # many ties between block maxima
        got = O.candidate_blocks(s, block, m)
        nblk = -(-n // block)
        best = [max(s[b * block:(b + 1) * block]) for b in range(nblk)]
        rank = sorted(range(nblk), key=lambda b: (-best[b], b))
        want = sorted(rank[:min(m, nblk)])
        assert got[:len(want)].tolist() == want and np.all(got[len(want):] == -1)


def test_masked_topk_brute_force_and_reductions():
    rng = np.random.default_rng(42)
    s = rng.standard_normal(5000).astype(np.float32)
    cand = np.array([1, 4, 7, -1], np.int32)
    got = O.masked_topk(s, 100, cand, 512)
    inc = [j for j in range(5000) if j // 512 in (1, 4, 7)]
    want = sorted(inc, key=lambda j: (-float(s[j]), j))[:100]
    assert set(got.tolist()) == set(want)
    # every block listed: plain top-k; fewer included entries than k: all of them
    assert set(O.masked_topk(s, 100, np.arange(10), 512).tolist()) == set(O.topk_select(s, 100).tolist())
    few = O.masked_topk(s[:700], 600, np.array([1], np.int32), 512)
    assert sorted(few[:188].tolist()) == list(range(512, 700)) and np.all(few[188:] == -1)
    assert np.all(O.masked_topk(s, 10, np.array([-1, -1]), 512) == -1)


def test_listed_blocks_is_the_increasing_run():
    assert O.listed_blocks([2, 5, 9, -1]) == [2, 5, 9]
    assert O.listed_blocks([2, 5, 5, 9]) == [2, 5]        # an equal entry ends the run
    assert O.listed_blocks([4, 1, 7]) == [4]              # so does a smaller one
    assert O.listed_blocks([-1, 3]) == [] and O.listed_blocks([]) == []
    s = np.arange(1000, dtype=np.float32)
    got = O.masked_topk(s, 10, np.array([1, 0, 2]), 128)   # only block 1 is listed
    assert sorted(got.tolist()) == list(range(246, 256))


def test_consumer_token_within_topk_takes_every_entry():
    # a consumer token whose entries all fit in the top-k selects all of them whatever its list says;
    # one with more entries keeps only its listed blocks
    import dataclasses
    cfg = dataclasses.replace(I.SMALL_CONFIGS["small_c4_cand"], B=2, explicit_lens=(400, 2200))
    st = I.make_step(cfg)
    st.cand_in[:] = -1
    st.cand_in[:, 0] = 0
    res = O.decode_step(st)
    n0 = 400 // 4
    assert sorted(res["topk"][0][:n0].tolist()) == list(range(n0)) and np.all(res["topk"][0][n0:] == -1)
    n1 = 2200 // 4                                   # 550 > 512: block 0 (entries 0..549 with 1024-entry blocks)
    assert sorted(res["topk"][1][res["topk"][1] >= 0].tolist()) == sorted(
        O.topk_select(res["scores"][1], cfg.topk)[:512].tolist())
    st.cand_in[1, 0] = 1                              # a block past the token's entries: nothing is listed
    res = O.decode_step(st)
    assert np.all(res["topk"][1] == -1) and n1 > cfg.topk
