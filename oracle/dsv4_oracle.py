"""Plain, slow CPU oracle of the DeepSeek-V4 hybrid compressed-attention decode step.

TEST INFRASTRUCTURE: only tests/, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg import this module.  It shares no code with the CUDA path and
imports nothing from it.

Arithmetic is numpy float64 on values first decoded exactly from their stored
form, except where the pages fix a precision: the compressor state is stored as
float32 (state + APE is an fp32 add), and the indexer score is an fp32 quantity
(the fp64 score is rounded to fp32 before ranking).  Quantisation decisions
(bf16 / e4m3 rounding, the UE8M0 block exponent) are written so that they do not
depend on the precision they are evaluated in.

Sources (page title, section):
  [MAP]    "DeepSeek V4 Attention: Code Reading Map"
  [ASCEND] "DeepSeek-V4 Inference on Ascend: The DSA Serving Stack in vllm-ascend"
  [API]    "vllm.models.deepseek_v41.attention" (API docs with source)

Readings taken where the pages leave a step open (each also listed in the design notes):
  * latent row = 576 dims: 512 no-pe + 64 rope; value = the first 512 dims (shared-KV MLA).
  * indexer score s_j = sum_h w_h * ReLU(q_h . k_j), fp32; softmax_scale * n_head^-0.5 is
    assumed folded into w by the caller.
  * compression gate scores are per channel; the softmax runs over the group's tokens per channel.
  * APE [ratio, coff*576] is added to the score half of each token's state row on store.
  * c4 overlap group of entry j = tokens [4j, 4j+4) through series A plus tokens [4j-4, 4j)
    through series B; for j = 0 only series A's four tokens.
  * the compressed entry j is RoPE-rotated (GPT-J pairs on dims 512..575) at position j*ratio.
  * the sliding window of a query at position p is positions max(0, p-127) .. p; compressed
    rows are not de-duplicated against it.
  * a query at position p sees n_c(p) = floor((p+1)/ratio) compressed entries.
  * the sink is one extra logit in the softmax denominator; -inf means no sink.
  * fp8_ds_mla record at 576 dims = 656 bytes: 512 e4m3fn | 64 bf16 rope | 8 UE8M0 bytes | 8 zero.
  * the UE8M0 exponent of a 64-dim block is the smallest e with 448 * 2^e >= amax (0 when amax = 0).
  * int8 indexer key record = 128 int8 + little-endian fp32 scale (132 bytes); k = q8 * scale.
  * MXFP4 indexer key record = d/2 bytes of E2M1 pairs (element 2i in the low nibble) + one UE8M0
    byte per 32 elements (68 bytes for d = 128); the block exponent is the smallest e with
    6 * 2^e >= the block's max |x| (never saturates); queries stay bf16.

Parity unpinned (model-fidelity readings the pages do not fix, so nothing outside the
oracle can confirm them): the APE target, the RoPE position of compressed entries, the c4
overlap row set, the gate granularity, the 656-byte record layout and the softmax scale.
"""
from __future__ import annotations

import numpy as np

D = 576
DV = 512
D_NOPE = 512
D_ROPE = 64
WINDOW = 128
PAGE = 64
FP8_BLOCK = 64
FP8_DS_MLA_BYTES = 656
E4M3_MAX = 448.0

F32, BF16, FP8_DS_MLA, I8_ROWSCALE, MXFP4 = 0, 1, 2, 3, 4
E2M1_MAX = 6.0
MXFP4_BLOCK = 32


# ----------------------------------------------------------------------------------------------
# Element codecs
# ----------------------------------------------------------------------------------------------

def bf16_decode(bits) -> np.ndarray:
    """bf16 bit patterns -> float64: a bf16 value is the upper half of an fp32 word."""
    b = np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def _round_to_grid(x: np.ndarray, mant_bits: int, min_exp: int) -> np.ndarray:
    """Round-to-nearest-even onto a binary float grid with `mant_bits` stored mantissa bits and
    smallest normal exponent `min_exp` (subnormals keep the spacing of the smallest binade)."""
    x = np.asarray(x, np.float64)
    out = x.copy()                        # zeros keep their sign
    nz = x != 0
    _, ex = np.frexp(x[nz])               # |x| = m * 2^ex, m in [0.5, 1)
    e = np.maximum(ex - 1, min_exp)       # binade exponent, clamped for subnormals
    ulp = np.ldexp(1.0, e - mant_bits)
    out[nz] = np.rint(x[nz] / ulp) * ulp  # np.rint rounds half to even; x/ulp is exact
    return out


def bf16_encode(x) -> np.ndarray:
    """Value -> bf16 bits, round to nearest even (8 significant bits, fp32 exponent range)."""
    v = _round_to_grid(x, 7, -126).astype(np.float32)
    return (v.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def e4m3_decode(code) -> np.ndarray:
    """e4m3fn byte -> float64: 1 sign, 4 exponent (bias 7), 3 mantissa bits; no inf,
    exponent 15 with mantissa 7 is NaN, exponent 0 is subnormal (m * 2^-9)."""
    c = np.asarray(code, np.uint8).astype(np.int64)
    s = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    v = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return s * v


def e4m3_encode(x) -> np.ndarray:
    """Value -> e4m3fn byte, round to nearest even, saturating to +-448 (satfinite)."""
    x = np.asarray(x, np.float64)
    v = np.clip(_round_to_grid(x, 3, -6), -E4M3_MAX, E4M3_MAX)
    a = np.abs(v)
    sign = (v < 0) | ((v == 0) & np.signbit(x))
    code = np.zeros(a.shape, np.int64)
    sub = a < 2.0 ** -6
    code[sub] = np.rint(a[sub] / 2.0 ** -9).astype(np.int64)      # exponent field 0
    nrm = ~sub
    _, ex = np.frexp(a[nrm])
    e = ex - 1
    m = np.rint((a[nrm] / np.exp2(e) - 1.0) * 8.0).astype(np.int64)
    code[nrm] = ((e + 7) << 3) | m
    return (code | (sign.astype(np.int64) << 7)).astype(np.uint8)


def ue8m0_exponent(amax: float) -> int:
    """Block exponent of UE8M0 scaling: the smallest integer e with 448 * 2^e >= amax
    ([MAP] "How Does Compression Actually Work?", step 6, "UE8M0 block scaling"),
    clamped to the byte's range [-127, 127]; 0 for an all-zero block."""
    amax = float(amax)
    if amax == 0.0:
        return 0
    e = int(np.ceil(np.log2(amax / E4M3_MAX)))
    while E4M3_MAX * 2.0 ** (e - 1) >= amax:
        e -= 1
    while E4M3_MAX * 2.0 ** e < amax:
        e += 1
    return max(-127, min(127, e))


def fp8_ds_mla_encode(row) -> np.ndarray:
    """One 576-dim row -> 656-byte fp8_ds_mla record ([MAP] "How Does Compression Actually Work?"
    steps 6-7; [API] DeepseekV4Attention, "fp8_ds_mla is UE8M0 block-scaled fp8 packed as uint8"):
    dims 0..511 as e4m3fn with one power-of-two scale per 64-dim block, dims 512..575 as bf16."""
    row = np.asarray(row, np.float64)
    rec = np.zeros(FP8_DS_MLA_BYTES, np.uint8)
    for blk in range(D_NOPE // FP8_BLOCK):
        seg = row[blk * FP8_BLOCK:(blk + 1) * FP8_BLOCK]
        e = ue8m0_exponent(np.max(np.abs(seg)))
        rec[blk * FP8_BLOCK:(blk + 1) * FP8_BLOCK] = e4m3_encode(seg / 2.0 ** e)
        rec[640 + blk] = e + 127
    rec[512:640] = bf16_encode(row[D_NOPE:]).view(np.uint8)
    return rec


def fp8_ds_mla_decode(rec) -> np.ndarray:
    """656-byte records [..., 656] -> float64 rows [..., 576]."""
    rec = np.asarray(rec, np.uint8)
    nope = e4m3_decode(rec[..., :512]).reshape(rec.shape[:-1] + (8, 64))
    scale = np.exp2(rec[..., 640:648].astype(np.float64) - 127.0)
    nope = (nope * scale[..., None]).reshape(rec.shape[:-1] + (512,))
    rope = bf16_decode(np.ascontiguousarray(rec[..., 512:640]).view(np.uint16))
    return np.concatenate([nope, rope], axis=-1)


def i8_rowscale_encode(row) -> np.ndarray:
    """d-dim key -> (d + 4)-byte record: int8 codes then the fp32 scale, the page's FP8 indexer
    row shape (d fp8 + 4-byte fp32 scale, [API] _indexer_k_cache_head_dim) with int8 codes
    ([ASCEND] "13. Hardware divergence": INT8 indexer cache).  scale = amax/127 in fp32
    (1 for an all-zero row), q = clamp(rne(x / scale), -127, 127), both in fp32."""
    x = np.asarray(row, np.float32)
    amax = np.float32(np.max(np.abs(x)))
    scale = np.float32(1.0) if amax == 0 else np.float32(amax / np.float32(127.0))
    q = np.clip(np.rint(x / scale), -127, 127).astype(np.int8)
    rec = np.zeros(x.shape[0] + 4, np.uint8)
    rec[:-4] = q.view(np.uint8)
    rec[-4:] = np.array([scale], np.float32).view(np.uint8)
    return rec


def i8_rowscale_decode(rec) -> np.ndarray:
    rec = np.asarray(rec, np.uint8)
    d = rec.shape[-1] - 4
    q = np.ascontiguousarray(rec[..., :d]).view(np.int8).astype(np.float64)
    s = np.ascontiguousarray(rec[..., d:]).view(np.float32).astype(np.float64)
    return q * s


def e2m1_decode(code) -> np.ndarray:
    """FP4 E2M1 code (low 4 bits) -> float64: 1 sign, 2 exponent (bias 1), 1 mantissa bit; exponent
    0 is subnormal (m * 0.5): magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6."""
    c = np.asarray(code, np.int64) & 0xF
    e, m = (c >> 1) & 3, c & 1
    mag = np.where(e == 0, 0.5 * m, (1.0 + 0.5 * m) * np.exp2(e - 1.0))
    return np.where(c >> 3, -mag, mag)


def e2m1_encode(x) -> np.ndarray:
    """Value -> E2M1 code, round to nearest even on the E2M1 grid, saturating to +-6."""
    x = np.asarray(x, np.float64)
    v = np.clip(_round_to_grid(x, 1, 0), -E2M1_MAX, E2M1_MAX)
    a = np.abs(v)
    code = np.zeros(a.shape, np.int64)
    sub = a < 1.0
    code[sub] = np.rint(a[sub] / 0.5).astype(np.int64)            # exponent field 0
    nrm = ~sub
    _, ex = np.frexp(a[nrm])
    e = ex - 1
    code[nrm] = ((e + 1) << 1) | np.rint((a[nrm] / np.exp2(e) - 1.0) * 2.0).astype(np.int64)
    sign = (v < 0) | ((v == 0) & np.signbit(x))
    return (code | (sign.astype(np.int64) << 3)).astype(np.uint8)


def mxfp4_exponent(amax: float) -> int:
    """Block exponent of an MXFP4 block: the smallest integer e with 6 * 2^e >= amax (the block's
    largest element never saturates), clamped to the UE8M0 byte's range; 0 for an all-zero block."""
    amax = float(amax)
    if amax == 0.0:
        return 0
    e = int(np.ceil(np.log2(amax / E2M1_MAX)))
    while E2M1_MAX * 2.0 ** (e - 1) >= amax:
        e -= 1
    while E2M1_MAX * 2.0 ** e < amax:
        e += 1
    return max(-127, min(127, e))


def mxfp4_encode(row) -> np.ndarray:
    """d-dim key -> MXFP4 record of d/2 + d/32 bytes ([API] _indexer_k_cache_head_dim: "MXFP4 stores
    two values per byte plus one UE8M0 byte per 32 values", 68 B for d = 128; [MAP] "What This Repo
    Is For": MXFP4 for indexer keys): E2M1 codes of x / 2^e (element 2i in the low nibble of byte i),
    then one byte e + 127 per 32-element block."""
    x = np.asarray(row, np.float64)
    d = x.shape[0]
    codes = np.zeros(d, np.uint8)
    scales = np.zeros(d // MXFP4_BLOCK, np.uint8)
    for blk in range(d // MXFP4_BLOCK):
        seg = slice(blk * MXFP4_BLOCK, (blk + 1) * MXFP4_BLOCK)
        e = mxfp4_exponent(np.max(np.abs(x[seg])))
        codes[seg] = e2m1_encode(x[seg] / 2.0 ** e)
        scales[blk] = e + 127
    packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    return np.concatenate([packed, scales])


def mxfp4_decode(rec) -> np.ndarray:
    """MXFP4 records [..., d/2 + d/32] -> float64 [..., d]."""
    rec = np.asarray(rec, np.uint8)
    nb = rec.shape[-1]
    d = nb * 32 // 17                                              # d/2 + d/32 = 17 d / 32
    packed = rec[..., :d // 2].astype(np.int64)
    codes = np.stack([packed & 0xF, packed >> 4], axis=-1).reshape(rec.shape[:-1] + (d,))
    vals = e2m1_decode(codes)
    scale = np.exp2(rec[..., d // 2:].astype(np.float64) - 127.0)
    return (vals.reshape(rec.shape[:-1] + (d // MXFP4_BLOCK, MXFP4_BLOCK)) * scale[..., None]).reshape(
        rec.shape[:-1] + (d,))


def decode_rows(stored, dtype: int) -> np.ndarray:
    """Stored rows in cache format `dtype` -> float64 values."""
    if dtype == F32:
        return np.asarray(stored, np.float32).astype(np.float64)
    if dtype == BF16:
        return bf16_decode(stored)
    if dtype == FP8_DS_MLA:
        return fp8_ds_mla_decode(stored)
    if dtype == I8_ROWSCALE:
        return i8_rowscale_decode(stored)
    if dtype == MXFP4:
        return mxfp4_decode(stored)
    raise ValueError(dtype)


def encode_row(x, dtype: int) -> np.ndarray:
    """One 576-dim value row -> its stored form in cache format `dtype`."""
    if dtype == F32:
        return np.asarray(x, np.float64).astype(np.float32)
    if dtype == BF16:
        return bf16_encode(x)
    if dtype == FP8_DS_MLA:
        return fp8_ds_mla_encode(x)
    raise ValueError(dtype)


# ----------------------------------------------------------------------------------------------
# Counts and row sets
# ----------------------------------------------------------------------------------------------

def n_compressed(p: int, ratio: int) -> int:
    """Compressed entries visible to a query at 0-based position p: one entry per completed
    group of `ratio` tokens ([MAP] "How Does Compression Actually Work?": an entry is made at
    every p with (p+1) % ratio == 0; [ASCEND] "8. The prefill path": 100 tokens -> 25 entries)."""
    return (int(p) + 1) // ratio if ratio > 0 else 0


def window_positions(p: int, window: int = WINDOW) -> np.ndarray:
    """Raw rows a query at p reads from the sliding-window cache: its own and the previous
    window-1 positions ([MAP] "Concrete Trace": token's own SWA entry + the last 127)."""
    return np.arange(max(0, int(p) - window + 1), int(p) + 1)


def emits(p: int, ratio: int) -> bool:
    return ratio > 0 and (int(p) + 1) % ratio == 0


# ----------------------------------------------------------------------------------------------
# Paged storage with a write overlay (the oracle never mutates its inputs)
# ----------------------------------------------------------------------------------------------

class Paged:
    """A paged cache [pages, PAGE, row] plus rows written during the step, keyed by (page, offset)."""

    def __init__(self, cache):
        self.cache = cache
        self.written = {}

    def put(self, page: int, off: int, row):
        self.written[(int(page), int(off))] = np.array(row, copy=True)

    def get(self, pages, offs) -> np.ndarray:
        pages = np.asarray(pages, np.int64)
        offs = np.asarray(offs, np.int64)
        if np.any(pages < 0) or np.any(pages >= self.cache.shape[0]):
            raise IndexError("block table names a page outside the cache")
        rows = self.cache[pages, offs].copy()
        if self.written:
            for i, (pg, of) in enumerate(zip(pages.tolist(), offs.tolist())):
                w = self.written.get((pg, of))
                if w is not None:
                    rows[i] = w
        return rows

    def logical(self, bt_row, idx) -> np.ndarray:
        """Rows at logical indices `idx` of one sequence through its block-table row."""
        idx = np.asarray(idx, np.int64)
        return self.get(np.asarray(bt_row)[idx // PAGE], idx % PAGE)


# ----------------------------------------------------------------------------------------------
# Step a1: SWA KV insert
# ----------------------------------------------------------------------------------------------

def rope_gptj(x, cos, sin) -> np.ndarray:
    """GPT-J (interleaved) rotary embedding on a 64-dim vector: pair i = dims (2i, 2i+1) rotates by
    angle i ([MAP] "Phase 2", default stream, "GPT-J style RoPE on the last 64 dims")."""
    x = np.asarray(x, np.float64)
    a, b = x[0::2], x[1::2]
    out = np.empty_like(x)
    out[0::2] = a * cos - b * sin
    out[1::2] = a * sin + b * cos
    return out


def qnorm_rope(q_t, p: int, cos_sin, norm_w, eps, apply_norm: bool, apply_rope: bool, h_pad: int) -> np.ndarray:
    """The query heads one token hands to the attention ([MAP] "Phase 2", default stream, item 2:
    per-head RMSNorm of every query head, GPT-J RoPE of the last 64 dims of each head; [API]
    DeepseekV4Attention._fused_qnorm_rope_kv_insert: the query is zero-padded to the backend's
    padded head count).  q_t [H, 576] values -> [h_pad, 576]: each head x becomes
    x / sqrt(mean(x^2) + eps) * w (w = 1 when norm_w is None) when apply_norm, then dims 512..575
    are rotated by the cos/sin row of position p when apply_rope; heads H .. h_pad-1 are zero."""
    q = np.asarray(q_t, np.float64)
    H = q.shape[0]
    out = np.zeros((h_pad, D), np.float64)
    w = np.ones(D) if norm_w is None else np.asarray(norm_w, np.float64)
    cs = np.asarray(cos_sin[int(p)], np.float64) if apply_rope else None
    for h in range(H):
        x = rms_norm(q[h], w, eps) if apply_norm else q[h].copy()
        if apply_rope:
            x[D_NOPE:] = rope_gptj(x[D_NOPE:], cs[:32], cs[32:])
        out[h] = x
    return out


def kv_insert(swa: Paged, kv_new, kv_dtype: int, slot_mapping, cache_dtype: int,
              positions=None, cos_sin=None):
    """Write each token's latent row into the paged SWA cache at its slot ([MAP] "4.
    _fused_qnorm_rope_kv_insert() - Where SWA Happens"; [API] _fused_qnorm_rope_kv_insert):
    optional GPT-J RoPE of dims 512..575 at the token position, then encode; slot -1 skips."""
    vals = decode_rows(kv_new, kv_dtype)
    for t, slot in enumerate(np.asarray(slot_mapping, np.int64)):
        if slot < 0:
            continue
        row = vals[t].copy()
        if cos_sin is not None:
            cs = np.asarray(cos_sin[int(positions[t])], np.float64)
            row[D_NOPE:] = rope_gptj(row[D_NOPE:], cs[:32], cs[32:])
        swa.put(slot // PAGE, slot % PAGE, encode_row(row, cache_dtype))


# ----------------------------------------------------------------------------------------------
# Step a2: compressor state update + fold
# ----------------------------------------------------------------------------------------------

def rms_norm(x, w, eps) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * w ([MAP] "How Does Compression Actually Work?", step 4)."""
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x) + eps) * np.asarray(w, np.float64)


def state_row(kv_score_t, p: int, ratio: int, coff: int, ape) -> np.ndarray:
    """The fp32 state row a token stores ([MAP] "What Are the Gate Scores?": kv_score splits into
    a kv half and a gate-score half; "Key design choices": state is float32 and APE
    [ratio, coff*head_dim] is added to each token's state on store)."""
    ks = np.asarray(kv_score_t, np.float32)
    row = ks.copy()
    if ape is not None:
        row[coff * D:] = ks[coff * D:] + np.asarray(ape[int(p) % ratio], np.float32)  # fp32 add
    return row


def fold_group(state_b: np.ndarray, j: int, ratio: int, coff: int):
    """Gathers the (kv, score) rows of compressed entry j from one sequence's state ring
    ([MAP] "How Does Compression Actually Work?", step 1).  Slot of position q = q mod (coff*ratio).
    Series A (channels [0, D) of each half) for tokens [j*r, (j+1)*r); with overlap (coff = 2)
    series B (channels [D, 2D)) for the previous block [(j-1)*r, j*r) when j >= 1."""
    nslots = coff * ratio
    kv, sc = [], []
    for q in range(j * ratio, (j + 1) * ratio):
        r = state_b[q % nslots]
        kv.append(r[0:D])
        sc.append(r[coff * D:coff * D + D])
    if coff == 2 and j >= 1:
        for q in range((j - 1) * ratio, j * ratio):
            r = state_b[q % nslots]
            kv.append(r[D:2 * D])
            sc.append(r[coff * D + D:coff * D + 2 * D])
    return np.asarray(kv, np.float64), np.asarray(sc, np.float64)


def fold_entry(kv: np.ndarray, sc: np.ndarray) -> np.ndarray:
    """Softmax of the gate scores over the group's tokens, per channel, then the weighted sum of
    kv ([MAP] "How Does Compression Actually Work?", steps 2-3; softmax over dim 0)."""
    m = sc.max(axis=0)
    e = np.exp(sc - m)
    w = e / e.sum(axis=0)
    return (w * kv).sum(axis=0)


def entry_latent(state_b, j, ratio, coff, norm_w, eps) -> np.ndarray:
    """The compressor's latent of entry j: fold, then RMSNorm * weight, before the RoPE ([MAP] "How
    Does Compression Actually Work?", steps 1-4)."""
    kv, sc = fold_group(state_b, j, ratio, coff)
    return rms_norm(fold_entry(kv, sc), norm_w, eps)


def compressed_entry(state_b, j, ratio, coff, norm_w, eps, cos_sin) -> np.ndarray:
    """Value of compressed entry j before encoding: fold, RMSNorm * weight, GPT-J RoPE of the last
    64 dims at position j*ratio ([MAP] "How Does Compression Actually Work?", steps 1-5)."""
    e = entry_latent(state_b, j, ratio, coff, norm_w, eps)
    cs = np.asarray(cos_sin[j * ratio], np.float64)
    e[D_NOPE:] = rope_gptj(e[D_NOPE:], cs[:32], cs[32:])
    return e


def index_key(latent, wk, kn_w, eps, cos_sin, pos: int) -> np.ndarray:
    """Index key of a compressed entry ([API] DeepseekV4Indexer (V4.1): the index key is derived from
    the compressor's latent, k = k_norm(wk(latent)); _produce_k: at group-boundary tokens, RoPE'd at
    the group position, then quantised into the indexer K cache; wk maps the main compressor's
    pre-RoPE latent to index keys).  latent [576] (entry_latent), wk [d, 576], kn_w [d]: k = wk latent,
    RMSNorm over its d dims times kn_w, then GPT-J RoPE of its last 64 dims at `pos` (reading: the
    key's rope dims are its last 64, as in the latent)."""
    k = np.asarray(wk, np.float64) @ np.asarray(latent, np.float64)
    k = rms_norm(k, kn_w, eps)
    cs = np.asarray(cos_sin[int(pos)], np.float64)
    k[-D_ROPE:] = rope_gptj(k[-D_ROPE:], cs[:32], cs[32:])
    return k


def encode_key(k, dtype: int) -> np.ndarray:
    """One index key -> its stored form in indexer-cache format `dtype` (F32, BF16, I8_ROWSCALE)."""
    if dtype == F32:
        return np.asarray(k, np.float64).astype(np.float32)
    if dtype == BF16:
        return bf16_encode(k)
    if dtype == I8_ROWSCALE:
        return i8_rowscale_encode(np.asarray(k, np.float64).astype(np.float32))
    if dtype == MXFP4:
        return mxfp4_encode(k)
    raise ValueError(dtype)


def compress_update(state, kv_score, positions, q_per_seq, ratio, coff, ape, norm_w, eps, cos_sin,
                    main: Paged, main_bt, cache_dtype, seqs=None, ik=None):
    """Per sequence, per new token in position order: store the token's state row, and when the
    token completes a group, fold the group and store the encoded entry into the main cache row
    j = p // ratio ([MAP] "Phase 2", compressor stream, items 1-4).  With `ik` (a dict: wk, kn_w,
    eps, cache: Paged, bt, dtype) the entry's index key (index_key, at the entry's RoPE position
    j * ratio) is also stored into row j of the indexer cache.
    Returns (new state for the processed sequences {b: array}, {(b, j): entry value},
    {(b, j): index key value})."""
    B = state.shape[0]
    seqs = range(B) if seqs is None else seqs
    new_state, entries, keys = {}, {}, {}
    for b in seqs:
        st = np.array(state[b], np.float32, copy=True)
        for i in range(q_per_seq):
            t = b * q_per_seq + i
            p = int(positions[t])
            st[p % (coff * ratio)] = state_row(kv_score[t], p, ratio, coff, ape)
            if emits(p, ratio):
                j = p // ratio
                e = compressed_entry(st, j, ratio, coff, norm_w, eps, cos_sin)
                entries[(b, j)] = e
                main.put(main_bt[b][j // PAGE], j % PAGE, encode_row(e, cache_dtype))
                if ik is not None:
                    k = index_key(entry_latent(st, j, ratio, coff, norm_w, eps), ik["wk"], ik["kn_w"], ik["eps"],
                                  cos_sin, j * ratio)
                    keys[(b, j)] = k
                    ik["cache"].put(ik["bt"][b][j // PAGE], j % PAGE, encode_key(k, ik["dtype"]))
        new_state[b] = st
    return new_state, entries, keys


# ----------------------------------------------------------------------------------------------
# Steps a3-a4: Lightning-Indexer scoring and top-k
# ----------------------------------------------------------------------------------------------

def indexer_scores(q_t, w_t, keys) -> np.ndarray:
    """s_j = sum_h w_h * ReLU(q_h . k_j) over the visible keys ([MAP] "Phase 2", indexer stream,
    item 4: per-block scores between indexer Q and compressed indexer K), returned as fp32."""
    logits = np.asarray(q_t, np.float64) @ np.asarray(keys, np.float64).T       # [I_h, n]
    s = (np.asarray(w_t, np.float64)[:, None] * np.maximum(logits, 0.0)).sum(axis=0)
    return s.astype(np.float32)


def topk_select(scores, k: int) -> np.ndarray:
    """The k best entries by (score desc, index asc); when there are at most k candidates every
    candidate is selected ([API] DeepseekV4Indexer.forward, short-context fill); -1 pads to k."""
    s = np.asarray(scores, np.float32)
    n = s.shape[0]
    order = np.lexsort((np.arange(n), -s.astype(np.float64)))
    out = np.full(k, -1, np.int32)
    m = min(n, k)
    out[:m] = order[:m]
    return out


def candidate_blocks(scores, block: int, m: int) -> np.ndarray:
    """Two-level candidate filtering, source side ([API] DeepseekV4Indexer: the indexer at
    candidate_source_layer_id additionally publishes the top candidate_topk_blocks blocks of
    candidate_block_size compressed positions).  Reading: a block's score is the largest score of
    its visible entries; the m best blocks by (score desc, block index asc), listed in increasing
    block index, -1 padded to m."""
    s = np.asarray(scores, np.float32)
    n = s.shape[0]
    nblk = (n + block - 1) // block
    keys = np.array([np.max(s[b * block:(b + 1) * block]) for b in range(nblk)], np.float64)
    order = np.lexsort((np.arange(nblk), -keys))
    out = np.full(m, -1, np.int32)
    sel = np.sort(order[:min(m, nblk)])
    out[:len(sel)] = sel
    return out


def listed_blocks(cand) -> list:
    """The blocks a candidate list names: its entries up to the first one that is negative or not
    larger than the entry before it (a source writes its blocks in increasing order, then -1; the
    pages fix no order, this is the reading taken so that a list is one increasing run)."""
    out = []
    for c in np.asarray(cand).tolist():
        if c < 0 or (out and c <= out[-1]):
            break
        out.append(int(c))
    return out


def masked_topk(scores, k: int, cand, block: int) -> np.ndarray:
    """Two-level candidate filtering, consumer side ([API] DeepseekV4Indexer: later indexers mask
    their scores to the candidate blocks before their own top-k): only entries whose block
    (j // block) is named by `cand` (listed_blocks) take part; the k best of them by (score desc,
    j asc), or all of them when there are at most k; -1 pads to k."""
    s = np.asarray(scores, np.float32)
    n = s.shape[0]
    blocks = set(listed_blocks(cand))
    inc = np.array([j for j in range(n) if j // block in blocks], np.int64)
    out = np.full(k, -1, np.int32)
    if inc.size == 0:
        return out
    order = inc[np.lexsort((inc, -s[inc].astype(np.float64)))]
    m = min(k, inc.size)
    out[:m] = order[:m]
    return out


# ----------------------------------------------------------------------------------------------
# Steps a5-a6: shared-KV sparse MLA attention and split merge
# ----------------------------------------------------------------------------------------------

def attention_rows(p, b, swa: Paged, swa_bt, cache_dtype, main: Paged | None, main_bt, ratio,
                   topk_row=None, window=WINDOW) -> np.ndarray:
    """The rows one query attends: the sliding window, then the selected compressed entries
    (top-k list; -1 and entries beyond n_c(p) are skipped) or, with no list, every visible
    compressed entry ([MAP] "Phase 3: forward_mqa()" items 1-3; "Layer-Type Summary")."""
    rows = [decode_rows(swa.logical(swa_bt[b], window_positions(p, window)), cache_dtype)]
    nc = n_compressed(p, ratio)
    if main is not None and nc > 0:
        if topk_row is None:
            idx = np.arange(nc)
        else:
            idx = np.asarray(topk_row, np.int64)
            idx = idx[(idx >= 0) & (idx < nc)]
        if idx.size:
            rows.append(decode_rows(main.logical(main_bt[b], idx), cache_dtype))
    return np.concatenate(rows, axis=0)


def mqa_decode(q_t, rows, sink, scale):
    """One softmax per head over all rows plus the sink logit ([MAP] "Phase 3" item 5: MQA over all
    the loaded KVs; item 4: optional sink; [API] DeepseekV4Attention: sink -inf = no effect).
    Logits use all 576 dims; values are the first 512.  Naive two-pass: max, then sums.
    Returns out [H, 512] and lse [H] (log of the full denominator, sink included)."""
    q = np.asarray(q_t, np.float64)
    kv = np.asarray(rows, np.float64)
    z = scale * (q @ kv.T)                                   # [H, R]
    s = np.full(q.shape[0], -np.inf) if sink is None else np.asarray(sink, np.float64)
    m = np.maximum(z.max(axis=1), s)
    p = np.exp(z - m[:, None])
    denom = p.sum(axis=1) + np.exp(s - m)
    out = (p @ kv[:, :DV]) / denom[:, None]
    return out, m + np.log(denom)


def mqa_partial(q_t, rows, scale):
    """Unnormalised partial over one chunk of rows: (o_c = sum p v / l_c, lse_c)."""
    return mqa_decode(q_t, rows, None, scale)


def merge_partials(outs, lses, sink=None):
    """Combine chunk results: lse = log(sum_c e^lse_c [+ e^sink]), o = sum_c e^(lse_c - lse) o_c."""
    lses = np.asarray(lses, np.float64)                     # [C, H]
    outs = np.asarray(outs, np.float64)                     # [C, H, DV]
    parts = lses if sink is None else np.concatenate([lses, np.asarray(sink, np.float64)[None]], 0)
    m = parts.max(axis=0)
    lse = m + np.log(np.exp(parts - m).sum(axis=0))
    wts = np.exp(lses - lse[None])
    return (wts[..., None] * outs).sum(axis=0), lse


# ----------------------------------------------------------------------------------------------
# The whole step
# ----------------------------------------------------------------------------------------------

def decode_step(st, seqs=None, topk_override=None):
    """Runs insert -> compress -> indexer + top-k -> attention for the tokens of `seqs`
    (all sequences by default) on a StepInputs bundle.  `topk_override` [T, k] feeds a given
    selection to the attention instead of the indexer's (attention-only cases).
    Returns a dict of per-token results keyed by token index."""
    cfg = st.cfg
    B, qps = cfg.B, cfg.q_per_seq
    seqs = list(range(B)) if seqs is None else list(seqs)
    toks = [b * qps + i for b in seqs for i in range(qps)]

    swa = Paged(st.swa_cache)
    sel = np.zeros(cfg.T, bool)
    sel[toks] = True
    slots = np.where(sel, st.slot_mapping, -1)
    q_prep = getattr(cfg, "q_prep", False)
    if q_prep:  # the fused insert also rotates the new kv rows at their positions
        kv_insert(swa, st.kv_new, cfg.act_dtype, slots, cfg.cache_dtype, st.positions, st.cos_sin)
    else:
        kv_insert(swa, st.kv_new, cfg.act_dtype, slots, cfg.cache_dtype)

    res = {"swa_written": dict(swa.written), "tokens": toks}
    # the queries the attention reads: as given, or normed, rotated and padded by the fused insert and
    # stored in the activation format
    q_att, q_out = {}, {}
    for t in toks:
        q_t = decode_rows(st.q[t], cfg.act_dtype)
        if q_prep:
            qv = qnorm_rope(q_t, int(st.positions[t]), st.cos_sin, st.q_norm_w, st.eps, True, True, cfg.H_pad)
            q_out[t] = encode_row(qv, cfg.act_dtype)
            q_t = decode_rows(q_out[t], cfg.act_dtype)[:cfg.H]
        q_att[t] = q_t
    res["q_out"] = q_out
    main = None
    idx = Paged(st.idx_cache) if (cfg.ratio > 0 and cfg.topk > 0) else None
    if cfg.ratio > 0:
        main = Paged(st.main_cache)
        ik = None
        if idx is not None and getattr(st, "wk", None) is not None:  # the compressor also stores index keys
            ik = {"wk": bf16_decode(st.wk), "kn_w": st.ik_norm_w, "eps": st.eps, "cache": idx, "bt": st.idx_bt,
                  "dtype": cfg.idx_dtype}
        new_state, entries, keys = compress_update(st.state, st.kv_score, st.positions, qps, cfg.ratio, cfg.coff,
                                                   st.ape, st.norm_w, st.eps, st.cos_sin, main, st.main_bt,
                                                   cfg.cache_dtype, seqs=seqs, ik=ik)
        res["state"] = new_state
        res["entries"] = entries
        res["main_written"] = dict(main.written)
        res["keys"] = keys
        res["idx_written"] = dict(idx.written) if idx is not None else {}

    topk, scores, cand_out = {}, {}, {}
    if cfg.ratio > 0 and cfg.topk > 0:
        for t in toks:
            b, p = t // qps, int(st.positions[t])
            nc = n_compressed(p, cfg.ratio)
            keys = decode_rows(idx.logical(st.idx_bt[b], np.arange(nc)), cfg.idx_dtype)
            q_t = decode_rows(st.q_idx[t], cfg.act_dtype)
            s = indexer_scores(q_t, st.w_idx[t], keys) if nc else np.zeros(0, np.float32)
            scores[t] = s
            cb = getattr(cfg, "cand_block", 0)
            # a consumer of another layer's candidate blocks; a token whose entries all fit in the top-k
            # takes every entry, as without candidates ([API] DeepseekV4Indexer.forward short-context fill)
            if cb and st.cand_in is not None and nc > cfg.topk:
                topk[t] = masked_topk(s, cfg.topk, st.cand_in[t], cb)
            else:
                topk[t] = topk_select(s, cfg.topk)
            if cb and getattr(cfg, "cand_write", False):  # the candidate source publishes its best blocks
                cand_out[t] = candidate_blocks(s, cb, cfg.cand_topk)
    res["scores"], res["topk"], res["cand_out"] = scores, topk, cand_out

    out, lse = {}, {}
    for t in toks:
        b, p = t // qps, int(st.positions[t])
        krow = None
        if cfg.ratio > 0 and cfg.topk > 0:
            krow = topk_override[t] if topk_override is not None else topk[t]
        rows = attention_rows(p, b, swa, st.swa_bt, cfg.cache_dtype, main, st.main_bt, cfg.ratio, krow)
        out[t], lse[t] = mqa_decode(q_att[t], rows, st.sink, st.softmax_scale)
    res["out"], res["lse"] = out, lse
    return res


# ----------------------------------------------------------------------------------------------
# Chunked prefill
# ----------------------------------------------------------------------------------------------

def apply_step(st, res) -> None:
    """Commits one step's writes to the caches of `st` in place: its SWA rows, the compressor state of
    the sequences it ran, its compressed entries and index keys."""
    for (pg, off), row in res["swa_written"].items():
        st.swa_cache[pg, off] = row
    for b, ring in res.get("state", {}).items():
        st.state[b] = ring
    for (pg, off), row in res.get("main_written", {}).items():
        st.main_cache[pg, off] = row
    for (pg, off), row in res.get("idx_written", {}).items():
        st.idx_cache[pg, off] = row


def prefill(chunks) -> dict:
    """Chunked prefill ([ASCEND] §8 "The prefill path": the same chain -- query/KV prologue, SWA
    insert, compressor, indexer, sparse attention -- for every prompt token; [API]
    DeepseekV4Attention.PREFILL_CHUNK_SIZE: in fixed-size chunks).  `chunks` gives the steps of
    consecutive positions of every sequence from position 0, sharing one set of caches; each runs
    decode_step and its writes are committed before the next.  Returns {(b, p): {"out", "lse",
    "topk", "q_out"}} for every token."""
    out = {}
    for st in chunks:
        res = decode_step(st)
        qps = st.cfg.q_per_seq
        for t in res["tokens"]:
            b, p = t // qps, int(st.positions[t])
            out[(b, p)] = {"out": res["out"][t], "lse": res["lse"][t], "topk": res["topk"].get(t),
                           "q_out": res["q_out"].get(t)}
        apply_step(st, res)
    return out
