"""Seeded synthetic inputs for the DeepSeek-V4 hybrid compressed-attention decode step.

This module is shared by the CPU oracle's tests, the GPU parity tests, ``smoke()``
and ``bench.py``.  It draws random numbers and lays them out in the paged-cache
byte formats; it holds none of the method's arithmetic (no fold, no indexer
score, no top-k, no attention, no UE8M0 scale selection).

Workload shapes follow the five decode configurations of the hot path:

  tiny_c4_f32    1 seq, context 1024, c4, 16 heads, indexer 4 x 64, top-k 64, fp32
  csa_c4_bf16    32 seqs, context 65536, c4, 64 heads, indexer 64 x 128 bf16, top-k 512
  hca_c128_bf16  64 seqs, context U[65536, 131072], c128 dense, 64 heads, no indexer
  csa_c4_fp8     128 seqs, context U[8192, 32768], 2 query tokens per seq,
                 fp8_ds_mla caches, int8 + fp32-scale indexer keys, top-k 512
  csa_c4_1m      4 seqs, context 1048576, 128 heads, top-k 2048
  csa_c4_mxfp4   csa_c4_bf16 with its indexer keys as 68-byte MXFP4 records

plus small variants (``small_*``) of the same dtypes and head counts that the
oracle finishes in seconds while still spanning several tiles and ragged tails.

Value recipe: q, kv_new, indexer queries, cache rows ~ N(0,1)*0.1; query and index-key RMSNorm
weights 1 + N(0,1)*0.1; latent -> index key projection N(0,1)*0.1 (bf16); kv_score
~ N(0,1); indexer weights ~ N(0,1)*0.1; RMSNorm weight 1 + N(0,1)*0.1; APE
~ N(0,1)*0.1; sink ~ N(0,1); RoPE table theta = 10000.  Large bf16 buffers are
drawn by inverse-CDF lookup: a uniform 16-bit integer indexes a table of the
65536 normal quantiles rounded to bf16, which is N(0,1)*0.1 at bf16 resolution
and costs one table gather per element.  Block tables are seeded random
permutations of the physical pages (shuffled paging).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

import numpy as np

D = 576          # latent width: 512 no-pe + 64 rope
DV = 512         # value width: the first 512 latent dims
D_ROPE = 64
WINDOW = 128
PAGE = 64
FP8_DS_MLA_BYTES = 656   # 512 e4m3 | 64 bf16 rope (128 B) | 8 UE8M0 scale bytes | 8 pad
FP8_SCALE_OFF = 640
FP8_ROPE_OFF = 512

# dtype tags, equal in value to the C enum dsv4_dtype
F32, BF16, FP8_DS_MLA, I8_ROWSCALE, MXFP4 = 0, 1, 2, 3, 4
DTYPE_NAMES = {F32: "f32", BF16: "bf16", FP8_DS_MLA: "fp8_ds_mla", I8_ROWSCALE: "i8_rowscale", MXFP4: "mxfp4"}


@dataclass(frozen=True)
class Config:
    name: str
    B: int
    q_per_seq: int
    ctx: tuple            # (lo, hi) inclusive range of total context length per seq, or explicit tuple of lengths
    H: int
    ratio: int            # 4 (CSA) or 128 (HCA); 0 = SWA only
    I_h: int              # indexer heads (0 = no indexer / dense)
    d_I: int
    topk: int             # 0 = dense over every compressed entry
    act_dtype: int        # q, kv_new, indexer q dtype (F32 or BF16)
    cache_dtype: int      # SWA + main cache dtype (F32, BF16, FP8_DS_MLA)
    idx_dtype: int        # indexer key cache dtype (F32, BF16, I8_ROWSCALE)
    out_dtype: int        # attention output dtype
    seed: int = 0xD5E4
    explicit_lens: tuple = ()
    q_prep: bool = True   # queries arrive un-normed and un-rotated: the fused insert norms, rotates and pads them
    ik_store: bool = True  # the compressor also writes each new entry's index key (CSA layers with an indexer)
    cand_block: int = 0    # two-level candidate filtering: entries per candidate block (0 = off)
    cand_topk: int = 0     # candidate blocks per token
    cand_write: bool = False  # this layer's indexer publishes its best blocks (else it consumes given ones)

    @property
    def T(self) -> int:
        return self.B * self.q_per_seq

    @property
    def H_pad(self) -> int:
        """Query heads of the attention's input and output buffers: a multiple of 64 for bf16 and
        fp8_ds_mla caches (the tensor-core attention takes heads in groups of 64), else H."""
        return self.H if self.cache_dtype == F32 else (self.H + 63) // 64 * 64

    @property
    def coff(self) -> int:
        return 2 if self.ratio == 4 else 1


CONFIGS = {
    "tiny_c4_f32": Config("tiny_c4_f32", B=1, q_per_seq=1, ctx=(1024, 1024), H=16, ratio=4, I_h=4, d_I=64,
                          topk=64, act_dtype=F32, cache_dtype=F32, idx_dtype=F32, out_dtype=F32, seed=0xD5E4 + 0),
    "csa_c4_bf16": Config("csa_c4_bf16", B=32, q_per_seq=1, ctx=(65536, 65536), H=64, ratio=4, I_h=64, d_I=128,
                          topk=512, act_dtype=BF16, cache_dtype=BF16, idx_dtype=BF16, out_dtype=BF16, seed=0xD5E4 + 1),
    "hca_c128_bf16": Config("hca_c128_bf16", B=64, q_per_seq=1, ctx=(65536, 131072), H=64, ratio=128, I_h=0, d_I=0,
                            topk=0, act_dtype=BF16, cache_dtype=BF16, idx_dtype=BF16, out_dtype=BF16, seed=0xD5E4 + 2),
    "csa_c4_fp8": Config("csa_c4_fp8", B=128, q_per_seq=2, ctx=(8192, 32768), H=64, ratio=4, I_h=64, d_I=128,
                         topk=512, act_dtype=BF16, cache_dtype=FP8_DS_MLA, idx_dtype=I8_ROWSCALE, out_dtype=BF16,
                         seed=0xD5E4 + 3),
    "csa_c4_1m": Config("csa_c4_1m", B=4, q_per_seq=1, ctx=(1048576, 1048576), H=128, ratio=4, I_h=64, d_I=128,
                        topk=2048, act_dtype=BF16, cache_dtype=BF16, idx_dtype=BF16, out_dtype=BF16, seed=0xD5E4 + 4),
    # the CSA c4 bf16 layer as a consumer of an earlier layer's candidate blocks (8 of 16 blocks of 1024)
    "csa_c4_cand": Config("csa_c4_cand", B=32, q_per_seq=1, ctx=(65536, 65536), H=64, ratio=4, I_h=64, d_I=128,
                          topk=512, act_dtype=BF16, cache_dtype=BF16, idx_dtype=BF16, out_dtype=BF16,
                          seed=0xD5E4 + 6, cand_block=1024, cand_topk=8),
    # the CSA c4 bf16 layer as the candidate source (publishes 8 blocks of 1024 per token)
    "csa_c4_src": Config("csa_c4_src", B=32, q_per_seq=1, ctx=(65536, 65536), H=64, ratio=4, I_h=64, d_I=128,
                         topk=512, act_dtype=BF16, cache_dtype=BF16, idx_dtype=BF16, out_dtype=BF16,
                         seed=0xD5E4 + 7, cand_block=1024, cand_topk=8, cand_write=True),
    # the CSA c4 bf16 layer with its indexer keys in the 68-byte MXFP4 record
    "csa_c4_mxfp4": Config("csa_c4_mxfp4", B=32, q_per_seq=1, ctx=(65536, 65536), H=64, ratio=4, I_h=64, d_I=128,
                           topk=512, act_dtype=BF16, cache_dtype=BF16, idx_dtype=MXFP4, out_dtype=BF16,
                           seed=0xD5E4 + 5),
}

# Small variants: same dtypes and head counts, ragged lengths spanning several key tiles,
# short-context cases (n_c <= top-k), contexts shorter than the window and an emitting fold.
SMALL_CONFIGS = {
    "small_c4_f32": dataclasses.replace(CONFIGS["tiny_c4_f32"], name="small_c4_f32", B=3,
                                        explicit_lens=(1024, 333, 50)),
    "small_c4_bf16": dataclasses.replace(CONFIGS["csa_c4_bf16"], name="small_c4_bf16", B=4,
                                         explicit_lens=(4100, 2048, 777, 9000)),
    "small_c128_bf16": dataclasses.replace(CONFIGS["hca_c128_bf16"], name="small_c128_bf16", B=4,
                                           explicit_lens=(20000, 8192, 1000, 131)),
    "small_c4_fp8": dataclasses.replace(CONFIGS["csa_c4_fp8"], name="small_c4_fp8", B=3,
                                        explicit_lens=(4100, 2048, 1023)),
    "small_c4_h128": dataclasses.replace(CONFIGS["csa_c4_1m"], name="small_c4_h128", B=2,
                                         explicit_lens=(20000, 9001)),
    "small_swa_only": dataclasses.replace(CONFIGS["csa_c4_bf16"], name="small_swa_only", B=2, ratio=0, I_h=0,
                                          d_I=0, topk=0, explicit_lens=(300, 7)),
    "edge_first_token": dataclasses.replace(CONFIGS["csa_c4_bf16"], name="edge_first_token", B=2,
                                            explicit_lens=(1, 4)),
    # two-level candidate filtering: a consumer of given candidate blocks and a source that publishes them
    "small_c4_cand": dataclasses.replace(CONFIGS["csa_c4_bf16"], name="small_c4_cand", B=4,
                                         explicit_lens=(20000, 9000, 2300, 700), cand_block=1024, cand_topk=3),
    "small_c4_cand_src": dataclasses.replace(CONFIGS["csa_c4_bf16"], name="small_c4_cand_src", B=3,
                                             explicit_lens=(20000, 6000, 900), cand_block=512, cand_topk=4,
                                             cand_write=True),
    # candidates with two query tokens a sequence (scored densely, masked per token), on CUDA-core fp32
    # keys, and on rows long enough for the sliced top-k (n_c > 32768)
    "small_c4_cand_mtp": dataclasses.replace(CONFIGS["csa_c4_fp8"], name="small_c4_cand_mtp", B=5,
                                             explicit_lens=(9000, 4100, 2050, 3000, 7000), cand_block=256,
                                             cand_topk=5),
    # three query tokens a sequence: more query columns than one tensor-core tile takes, so the
    # indexer takes each token as its own sequence (plain, and as a candidate consumer)
    "small_c4_q3": dataclasses.replace(CONFIGS["csa_c4_bf16"], name="small_c4_q3", B=4, q_per_seq=3,
                                       explicit_lens=(9000, 3001, 700, 2050)),
    "small_c4_cand_q3": dataclasses.replace(CONFIGS["csa_c4_bf16"], name="small_c4_cand_q3", B=3, q_per_seq=3,
                                            explicit_lens=(12000, 5003, 2400), cand_block=512, cand_topk=4),
    "small_c4_cand_f32": dataclasses.replace(CONFIGS["tiny_c4_f32"], name="small_c4_cand_f32", B=5,
                                             explicit_lens=(2400, 1300, 1029, 2000, 3333), cand_block=128,
                                             cand_topk=3),
    "small_c4_cand_long": dataclasses.replace(CONFIGS["csa_c4_bf16"], name="small_c4_cand_long", B=5,
                                              explicit_lens=(140000, 8000, 4000, 3000, 139001), cand_block=2048,
                                              cand_topk=6),
    "small_c4_cand_src_long": dataclasses.replace(CONFIGS["csa_c4_mxfp4"], name="small_c4_cand_src_long", B=2,
                                                  q_per_seq=2, explicit_lens=(140000, 5000), cand_block=128,
                                                  cand_topk=16, cand_write=True),
    "small_c4_mxfp4": dataclasses.replace(CONFIGS["csa_c4_mxfp4"], name="small_c4_mxfp4", B=3, q_per_seq=2,
                                          explicit_lens=(9001, 2050, 700)),
    # 32 query heads padded to 64 by the fused query preparation
    "small_c4_h32pad": dataclasses.replace(CONFIGS["csa_c4_bf16"], name="small_c4_h32pad", B=3, H=32,
                                           explicit_lens=(3000, 700, 129)),
}

ALL_CONFIGS = {**CONFIGS, **SMALL_CONFIGS}


def n_pages(rows: int) -> int:
    return (rows + PAGE - 1) // PAGE


def row_elems(dtype: int, width: int) -> tuple:
    """numpy dtype and trailing shape of one stored cache row of `width` logical elements."""
    if dtype == F32:
        return np.float32, (width,)
    if dtype == BF16:
        return np.uint16, (width,)
    if dtype == FP8_DS_MLA:
        assert width == D
        return np.uint8, (FP8_DS_MLA_BYTES,)
    if dtype == I8_ROWSCALE:
        return np.uint8, (width + 4,)
    if dtype == MXFP4:
        return np.uint8, (width // 2 + width // 32,)
    raise ValueError(dtype)


class _Draw:
    """Seeded draws; every tensor gets its own stream keyed by (seed, name)."""

    _bf16_table = None
    _e4m3_table = None
    _i8_table = None

    def __init__(self, seed: int):
        self.seed = seed

    def rng(self, name: str) -> np.random.Generator:
        key = [self.seed] + [ord(c) for c in name]
        return np.random.default_rng(key)

    @classmethod
    def quantiles(cls) -> np.ndarray:
        from scipy.special import ndtri
        return ndtri((np.arange(65536, dtype=np.float64) + 0.5) / 65536.0)

    @classmethod
    def bf16_table(cls) -> np.ndarray:
        if cls._bf16_table is None:
            import torch
            t = torch.from_numpy((cls.quantiles() * 0.1).astype(np.float32)).to(torch.bfloat16)
            cls._bf16_table = t.view(torch.int16).numpy().view(np.uint16).copy()
        return cls._bf16_table

    @classmethod
    def e4m3_table(cls) -> np.ndarray:
        # N(0,1)*0.1 expressed in units of 2^-7 (the nominal block scale), as e4m3fn codes
        if cls._e4m3_table is None:
            import torch
            v = np.clip(cls.quantiles() * 0.1 * 128.0, -448.0, 448.0).astype(np.float32)
            cls._e4m3_table = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
        return cls._e4m3_table

    @classmethod
    def i8_table(cls) -> np.ndarray:
        if cls._i8_table is None:
            cls._i8_table = np.clip(np.rint(cls.quantiles() * 40.0), -127, 127).astype(np.int8)
        return cls._i8_table

    def normal_f32(self, name, shape, scale=1.0, loc=0.0):
        return (self.rng(name).standard_normal(shape, dtype=np.float32) * np.float32(scale)
                + np.float32(loc)).astype(np.float32)

    def bf16(self, name, shape):
        """bf16 bit patterns of N(0,1)*0.1 by inverse-CDF lookup."""
        u = self.rng(name).integers(0, 65536, size=shape, dtype=np.uint16)
        return self.bf16_table()[u]

    def act(self, name, shape, dtype):
        """Activation-like values N(0,1)*0.1 stored as fp32 or bf16 bits."""
        if dtype == F32:
            return self.normal_f32(name, shape, 0.1)
        if dtype == BF16:
            return self.bf16(name, shape)
        raise ValueError(dtype)

    def cache_rows(self, name, n_rows, width, dtype):
        """`n_rows` stored rows of `width` logical elements in cache format `dtype`."""
        if dtype in (F32, BF16):
            return self.act(name, (n_rows, width), dtype)
        rng = self.rng(name)
        if dtype == FP8_DS_MLA:
            rec = np.zeros((n_rows, FP8_DS_MLA_BYTES), np.uint8)
            u = rng.integers(0, 65536, size=(n_rows, 512), dtype=np.uint16)
            rec[:, :512] = self.e4m3_table()[u]
            rope = self.bf16(name + ".rope", (n_rows, D_ROPE))
            rec[:, FP8_ROPE_OFF:FP8_ROPE_OFF + 128] = rope.view(np.uint8).reshape(n_rows, 128)
            # scale bytes around 2^-7 so decoded values are ~N(0,1)*0.1
            rec[:, FP8_SCALE_OFF:FP8_SCALE_OFF + 8] = rng.integers(119, 122, size=(n_rows, 8), dtype=np.uint8)
            return rec
        if dtype == MXFP4:
            # E2M1 codes (magnitude codes 0..7 drawn with weights favouring small values, random sign)
            # and block exponent bytes 122..124
            w = np.array([4, 6, 6, 5, 4, 3, 2, 1], np.float64)
            mag = rng.choice(8, size=(n_rows, width), p=w / w.sum()).astype(np.uint8)
            codes = mag | (rng.integers(0, 2, size=(n_rows, width), dtype=np.uint8) << 3)
            rec = np.zeros((n_rows, width // 2 + width // 32), np.uint8)
            rec[:, :width // 2] = codes[:, 0::2] | (codes[:, 1::2] << 4)
            rec[:, width // 2:] = rng.integers(122, 125, size=(n_rows, width // 32), dtype=np.uint8)
            return rec
        if dtype == I8_ROWSCALE:
            rec = np.zeros((n_rows, width + 4), np.uint8)
            u = rng.integers(0, 65536, size=(n_rows, width), dtype=np.uint16)
            rec[:, :width] = self.i8_table()[u].view(np.uint8)
            scale = (0.1 / 40.0 * rng.uniform(0.75, 1.25, size=n_rows)).astype(np.float32)
            rec[:, width:width + 4] = scale.view(np.uint8).reshape(n_rows, 4)
            return rec
        raise ValueError(dtype)


@dataclass
class StepInputs:
    """Everything one decode step reads, in host memory, in the exact stored formats."""
    cfg: Config
    ctx_len: np.ndarray          # [B] int64, total length after this step's tokens
    positions: np.ndarray        # [T] int32
    kv_new: np.ndarray           # [T, D] f32 or bf16 bits
    slot_mapping: np.ndarray     # [T] int64 SWA slot (page * PAGE + offset)
    swa_cache: np.ndarray        # [swa_pages, PAGE, row]
    swa_bt: np.ndarray           # [B, swa_max_pages] int32 (-1 = not resident)
    q: np.ndarray                # [T, H, D]
    sink: np.ndarray             # [H] f32
    softmax_scale: float
    q_norm_w: np.ndarray = None  # [D] f32 per-channel weight of the per-head query RMSNorm
    wk: np.ndarray = None        # [d_I, D] bf16 bits: latent -> index key projection (CSA layers)
    ik_norm_w: np.ndarray = None # [d_I] f32 weight of the index key's RMSNorm
    cos_sin: np.ndarray = None   # [max_pos, 64] f32: 32 cos | 32 sin (RoPE of q, kv and compressed entries)
    kv_score: np.ndarray = None  # [T, 2*coff*D] f32
    state: np.ndarray = None     # [B, coff*ratio, 2*coff*D] f32
    ape: np.ndarray = None       # [ratio, coff*D] f32
    norm_w: np.ndarray = None    # [D] f32
    eps: float = 1e-6
    main_cache: np.ndarray = None
    main_bt: np.ndarray = None   # [B, main_max_pages] int32
    idx_cache: np.ndarray = None
    idx_bt: np.ndarray = None
    q_idx: np.ndarray = None     # [T, I_h, d_I]
    w_idx: np.ndarray = None     # [T, I_h] f32
    given_topk: np.ndarray = None  # [T, topk] int32: a fixed valid selection for standalone attention cases
    cand_in: np.ndarray = None   # [T, cand_topk] int32: candidate blocks published by an earlier layer (consumer)
    extra: dict = field(default_factory=dict)


def context_lengths(cfg: Config) -> np.ndarray:
    if cfg.explicit_lens:
        assert len(cfg.explicit_lens) == cfg.B
        return np.asarray(cfg.explicit_lens, np.int64)
    lo, hi = cfg.ctx
    if lo == hi:
        return np.full(cfg.B, lo, np.int64)
    return _Draw(cfg.seed).rng("ctx_len").integers(lo, hi + 1, size=cfg.B).astype(np.int64)


def rope_table(max_pos: int, theta: float = 10000.0) -> np.ndarray:
    """Rotary table [max_pos, 64]: cos of the 32 pair angles, then their sin (model constant)."""
    inv = theta ** (-np.arange(0, D_ROPE, 2, dtype=np.float64) / D_ROPE)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def _paged_table(draw: _Draw, name: str, rows_per_seq: np.ndarray, first_row: np.ndarray, max_rows: int):
    """Block table covering rows [first_row[b], rows_per_seq[b]) of each seq with shuffled physical pages.

    Logical pages outside that range are -1.  Returns (table [B, max_pages], n_physical_pages)."""
    B = len(rows_per_seq)
    max_pages = max(1, n_pages(max_rows))
    lp_lo = first_row // PAGE
    lp_hi = np.array([n_pages(int(r)) for r in rows_per_seq], np.int64)
    counts = np.maximum(lp_hi - lp_lo, 0)
    total = int(counts.sum())
    perm = draw.rng(name + ".perm").permutation(max(total, 1)).astype(np.int32)
    bt = np.full((B, max_pages), -1, np.int32)
    k = 0
    for b in range(B):
        c = int(counts[b])
        bt[b, lp_lo[b]:lp_lo[b] + c] = perm[k:k + c]
        k += c
    return bt, max(total, 1)


def make_step(cfg: Config, with_given_topk: bool = True) -> StepInputs:
    draw = _Draw(cfg.seed)
    B, qps, T, H = cfg.B, cfg.q_per_seq, cfg.T, cfg.H
    L = context_lengths(cfg)
    assert np.all(L >= qps)
    positions = (L[:, None] - qps + np.arange(qps)[None, :]).reshape(T).astype(np.int32)
    max_ctx = int(L.max())

    # ---- SWA cache: only pages that hold the last WINDOW + q_per_seq positions are resident
    swa_first = np.maximum(L - qps - WINDOW + 1, 0)
    swa_bt, swa_pages = _paged_table(draw, "swa_bt", L, swa_first, max_ctx)
    erow_t, erow_shape = row_elems(cfg.cache_dtype, D)
    swa_cache = draw.cache_rows("swa_cache", swa_pages * PAGE, D, cfg.cache_dtype).reshape(
        (swa_pages, PAGE) + erow_shape)
    tok_b = np.repeat(np.arange(B), qps)
    slot = swa_bt[tok_b, positions // PAGE].astype(np.int64) * PAGE + positions % PAGE

    kv_new = draw.act("kv_new", (T, D), cfg.act_dtype)
    q = draw.act("q", (T, H, D), cfg.act_dtype)
    sink = draw.normal_f32("sink", (H,), 1.0)
    st = StepInputs(cfg=cfg, ctx_len=L, positions=positions, kv_new=kv_new, slot_mapping=slot,
                    swa_cache=swa_cache, swa_bt=swa_bt, q=q, sink=sink, softmax_scale=float(D) ** -0.5)
    st.cos_sin = rope_table(max_ctx + 1)
    st.q_norm_w = draw.normal_f32("q_norm_w", (D,), 0.1, 1.0)
    if cfg.ratio == 0:
        return st

    r, coff = cfg.ratio, cfg.coff
    # ---- compressor inputs and fp32 state ring (coff*r slots per seq)
    st.kv_score = draw.normal_f32("kv_score", (T, 2 * coff * D), 1.0)
    st.state = draw.normal_f32("state", (B, coff * r, 2 * coff * D), 1.0)
    st.ape = draw.normal_f32("ape", (r, coff * D), 0.1)
    st.norm_w = draw.normal_f32("norm_w", (D,), 0.1, 1.0)

    # ---- main (compressed) cache: rows j < floor(L/r) exist after the step
    nc_after = L // r
    main_bt, main_pages = _paged_table(draw, "main_bt", nc_after, np.zeros(B, np.int64), int(nc_after.max()))
    st.main_bt = main_bt
    st.main_cache = draw.cache_rows("main_cache", main_pages * PAGE, D, cfg.cache_dtype).reshape(
        (main_pages, PAGE) + erow_shape)

    if cfg.I_h > 0:
        idx_bt, idx_pages = _paged_table(draw, "idx_bt", nc_after, np.zeros(B, np.int64), int(nc_after.max()))
        ir_t, ir_shape = row_elems(cfg.idx_dtype, cfg.d_I)
        st.idx_bt = idx_bt
        st.idx_cache = draw.cache_rows("idx_cache", idx_pages * PAGE, cfg.d_I, cfg.idx_dtype).reshape(
            (idx_pages, PAGE) + ir_shape)
        st.q_idx = draw.act("q_idx", (T, cfg.I_h, cfg.d_I), cfg.act_dtype)
        st.w_idx = draw.normal_f32("w_idx", (T, cfg.I_h), 0.1)
        if cfg.ik_store:
            st.wk = draw.bf16("wk", (cfg.d_I, D))
            st.ik_norm_w = draw.normal_f32("ik_norm_w", (cfg.d_I,), 0.1, 1.0)

    if cfg.cand_block and not cfg.cand_write:
        # another layer's published candidates: distinct visible blocks of each token, increasing, -1
        # padded; by token: full lists, lists holding the partial last block, half-full lists, an empty
        # list, and lists whose increasing run ends early (a smaller or equal entry, then more blocks)
        M = cfg.cand_topk
        c = np.full((T, M), -1, np.int32)
        rng = draw.rng("cand_in")
        for t in range(T):
            nblk = ((int(positions[t]) + 1) // r + cfg.cand_block - 1) // cfg.cand_block
            kind = t % 5
            m = min(nblk, M) if kind != 2 else min(nblk, M) // 2
            if t % 7 == 5:
                m = 0
            if m == 0:
                continue
            sel = rng.choice(nblk, size=m, replace=False) if nblk > m else np.arange(nblk)
            if kind == 1 and nblk - 1 not in sel:
                sel[0] = nblk - 1
            sel = np.sort(sel)
            if kind == 4 and m >= 3:
                sel[m // 2] = sel[m // 2 - 1]  # the run ends here; the entries after it are not listed
            c[t, :m] = sel
        st.cand_in = c

    if cfg.topk > 0 and with_given_topk:
        # an arbitrary valid selection (distinct visible indices, ascending, -1 padded) for attention-only cases
        g = np.full((T, cfg.topk), -1, np.int32)
        rng = draw.rng("given_topk")
        for t in range(T):
            nc = int((int(positions[t]) + 1) // r)
            m = min(nc, cfg.topk)
            if m:
                sel = rng.choice(nc, size=m, replace=False) if nc > m else np.arange(nc)
                g[t, :m] = np.sort(sel)
        st.given_topk = g
    return st


# ------------------------------------------------------------------------------------------------
# Prefill: P tokens of every sequence from position 0, on caches that hold nothing yet
# ------------------------------------------------------------------------------------------------

@dataclass
class PrefillInputs:
    """A prefill of positions 0 .. P-1 of each of B sequences.  `base` holds every token (token (b, p)
    at row b * P + p of its per-token arrays) and the caches, whose rows hold seeded garbage until
    the prefill writes them; chunk() cuts the decode step of some consecutive positions of every
    sequence out of it, sharing those caches (what one chunk writes, the next reads)."""
    cfg: Config
    P: int
    base: StepInputs

    def chunk(self, p0: int, n: int) -> StepInputs:
        """The step of positions p0 .. p0 + n - 1 of every sequence (T = B * n, sequence-major)."""
        cfg, P, st = self.cfg, self.P, self.base
        rows = (np.arange(cfg.B)[:, None] * P + p0 + np.arange(n)[None, :]).reshape(-1)
        ccfg = dataclasses.replace(cfg, q_per_seq=n, explicit_lens=tuple([p0 + n] * cfg.B))
        tok = lambda a: None if a is None else a[rows]  # noqa: E731
        return dataclasses.replace(st, cfg=ccfg, ctx_len=np.full(cfg.B, p0 + n, np.int64), positions=st.positions[rows],
                                   kv_new=st.kv_new[rows], slot_mapping=st.slot_mapping[rows], q=st.q[rows],
                                   kv_score=tok(st.kv_score), q_idx=tok(st.q_idx), w_idx=tok(st.w_idx),
                                   given_topk=None, cand_in=None, extra={})

    def spans(self, chunk: int):
        """(p0, n) of the chunks of `chunk` positions (the last one ragged)."""
        return [(p0, min(chunk, self.P - p0)) for p0 in range(0, self.P, chunk)]


def make_prefill(cfg: Config, P: int) -> PrefillInputs:
    """Inputs of a P-token prefill of B sequences: the decode-step generator with every position a
    new token (pages for all P positions; caches, state ring and indexer keys seeded garbage)."""
    assert P >= 1
    full = dataclasses.replace(cfg, q_per_seq=P, explicit_lens=tuple([P] * cfg.B), cand_block=0)
    return PrefillInputs(cfg=dataclasses.replace(cfg, explicit_lens=tuple([P] * cfg.B)), P=P,
                         base=make_step(full, with_given_topk=False))


PREFILL_CONFIGS = {
    # (layer configuration, prompt length): c4 with the indexer (top-k below n_c late in the prompt,
    # ragged last chunk), fp32 keys on the CUDA-core indexer, c128 without an indexer, and the
    # full-size c4 bf16 prefill the benchmark times
    "prefill_c4_small": (dataclasses.replace(CONFIGS["csa_c4_bf16"], name="prefill_c4_small", B=3, topk=32), 301),
    "prefill_c4_f32": (dataclasses.replace(CONFIGS["tiny_c4_f32"], name="prefill_c4_f32", B=2, topk=16), 150),
    "prefill_c128_small": (dataclasses.replace(CONFIGS["hca_c128_bf16"], name="prefill_c128_small", B=2), 300),
    "prefill_c4_bf16": (dataclasses.replace(CONFIGS["csa_c4_bf16"], name="prefill_c4_bf16", B=16), 512),
}


def max_compressed(cfg: Config) -> int:
    L = context_lengths(cfg)
    return int(L.max() // cfg.ratio) if cfg.ratio else 0
