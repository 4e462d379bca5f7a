// Lightning-Indexer scoring and per-query top-k.
//
// "DeepSeek V4 Attention: Code Reading Map", §Phase 2 (indexer stream, item 4: scores between the
// indexer queries and the compressed indexer keys, then the top-k compressed blocks) and
// §Concrete Trace (top-1024 of ~125,000); "vllm.models.deepseek_v41.attention",
// DeepseekV4Indexer.forward (when the candidates fit in top-k, every candidate is selected).
// Score: s[t][j] = sum_h w[t][h] * ReLU(q[t][h] . k_j) in fp32.
//
// One call:
//  1. score: a CTA works on 128-key tiles of one sequence for all of that sequence's query tokens,
//     so each key row leaves HBM once per step.  bf16 keys run on the tensor cores (tcgen05 MMA,
//     TMA-fed); fp32 and int8 keys on the CUDA cores.  Besides the score row of each token, the
//     epilogue builds a 4096-bin histogram of the scores' top 12 order-preserving key bits.
//  2. top-k (tk::topk_token, one CTA per token): from the histogram, the bin B* holding the k-th
//     best score; every entry above B* is selected outright, the k - A best entries inside B* are
//     chosen exactly (larger score first, then smaller j); the selection is written sorted by j.
//     On the tensor-core path the CTA that scores the last tile of a sequence runs it at its end
//     (no further launch); the CUDA-core path launches one CTA per token after scoring.
#include "dsv4_common.cuh"
#include "dsv4_launch.h"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace dsv4 {

static __device__ unsigned int g_flags_ix = 0;

constexpr int IX_TILE = 128;
constexpr int HIST_BITS = 12;
constexpr int HIST_BINS = 1 << HIST_BITS;
constexpr int HIST_SHIFT = 32 - HIST_BITS;
constexpr uint32_t FLAG_TIMEOUT = 4u;
constexpr int TOPK_FUSED_MAX = 32768;  // longer rows: top-k spread over CTAs by topk_slice_kernel

// Order-preserving map of an fp32 score to uint32 (larger score -> larger key).
__device__ __forceinline__ uint32_t order_key(float s) {
  uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// n_c of token t, clamped to what the workspace and grid were sized for (max_context); a position
// outside [0, max_context) is flagged.
__device__ __forceinline__ int visible_entries(const int32_t* positions, int t, int max_context, int ratio) {
  const int pos = positions[t];
  if (pos < 0 || pos >= max_context) {
    atomicOr(&g_flags_ix, FLAG_PAGE);
    return pos < 0 ? 0 : max_context / ratio;
  }
  return (pos + 1) / ratio;
}
__device__ __forceinline__ int visible_entries(const dsv4_indexer_topk_params& p, int t) {
  return visible_entries(p.positions, t, p.max_context, p.ratio);
}

// ------------------------------------------------------------------------------------------------
// Workspace
// ------------------------------------------------------------------------------------------------
struct IxLayout {
  size_t nc_stride;
  size_t scores_off, hist_off, done_off, tcnt_off, cand_off, bits_off, total;
};

static IxLayout ix_layout(const dsv4_indexer_topk_params& p) {
  IxLayout L;
  const int64_t max_nc = (int64_t)p.max_context / p.ratio;
  L.nc_stride = align_up((size_t)(max_nc > 0 ? max_nc : 1), 128);  // whole 128-entry scan blocks
  L.scores_off = 0;
  L.hist_off = align_up(L.scores_off + (size_t)p.T * L.nc_stride * sizeof(float), 256);
  L.done_off = L.hist_off + (size_t)p.T * HIST_BINS * sizeof(uint32_t);  // zeroed together with hist
  // completion counters: one a sequence, or one a token when the tensor-core kernel takes each query
  // token as its own sequence (T >= B)
  L.tcnt_off = L.done_off + (size_t)p.T * sizeof(uint32_t);                // zeroed together with hist
  L.cand_off = align_up(L.tcnt_off + (size_t)p.T * 2 * sizeof(uint32_t), 256);
  L.bits_off = align_up(L.cand_off + (size_t)p.T * L.nc_stride * sizeof(uint64_t), 256);
  L.total = align_up(L.bits_off + (size_t)p.T * (L.nc_stride / 32) * sizeof(uint32_t), 256);
  return L;
}

size_t indexer_topk_workspace(const dsv4_indexer_topk_params& p) { return ix_layout(p).total; }

struct TopkBufs {
  float* scores;       // [T][nc_stride]
  uint32_t* hist;      // [T][HIST_BINS] counts of the scores' top 12 order-key bits
  uint32_t* seq_done;  // [T] key tiles of the sequence (or token) scored so far (tensor-core path)
  uint64_t* cand;      // [T][nc_stride] top-k candidates that do not fit in shared memory
  uint32_t* tcnt;      // [T][2] sliced top-k: candidates appended, slices finished
  uint32_t* bits;      // [T][nc_stride / 32] sliced top-k: selection bitmap (layout of bitmap_words)
  int nc_stride;
};

// Adds one to bin `bin` of `hist` for each lane with `on`, one atomic per distinct bin of the warp.
// Every lane of the warp must call it.
__device__ __forceinline__ void hist_add_warp(uint32_t* hist, uint32_t bin, bool on) {
  const unsigned active = __ballot_sync(0xffffffffu, on);
  if (!on) return;
  const unsigned peers = __match_any_sync(active, bin);
  if ((int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
}

// ------------------------------------------------------------------------------------------------
// Two-level candidate filtering ("vllm.models.deepseek_v41.attention", DeepseekV4Indexer: the source
// indexer publishes each token's best blocks of candidate_block_size entries, later indexers keep to
// them).  A token's list names the blocks of its increasing run: its entries up to the first one that
// is negative or not larger than the entry before it.
// ------------------------------------------------------------------------------------------------
struct CandArgs {
  int32_t* blocks;  // [T][M]; null: no candidate filtering
  int M;            // entries a token
  int lg;           // log2 of the entries of a block (7 .. 16)
  int write;        // 1: the source (publishes), 0: a consumer (reads)
};

__host__ inline CandArgs cand_args(const dsv4_indexer_topk_params& p) {
  CandArgs c{nullptr, 0, 0, 0};
  if (p.cand_block_size > 0) {
    c.blocks = p.cand_blocks;
    c.M = p.cand_topk;
    while ((1 << c.lg) < p.cand_block_size) ++c.lg;
    c.write = p.cand_write;
  }
  return c;
}

// Whether list row[0, M) names block blk.
__device__ __forceinline__ bool cand_names(const int32_t* row, int M, int blk) {
  int prev = -1;
  for (int i = 0; i < M; ++i) {
    const int c = __ldg(row + i);
    if (c <= prev) return false;
    if (c >= blk) return c == blk;
    prev = c;
  }
  return false;
}

// ------------------------------------------------------------------------------------------------
// Top-k of one token, run by one whole CTA once the token's scores and histogram are complete.
// The score row reaches shared memory by bulk (TMA) copies in 16 KB chunks with up to four in flight
// (plain loads would go through an L1 that the kernels' large shared memory leaves almost no room).
//  1. From the histogram, the bin B* holding the k-th best score and the count A of scores above it
//     (256 threads own 16 bins each, read straight from L2; a block scan from the top finds the
//     crossing thread).
//  2. One pass over the scores: lane l of a warp takes entries 4l .. 4l + 3 of a 128-entry block;
//     the four ballots of "bin > B*" are the block's four words of the selection bitmap (bit l of
//     word c = entry 4l + c), and entries in B* go to a list of candidate values (low 20 key bits,
//     j): a resident row through a second bitmap (four more ballots, no branch) listed afterwards,
//     a longer row chunk by chunk through per-warp slots.
//  3. The k - A largest candidates (larger score first, then smaller j: the values are unique) by a
//     radix select of 10-bit digits over the 40-bit values, stopping at the first digit whose bin
//     holds exactly the entries still needed; they are added to the bitmap.
//  4. The bitmap is compacted in increasing j into the output row; -1 pads it.
// ------------------------------------------------------------------------------------------------
namespace tk {
constexpr int RBINS = 1024;       // radix bins (10-bit digits)
constexpr int J_BITS = 20;        // n_c <= 2^20 (checked on the host)
constexpr int CTL_BYTES = 512;
constexpr int FIND_THREADS = 256;  // threads that own histogram bins in block_find_bin
constexpr int CHUNK = 4096;       // scores per bulk copy (16 KB)
constexpr int NBUF = 4;           // chunk buffers (copies in flight)
constexpr int SCAN_WARPS_MIN = 8;  // the kernels run top-k with at least 8 warps

struct Ctl {
  uint64_t bar[NBUF + 1];  // chunk buffers, histogram
  uint32_t bin, above, cnt, ncand;
  uint32_t total;  // block_find_bin: the sum of the histogram
  int run;         // candidate filtering: entries of the token's list that name blocks
  int last;        // topk_part: this CTA completed the token's count
  int wt[40];      // block scan scratch
};
static_assert(sizeof(Ctl) <= CTL_BYTES, "top-k control block");

// Candidate value: (low 20 order-key bits << 20) | (2^20 - 1 - j); larger = better score, then smaller j.
__device__ __forceinline__ uint64_t cand_value(uint32_t key, int j) {
  return ((uint64_t)(key & ((1u << HIST_SHIFT) - 1u)) << J_BITS) | (uint64_t)((1u << J_BITS) - 1u - (uint32_t)j);
}
__device__ __forceinline__ int cand_j(uint64_t v) {
  return (int)((1u << J_BITS) - 1u - (uint32_t)(v & ((1u << J_BITS) - 1u)));
}

// Offsets in the shared buffer: control, radix bins, bitmap, histogram, chunks, candidates.
// Selection bitmap layout: 128-entry block b has the four words 4 b + c, and bit l of word 4 b + c
// stands for entry 128 b + 4 l + c (lane l of a warp reads entries 4 l .. 4 l + 3 of a block as one
// float4, so each of the four ballots of a block is one word).
__host__ __device__ inline int bitmap_words(int n) { return (n + 127) / 128 * 4; }
__device__ __forceinline__ int bit_word(int j) { return ((j >> 7) << 2) | (j & 3); }
__device__ __forceinline__ uint32_t bit_mask(int j) { return 1u << ((j >> 2) & 31); }
// Candidate filtering: one bit per 128-entry block of the row, set when the block lies in a block the
// token's list names.
__host__ __device__ inline int incl_words(int n) { return ((n + 127) / 128 + 31) / 32; }

__host__ __device__ inline size_t hist_offset(int n) {
  return (CTL_BYTES + RBINS * 4 + (size_t)bitmap_words(n) * 4 + (size_t)incl_words(n) * 4 + 127) / 128 * 128;
}
__host__ __device__ inline size_t fixed_bytes(int n) {
  return hist_offset(n) + (size_t)HIST_BINS * 4 + (size_t)NBUF * CHUNK * 4;
}

// Exclusive prefix sum of one value per thread over the CTA; *total gets the sum.  Warp scans by
// shuffles, then every thread adds up the totals of the warps before its own (wt: 32 ints).
__device__ __forceinline__ int block_excl_scan(int v, int* wt, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) wt[warp] = incl;
  __syncthreads();
  int before = 0, all = 0;
  for (int w = 0; w < nw; ++w) {
    const int t = wt[w];
    before += w < warp ? t : 0;
    all += t;
  }
  *total = all;
  __syncthreads();  // wt is free again for the next call
  return before + incl - v;
}

// The bin of histogram h (256 * PER bins; in shared memory, or with GLOBAL in global memory, read
// through L2) where the count from the top first reaches rem: c->bin, the count in the bins above
// it: c->above, its own count: c->cnt.  Thread i < 256 owns bins [256 PER - PER (i + 1), 256 PER -
// PER i) (the top bins first).  Called by the whole CTA.
template <int PER, bool GLOBAL = false>
__device__ __forceinline__ void block_find_bin(const uint32_t* h, uint32_t rem, Ctl* c) {
  const int tid = threadIdx.x;
  uint32_t v[PER];
  uint32_t sum = 0;
  if (tid < FIND_THREADS) {
    const uint4* src = reinterpret_cast<const uint4*>(h + FIND_THREADS * PER - PER * (tid + 1));
#pragma unroll
    for (int q = 0; q < PER / 4; ++q) {
      const uint4 u = GLOBAL ? __ldcg(src + q) : src[q];
      v[4 * q] = u.x;
      v[4 * q + 1] = u.y;
      v[4 * q + 2] = u.z;
      v[4 * q + 3] = u.w;
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) sum += v[i];
  }
  int total;
  const uint32_t excl = (uint32_t)block_excl_scan((int)sum, c->wt, &total);
  if (tid == 0) c->total = (uint32_t)total;
  if (tid < FIND_THREADS && excl < rem && excl + sum >= rem) {
    uint32_t cum = excl;
#pragma unroll
    for (int i = PER - 1; i >= 0; --i) {
      if (cum < rem && cum + v[i] >= rem) {
        c->bin = (uint32_t)(FIND_THREADS * PER - PER * (tid + 1) + i);
        c->above = cum;
        c->cnt = v[i];
      }
      cum += v[i];
    }
  }
  __syncthreads();
}

// Bitmap words and candidates of scores in shared memory: sb holds entries j_base .. j_base + 128
// nblocks - 1 (j_base a multiple of 128; entries >= n are ignored).  Entries with bin > bstar set
// their bit in `bits` (every word of the scanned blocks below `words` is written, 16 bytes at a
// time), entries in bstar are appended to `cand` (capacity ccap) through the counter *ncand.  With an
// inclusion bitmap `incl` (candidate filtering), entries of 128-entry blocks whose bit is clear take
// no part, and all_in selects every other entry (no candidates).  bits (16-byte aligned), cand and
// ncand may be in shared or global memory.  Warp w owns the consecutive blocks w P .. w P + P - 1 (P =
// ceil(nblocks / warps)), taken SCAN_B at a time: lane l reads entries 4 l .. 4 l + 3 of a block as
// one float4, and the four ballots of "bin > bstar" are the block's four bitmap words.  Candidates
// are rare: per group of SCAN_B blocks each lane counts its own, the warp takes their slots with one
// atomic, and each lane writes its candidates to consecutive slots from the scores in its registers.
constexpr int SCAN_B = CHUNK / 128 / SCAN_WARPS_MIN;  // 128-entry blocks a warp reads at once (4)
__device__ __forceinline__ void scan_chunk(const float* sb, int nblocks, int j_base, int n, uint32_t bstar,
                                           uint32_t* bits, int words, uint64_t* cand, uint32_t ccap,
                                           uint32_t* ncand, const uint32_t* incl = nullptr, bool all_in = false) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, NW = blockDim.x >> 5;
  const float4* sb4 = reinterpret_cast<const float4*>(sb);
  const int per = (nblocks + NW - 1) / NW;
  const int b0 = min(nblocks, warp * per), b1 = min(nblocks, b0 + per);
  for (int g = b0; g < b1; g += SCAN_B) {
    float4 v[SCAN_B];
#pragma unroll
    for (int i = 0; i < SCAN_B; ++i) v[i] = g + i < b1 ? sb4[(g + i) * 32 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
    int nvs[SCAN_B];
    int lc = 0;  // this lane's candidates in the group
#pragma unroll
    for (int i = 0; i < SCAN_B; ++i) {
      const int blk = g + i;
      const int gb = (j_base >> 7) + blk;
      const bool live = blk < b1 && (incl == nullptr || ((incl[gb >> 5] >> (gb & 31)) & 1u));  // warp-uniform
      nvs[i] = live ? n - (j_base + blk * 128 + 4 * lane) : 0;  // entries c < nvs[i] of the lane count
      const float e[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
      uint32_t sw[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t bin = order_key(e[c]) >> HIST_SHIFT;
        sw[c] = __ballot_sync(0xffffffffu, c < nvs[i] && (all_in || bin > bstar));
        lc += (!all_in && c < nvs[i] && bin == bstar) ? 1 : 0;
      }
      const int wg = gb * 4;
      if (lane == 0 && blk < b1 && wg < words)
        *reinterpret_cast<uint4*>(bits + wg) = make_uint4(sw[0], sw[1], sw[2], sw[3]);
    }
    // the group's candidates, written while its scores are in registers: one atomic for the warp
    const int wtot = __reduce_add_sync(0xffffffffu, lc);
    if (wtot == 0) continue;  // warp-uniform
    int scan = lc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, scan, o);
      if (lane >= o) scan += u;
    }
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(ncand, (uint32_t)wtot);
    uint32_t idx = __shfl_sync(0xffffffffu, base, 0) + (uint32_t)(scan - lc);
    if (lc == 0) continue;
#pragma unroll
    for (int i = 0; i < SCAN_B; ++i) {
      const float e[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
      const int j0 = j_base + (g + i) * 128 + 4 * lane;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t key = order_key(e[c]);
        if (c < nvs[i] && (key >> HIST_SHIFT) == bstar) {
          if (idx < ccap) cand[idx] = cand_value(key, j0 + c);
          ++idx;
        }
      }
    }
  }
}

// The bitmap words of a whole resident row in one pass (sb: the row from entry 0; nblk 128-entry
// blocks): entries above the threshold bin in `bits`, entries in it in `cbits` (same layout), entries j
// >= n and, with `incl`, blocks not named in neither (all_in: every other entry in bits).  Warp w takes
// blocks w, w + NW, ..., GB at a time with all of a group's scores loaded first; per column two
// ballots and no branch.  With both bin edges among the non-negative scores (FAST) the float bits are
// compared as signed integers, which orders them as the order keys do.
template <bool FAST>
__device__ __forceinline__ void scan_bits_t(const float4* sb4, int nblk, int n, uint32_t lo, uint32_t hi,
                                            bool none_above, uint32_t* bits, uint32_t* cbits, const uint32_t* incl,
                                            bool all_in) {
  constexpr int GB = 7;  // blocks a warp loads at once (28 registers)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, NW = blockDim.x >> 5;
  for (int g0 = warp; g0 < nblk; g0 += GB * NW) {
    float4 v[GB];
#pragma unroll
    for (int k = 0; k < GB; ++k) {
      const int blk = g0 + k * NW;
      v[k] = blk < nblk ? sb4[blk * 32 + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < GB; ++k) {
      const int blk = g0 + k * NW;
      if (blk >= nblk) break;  // warp-uniform
      const float e[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
      uint32_t sw[4], cw[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        bool ge, gt;
        if (FAST) {
          const int xb = __float_as_int(e[c]);
          ge = xb >= (int)lo;
          gt = !none_above && xb >= (int)hi;
        } else {
          const uint32_t key = order_key(e[c]);
          ge = key >= lo;
          gt = !none_above && key >= hi;
        }
        sw[c] = __ballot_sync(0xffffffffu, gt);
        cw[c] = __ballot_sync(0xffffffffu, ge);
      }
      const int rem = n - blk * 128;  // >= 1
      const bool live = incl == nullptr || ((incl[blk >> 5] >> (blk & 31)) & 1u);
      if (rem < 128 || !live || all_in) {  // warp-uniform: the row's last block, or candidate filtering
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int kk = rem >= 128 ? 32 : (rem - c + 3) >> 2;  // lanes holding an entry j < n in column c
          const uint32_t vm = live ? (kk >= 32 ? ~0u : (1u << kk) - 1u) : 0u;
          sw[c] = all_in ? vm : sw[c] & vm;
          cw[c] = all_in ? 0u : cw[c] & vm;
        }
      }
      if (lane == 0) {
        *reinterpret_cast<uint4*>(bits + 4 * blk) = make_uint4(sw[0], sw[1], sw[2], sw[3]);
        *reinterpret_cast<uint4*>(cbits + 4 * blk) =
            make_uint4(cw[0] & ~sw[0], cw[1] & ~sw[1], cw[2] & ~sw[2], cw[3] & ~sw[3]);
      }
    }
  }
}
__device__ __forceinline__ void scan_bits(const float* sb, int nblk, int n, uint32_t bstar, uint32_t* bits,
                                          uint32_t* cbits, const uint32_t* incl, bool all_in) {
  const uint32_t lo = bstar << HIST_SHIFT, hi = (bstar + 1u) << HIST_SHIFT;
  const bool none_above = bstar == (uint32_t)(HIST_BINS - 1);
  const float4* sb4 = reinterpret_cast<const float4*>(sb);
  if (lo >= 0x80000000u)
    scan_bits_t<true>(sb4, nblk, n, lo - 0x80000000u, none_above ? 0u : hi - 0x80000000u, none_above, bits, cbits,
                      incl, all_in);
  else
    scan_bits_t<false>(sb4, nblk, n, lo, hi, none_above, bits, cbits, incl, all_in);
}

// The entries marked in cbits (words words; row sb in shared memory) listed as candidate values into
// cand[0, min(m, cap)); c->ncand = m.  Thread i takes words i, i + NT, ...  Whole CTA.
__device__ void list_cands(const float* sb, const uint32_t* cbits, int words, uint64_t* cand, uint32_t cap, Ctl* c) {
  const int tid = threadIdx.x, NT = blockDim.x;
  int cnt = 0;
  for (int w = tid; w < words; w += NT) cnt += __popc(cbits[w]);
  int total;
  uint32_t pos = (uint32_t)block_excl_scan(cnt, c->wt, &total);
  for (int w = tid; w < words; w += NT) {
    uint32_t m = cbits[w];
    while (m) {
      const int l = __ffs(m) - 1;
      m &= m - 1;
      const int j = ((w >> 2) << 7) | (l << 2) | (w & 3);
      if (pos < cap) cand[pos] = cand_value(order_key(sb[j]), j);
      ++pos;
    }
  }
  if (tid == 0) c->ncand = (uint32_t)total;
}

// Threshold of the R largest (0 < R < m) of m unique values get(i) < 2^(TOP + 10): a radix select of
// 10-bit digits from bit TOP down that stops at the first digit whose bin holds exactly the values
// still needed; the R largest are the values >= the result.  rb: RBINS shared bins.  Whole CTA.
template <int TOP, typename Get>
__device__ uint64_t radix_threshold(uint32_t m, int R, uint32_t* rb, Ctl* c, Get get) {
  const int tid = threadIdx.x, NT = blockDim.x;
  uint64_t prefix = 0, thr = 0;
  uint32_t rem = (uint32_t)R;
  for (int shift = TOP; shift >= 0; shift -= 10) {
    for (int x = tid; x < RBINS; x += NT) rb[x] = 0u;
    __syncthreads();
    const uint64_t hmask = shift == TOP ? 0ull : (~0ull << (shift + 10)) & ((1ull << (TOP + 10)) - 1ull);
    for (uint32_t i = tid; i < m; i += NT) {
      const uint64_t v = get(i);
      if ((v & hmask) == prefix) atomicAdd(&rb[(v >> shift) & (RBINS - 1)], 1u);
    }
    __syncthreads();
    block_find_bin<RBINS / FIND_THREADS>(rb, rem, c);
    prefix |= (uint64_t)c->bin << shift;
    rem -= c->above;
    thr = prefix;
    if (c->cnt == rem) break;  // every value of this digit is needed: v >= prefix selects them
  }
  return thr;
}

// Exact choice of the R largest of m candidate values (unique), OR-ed into the bitmap.  Whole CTA.
__device__ void select_candidates(const uint64_t* cand, uint32_t m, int R, uint32_t* rb, Ctl* c, uint32_t* bits) {
  const int tid = threadIdx.x, NT = blockDim.x;
  if (R <= 0) return;
  const uint64_t thr =
      (uint32_t)R < m ? radix_threshold<30>(m, R, rb, c, [&](uint32_t i) { return cand[i]; }) : 0ull;
  for (uint32_t i = tid; i < m; i += NT) {
    const uint64_t v = cand[i];
    if (v >= thr) {
      const int j = cand_j(v);
      atomicOr(&bits[bit_word(j)], bit_mask(j));
    }
  }
}

// The selection in increasing j from the bitmap (words written by this CTA or, for a global bitmap,
// by others before a fence), listed first in sel_s (K ints of shared memory), then written out with
// -1 padding together with the scores of the selected entries (from `row_s` when the row is in
// shared memory, else from global s_g).  Thread i takes a run of 128-entry blocks; within a block
// the entries of lane position l come in the order c = 0..3, which is increasing j.  Whole CTA.
__device__ void write_selection(const uint32_t* bits, bool bits_global, int words, int K, int32_t* out, float* out_s,
                                const float* row_s, const float* s_g, Ctl* c, int* sel_s) {
  const int tid = threadIdx.x, NT = blockDim.x;
  const int nblk = words >> 2;
  const int per = (nblk + NT - 1) / NT;
  const int k0 = min(nblk, tid * per), k1 = min(nblk, k0 + per);
  auto block = [&](int b) {
    const uint4* p4 = reinterpret_cast<const uint4*>(bits) + b;
    return bits_global ? __ldcg(p4) : *p4;
  };
  int cnt = 0;
  for (int b = k0; b < k1; ++b) {
    const uint4 w = block(b);
    cnt += __popc(w.x) + __popc(w.y) + __popc(w.z) + __popc(w.w);
  }
  int total;
  int pos = block_excl_scan(cnt, c->wt, &total);
  for (int b = k0; b < k1 && pos < K; ++b) {
    const uint4 w = block(b);
    uint32_t any = w.x | w.y | w.z | w.w;
    while (any && pos < K) {
      const int l = __ffs(any) - 1;
      any &= any - 1;
      const int j = b * 128 + 4 * l;
      if ((w.x >> l) & 1u && pos < K) sel_s[pos++] = j;
      if ((w.y >> l) & 1u && pos < K) sel_s[pos++] = j + 1;
      if ((w.z >> l) & 1u && pos < K) sel_s[pos++] = j + 2;
      if ((w.w >> l) & 1u && pos < K) sel_s[pos++] = j + 3;
    }
  }
  __syncthreads();
  const int m = min(total, K);
  for (int x = tid; x < K; x += NT) {
    const int j = x < m ? sel_s[x] : -1;
    out[x] = j;
    if (out_s) out_s[x] = j < 0 ? -INFINITY : (row_s ? row_s[j] : __ldcg(s_g + j));
  }
}

// Inclusion bitmap (incl_words(n) words of shared memory) of a consumer token with list row[0, M) and
// blocks of 2^lg entries: bit g set when 128-entry block g of the row lies in a named block.  Whole CTA.
__device__ void build_incl(const int32_t* row, int M, int lg, int n, uint32_t* incl, Ctl* c) {
  const int tid = threadIdx.x, NT = blockDim.x, lane = tid & 31;
  const int nb = (n + 127) >> 7, iw = incl_words(n);
  for (int x = tid; x < iw; x += NT) incl[x] = 0u;
  if (tid < 32) {  // the run: the first entry that is negative or not above the one before ends it
    int run = M;
    for (int base = 0; base < M; base += 32) {
      const int i = base + lane;
      const int ci = i < M ? __ldg(row + i) : 0;
      const int cp = i == 0 ? -1 : (i < M ? __ldg(row + i - 1) : 0);
      const unsigned bad = __ballot_sync(0xffffffffu, i < M && ci <= cp);
      if (bad) {
        run = base + __ffs(bad) - 1;
        break;
      }
    }
    if (lane == 0) c->run = run;
  }
  __syncthreads();
  const int sh = lg - 7, per = 1 << sh;  // 128-entry blocks of a candidate block
  const int run = c->run;
  for (int x = tid; x < run * per; x += NT) {
    const int blk = __ldg(row + (x >> sh));
    if (blk > ((nb - 1) >> sh)) continue;  // past the row
    const int g = (blk << sh) + (x & (per - 1));
    if (g < nb) atomicOr(&incl[g >> 5], 1u << (g & 31));
  }
  __syncthreads();
}

// The source's publication for one token: out[0, M) = the M blocks of 2^lg entries with the largest
// block score (the largest score of the block's entries j < n; ties: lower block first) in increasing
// order, or every block then -1 when there are at most M.  The row s_g is read from global memory
// (16-byte aligned, room for round_up(n, 128) entries); buf: shared memory of at least
// CTL_BYTES + 4 RBINS + 4 ceil(n / 2^lg) bytes.  Whole CTA.
__device__ void publish_blocks(const float* s_g, int n, int lg, int M, int32_t* out, uint8_t* buf) {
  const int tid = threadIdx.x, NT = blockDim.x, lane = tid & 31, warp = tid >> 5, NW = NT >> 5;
  const int nblk = n > 0 ? ((n - 1) >> lg) + 1 : 0;
  if (nblk <= M) {
    for (int x = tid; x < M; x += NT) out[x] = x < nblk ? x : -1;
    return;
  }
  Ctl* c = reinterpret_cast<Ctl*>(buf);
  uint32_t* rb = reinterpret_cast<uint32_t*>(buf + CTL_BYTES);
  uint32_t* bkey = rb + RBINS;  // order key of each block's largest score
  for (int x = tid; x < nblk; x += NT) bkey[x] = 0u;
  __syncthreads();
  const int n128 = (n + 127) >> 7;
  for (int g = warp; g < n128; g += NW) {
    const int j0 = (g << 7) + 4 * lane;
    const float4 v = __ldcg(reinterpret_cast<const float4*>(s_g + j0));
    uint32_t k = 0u;  // below every score's order key
    if (j0 < n) k = order_key(v.x);
    if (j0 + 1 < n) k = max(k, order_key(v.y));
    if (j0 + 2 < n) k = max(k, order_key(v.z));
    if (j0 + 3 < n) k = max(k, order_key(v.w));
    k = __reduce_max_sync(0xffffffffu, k);
    if (lane == 0) atomicMax(&bkey[(g << 7) >> lg], k);
  }
  __syncthreads();
  // value of block i: its key, then the lower block first (blocks < 2^20)
  auto val = [&](uint32_t i) { return ((uint64_t)bkey[i] << J_BITS) | (uint64_t)((1u << J_BITS) - 1u - i); };
  const uint64_t thr = radix_threshold<50>((uint32_t)nblk, M, rb, c, val);
  // the M selected blocks in increasing order: thread i takes a run of blocks
  const int per = (nblk + NT - 1) / NT;
  const int k0 = min(nblk, tid * per), k1 = min(nblk, k0 + per);
  int cnt = 0;
  for (int i = k0; i < k1; ++i) cnt += val((uint32_t)i) >= thr ? 1 : 0;
  int total;
  int pos = block_excl_scan(cnt, c->wt, &total);
  for (int i = k0; i < k1; ++i)
    if (val((uint32_t)i) >= thr && pos < M) out[pos++] = i;
  for (int x = total + tid; x < M; x += NT) out[x] = -1;  // never: exactly M values are >= thr
  __syncthreads();
}

// The whole CTA selects the top K of token scores s_g[0, n) (row 16-byte aligned with room for
// round_up(n, 128) entries; the histogram hist_g of their order keys is complete) into out[0, K) in
// increasing j (out_s: their scores, may be null); gcand (n entries) holds candidates that do not fit
// in `buf` (buf_bytes of 128-byte aligned shared memory).  A consumer of candidate blocks passes its
// list crow[0, cM) (blocks of 2^clg entries): when n > K only entries of named blocks take part (the
// histogram counts only those), and when they are at most K all of them are selected.  Returns false
// if a copy timed out.
__device__ bool topk_token(const float* s_g, uint32_t* hist_g, int n, int K, int32_t* out, float* out_s,
                           uint64_t* gcand, uint8_t* buf, size_t buf_bytes, volatile int* abort,
                           const int32_t* crow = nullptr, int cM = 0, int clg = 0) {
  const int tid = threadIdx.x, NT = blockDim.x;
  if (n <= K) {  // short context: every entry, in order (the histogram is cleared for the next call)
    for (int x = tid; x < K; x += NT) {
      out[x] = x < n ? x : -1;
      if (out_s) out_s[x] = x < n ? __ldcg(s_g + x) : -INFINITY;
    }
    for (int x = tid; x < HIST_BINS; x += NT) hist_g[x] = 0u;
    return true;
  }
  const size_t fixed = fixed_bytes(n);
  if (fixed > buf_bytes) {  // cannot happen for n <= 2^20 with the buffers the kernels pass
    if (tid == 0) atomicOr(&g_flags_ix, FLAG_TOPK);
    for (int x = tid; x < K; x += NT) out[x] = -1;
    return false;
  }
  Ctl* c = reinterpret_cast<Ctl*>(buf);
  uint32_t* rb = reinterpret_cast<uint32_t*>(buf + CTL_BYTES);
  const int words = bitmap_words(n);
  uint32_t* bits = rb + RBINS;
  uint32_t* incl = crow ? bits + words : nullptr;  // consumer: named 128-entry blocks
  uint32_t* hist_s = reinterpret_cast<uint32_t*>(buf + hist_offset(n));
  uint8_t* chunks = reinterpret_cast<uint8_t*>(hist_s + HIST_BINS);
  uint64_t* cand_s = reinterpret_cast<uint64_t*>(buf + fixed);
  const uint32_t cap = (uint32_t)((buf_bytes - fixed) / 8);
  if ((size_t)K > 2 * (size_t)cap) {  // the selection is listed over the candidate area (never short for
                                      // the buffers the kernels pass)
    if (tid == 0) atomicOr(&g_flags_ix, FLAG_TOPK);
    for (int x = tid; x < K; x += NT) out[x] = -1;
    return false;
  }
  const int nchunks = (n + CHUNK - 1) / CHUNK;
  const int n128 = (n + 127) & ~127;  // copy whole 128-entry blocks (the row has room)
  // the whole row stays in the chunk buffers when it fits (then the output scores come from there)
  const bool resident = nchunks <= NBUF;

  if (tid == 0) {
    c->bin = 0;
    c->above = 0;
    c->cnt = 0;
    c->ncand = 0;
    for (int i = 0; i <= NBUF; ++i) tc::mbar_init(&c->bar[i], 1);
    tc::fence_barrier_init();
  }
  // (no barrier here: the other threads touch the control block and the mbarriers only after the
  // barriers inside the threshold search below)
  auto issue = [&](int cc) {
    const uint32_t bytes = (uint32_t)min(CHUNK, n128 - cc * CHUNK) * 4u;
    uint64_t* bar = &c->bar[cc % NBUF];
    tc::mbar_arrive_expect_tx(bar, bytes);
    tc::bulk_load(chunks + (size_t)(cc % NBUF) * CHUNK * 4, s_g + (size_t)cc * CHUNK, bytes, bar);
  };
  if (tid == 0) {
    // the scores were written through the generic proxy (possibly by other CTAs): order them before
    // the bulk copies read them
    asm volatile("fence.proxy.async;" ::: "memory");
    for (int cc = 0; cc < min(NBUF, nchunks); ++cc) issue(cc);
  }
  if (incl) build_incl(crow, cM, clg, n, incl, c);  // while the copies are in flight

  // 1. threshold bin, from the global histogram read through L2 (each counting thread loads its own
  // 16 bins), which is then cleared for the next call (this CTA is its last reader)
  block_find_bin<HIST_BINS / FIND_THREADS, true>(hist_g, (uint32_t)K, c);
  for (int x = tid; x < HIST_BINS; x += NT) hist_g[x] = 0u;
  // a consumer whose named blocks hold at most K entries (the histogram counts them) takes all of them
  const bool all_in = incl != nullptr && c->total <= (uint32_t)K;
  const uint32_t bstar = c->bin;
  const int R = all_in ? 0 : K - (int)c->above;  // still to choose among the candidates
  const uint32_t C = all_in ? 0u : c->cnt;       // scores in the threshold bin
  uint64_t* cand = C <= cap ? cand_s : gcand;
  const uint32_t ccap = C <= cap ? cap : (uint32_t)n;

  // 2. selection bitmap and candidates: a resident row in one pass once all of it has landed, a
  // longer one chunk by chunk
  int stop = nchunks;  // first chunk not consumed
  if (resident) {
    bool ok = true;
    for (int cc = 0; cc < nchunks && ok; ++cc) ok = tc::mbar_wait_bounded(&c->bar[cc], 0, abort);
    if (!__syncthreads_and(ok)) {
      stop = 0;
    } else {  // the threshold bin's entries marked in a second bitmap (over the unused histogram area)
      uint32_t* cbits = hist_s;
      scan_bits(reinterpret_cast<const float*>(chunks), n128 >> 7, n, bstar, bits, cbits, incl, all_in);
      __syncthreads();
      list_cands(reinterpret_cast<const float*>(chunks), cbits, words, cand, ccap, c);
    }
  }
  for (int cc = 0; cc < nchunks && !resident; ++cc) {
    if (!__syncthreads_and(tc::mbar_wait_bounded(&c->bar[cc % NBUF], (cc / NBUF) & 1, abort))) {
      stop = cc;
      break;
    }
    const float* sb = reinterpret_cast<const float*>(chunks + (size_t)(cc % NBUF) * CHUNK * 4);
    scan_chunk(sb, min(CHUNK, n128 - cc * CHUNK) >> 7, cc * CHUNK, n, bstar, bits, words, cand, ccap, &c->ncand,
               incl, all_in);
    if (cc + NBUF < nchunks) {
      tc::fence_proxy_async_smem();  // reads of this buffer come before the next copy into it
      __syncthreads();
      if (tid == 0) issue(cc + NBUF);
    }
  }
  if (stop < nchunks) {
    if (tid == 0)  // copies in flight (chunks stop .. stop + NBUF - 1) land before the buffer is given back
      for (int cc = stop; cc < min(nchunks, stop + NBUF); ++cc)
        tc::mbar_wait_bounded(&c->bar[cc % NBUF], (cc / NBUF) & 1, abort, 100000000ull);
    for (int x = tid; x < K; x += NT) out[x] = -1;
    __syncthreads();
    return false;
  }
  __syncthreads();

  // 3. exact choice among the candidates, 4. the selection in increasing j, listed over the candidate
  // area (its candidates are no longer needed; it holds at least 2 cap >= K ints)
  select_candidates(cand, min(c->ncand, ccap), R, rb, c, bits);
  __syncthreads();
  write_selection(bits, false, words, K, out, out_s, resident ? reinterpret_cast<const float*>(chunks) : nullptr,
                  s_g, c, reinterpret_cast<int*>(cand_s));
  __syncthreads();  // the buffer may be reused right away
  return true;
}
constexpr int INCL_MAX_WORDS = (1 << 20) / 128 / 32;  // inclusion bitmap of the longest row

// One CTA's part of a token's top-k that several CTAs share, a slice of the row each: the scores
// s_g[j_lo, j_hi) (j_lo a multiple of 128; entries >= n ignored) are scanned against the threshold
// bin of the token's complete histogram into the token's selection bitmap bits_g and candidate list
// cand_g (counter tcnt[0]).  `mine` of the token's `total` units are this CTA's (counter tcnt[1]); the
// CTA that adds the last of them chooses among the candidates, writes the selection (out, out_s),
// clears the histogram and both counters and, for a candidate source (pub_row), publishes the
// token's best blocks.  A consumer passes its list (crow, cM, clg): only its named blocks take part.
// When n <= K the last CTA writes every entry.  Returns 1 if this CTA was the last, 0 if not, -1 if a
// copy timed out (the token's output is then left as it was; the caller raises the flag).  Whole
// CTA; buf: buf_bytes of 128-byte aligned shared memory.
__device__ __noinline__ int topk_part(const float* s_g, uint32_t* hist_g, int n, int K, int j_lo, int j_hi, uint32_t mine,
                         uint32_t total, uint32_t* bits_g, uint64_t* cand_g, uint32_t* tcnt, int32_t* out,
                         float* out_s, uint8_t* buf, size_t buf_bytes, volatile int* abort, const int32_t* crow,
                         int cM, int clg, int32_t* pub_row, int pub_M) {
  const int tid = threadIdx.x, NT = blockDim.x;
  Ctl* c = reinterpret_cast<Ctl*>(buf);
  uint32_t* rb = reinterpret_cast<uint32_t*>(buf + CTL_BYTES);
  uint32_t* hist_s = rb + RBINS;
  uint8_t* chunks = reinterpret_cast<uint8_t*>(hist_s + HIST_BINS);
  uint32_t* incl = reinterpret_cast<uint32_t*>(chunks + (size_t)NBUF * CHUNK * 4);
  uint64_t* cand_s = reinterpret_cast<uint64_t*>(incl + INCL_MAX_WORDS);
  const size_t fixed = CTL_BYTES + RBINS * 4 + HIST_BINS * 4 + (size_t)NBUF * CHUNK * 4 + INCL_MAX_WORDS * 4;
  const uint32_t cap = buf_bytes > fixed ? (uint32_t)((buf_bytes - fixed) / 8) : 0u;
  auto count_done = [&]() {  // this CTA's units, after all its writes; true for the CTA that completes the count
    __threadfence();
    __syncthreads();
    if (tid == 0) c->last = atomicAdd(&tcnt[1], mine) + mine == total;
    __syncthreads();
    return c->last != 0;
  };
  if (n <= K) {  // short context: the last CTA writes every entry, in order
    if (!count_done()) return 0;
    for (int x = tid; x < K; x += NT) {
      out[x] = x < n ? x : -1;
      if (out_s) out_s[x] = x < n ? __ldcg(s_g + x) : -INFINITY;
    }
    for (int x = tid; x < HIST_BINS; x += NT) hist_g[x] = 0u;
    if (tid == 0) tcnt[1] = 0u;
    if (pub_row) {
      __syncthreads();
      publish_blocks(s_g, n, clg, pub_M, pub_row, buf);
    }
    __syncthreads();
    return 1;
  }
  if ((size_t)K > 2 * (size_t)cap) {  // the selection is listed over the candidate area (never short here)
    if (tid == 0) atomicOr(&g_flags_ix, FLAG_TOPK);
    return -1;
  }
  const int n128 = (n + 127) & ~127;
  const int hi = min(j_hi, n128);
  const int nchunks = hi > j_lo ? (hi - j_lo + CHUNK - 1) / CHUNK : 0;
  const int words = bitmap_words(n);
  if (tid == 0) {
    c->bin = 0;
    c->above = 0;
    c->cnt = 0;
    for (int i = 0; i <= NBUF; ++i) tc::mbar_init(&c->bar[i], 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  auto issue = [&](int cc) {
    const uint32_t bytes = (uint32_t)min(CHUNK, hi - j_lo - cc * CHUNK) * 4u;
    uint64_t* bar = &c->bar[cc % NBUF];
    tc::mbar_arrive_expect_tx(bar, bytes);
    tc::bulk_load(chunks + (size_t)(cc % NBUF) * CHUNK * 4, s_g + j_lo + (size_t)cc * CHUNK, bytes, bar);
  };
  if (tid == 0) {
    asm volatile("fence.proxy.async;" ::: "memory");  // scores and counts came through the generic proxy
    tc::mbar_arrive_expect_tx(&c->bar[NBUF], HIST_BINS * 4);
    tc::bulk_load(hist_s, hist_g, HIST_BINS * 4, &c->bar[NBUF]);
    for (int cc = 0; cc < min(NBUF, nchunks); ++cc) issue(cc);
  }
  if (crow) build_incl(crow, cM, clg, n, incl, c);  // while the copies are in flight
  const bool ok = __syncthreads_and(tc::mbar_wait_bounded(&c->bar[NBUF], 0, abort));
  bool all_in = false;  // a consumer whose named blocks hold at most K entries takes all of them
  int stop = ok ? nchunks : 0;
  if (ok) {
    block_find_bin<HIST_BINS / FIND_THREADS>(hist_s, (uint32_t)K, c);
    all_in = crow != nullptr && c->total <= (uint32_t)K;
    const uint32_t bstar = c->bin;
    for (int cc = 0; cc < nchunks; ++cc) {
      if (!__syncthreads_and(tc::mbar_wait_bounded(&c->bar[cc % NBUF], (cc / NBUF) & 1, abort))) {
        stop = cc;
        break;
      }
      scan_chunk(reinterpret_cast<const float*>(chunks + (size_t)(cc % NBUF) * CHUNK * 4),
                 min(CHUNK, hi - j_lo - cc * CHUNK) >> 7, j_lo + cc * CHUNK, n, bstar, bits_g, words, cand_g,
                 (uint32_t)n, &tcnt[0], crow ? incl : nullptr, all_in);
      if (cc + NBUF < nchunks) {
        tc::fence_proxy_async_smem();  // reads of this buffer come before the next copy into it
        __syncthreads();
        if (tid == 0) issue(cc + NBUF);
      }
    }
  }
  if (stop < nchunks || !ok) {
    if (tid == 0) {  // copies in flight land before the buffer is given back
      if (!ok) tc::mbar_wait_bounded(&c->bar[NBUF], 0, abort, 100000000ull);
      for (int cc = stop; cc < min(nchunks, stop + NBUF); ++cc)
        tc::mbar_wait_bounded(&c->bar[cc % NBUF], (cc / NBUF) & 1, abort, 100000000ull);
    }
    __syncthreads();
    return -1;  // the token's count never completes: its output stays as it was (flagged)
  }
  if (!count_done()) return 0;
  // the last CTA: every other part of the token is done with the histogram and the counters
  __threadfence();
  const int R = all_in ? 0 : K - (int)c->above;
  const uint32_t m = min(__ldcg(&tcnt[0]), (uint32_t)n);
  for (int x = tid; x < HIST_BINS; x += NT) hist_g[x] = 0u;
  __syncthreads();  // m is read by every thread before the counters are cleared
  if (tid == 0) {
    tcnt[0] = 0u;
    tcnt[1] = 0u;
  }
  const uint64_t* cand = cand_g;
  if (m <= cap) {
    for (uint32_t i = tid; i < m; i += NT) cand_s[i] = __ldcg(cand_g + i);
    __syncthreads();
    cand = cand_s;
  }
  select_candidates(cand, m, R, rb, c, bits_g);
  __threadfence();
  __syncthreads();
  write_selection(bits_g, true, words, K, out, out_s, nullptr, s_g, c, reinterpret_cast<int*>(cand_s));
  if (pub_row) {
    __syncthreads();
    publish_blocks(s_g, n, clg, pub_M, pub_row, buf);
  }
  __syncthreads();
  return 1;
}
}  // namespace tk

// ------------------------------------------------------------------------------------------------
// SIMT score kernel (any key dtype): thread jj of the CTA owns key tile*128 + jj.
// ------------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(IX_TILE) indexer_score_simt(dsv4_indexer_topk_params p, TopkBufs bufs) {
  extern __shared__ float smem[];
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.y, tile = blockIdx.x, jj = threadIdx.x;
  const int Ih = p.n_heads, d = p.head_dim, qps = p.q_per_seq;
  const int t0 = b * qps;
  const int nc_last = visible_entries(p, t0 + qps - 1);  // largest n_c among the seq's tokens
  const int j0 = tile * IX_TILE;
  if (j0 >= nc_last) return;
  // candidate consumer: the tokens whose list names this tile's block (or whose entries all fit in the
  // top-k); a tile no token counts is not scored
  uint32_t incm = 0xFu;
  if (p.cand_block_size > 0 && !p.cand_write) {
    const int lg = __ffs(p.cand_block_size) - 1;
    incm = 0u;
    for (int k = 0; k < qps; ++k) {
      const int nk = visible_entries(p, t0 + k);
      if (j0 < nk && (nk <= p.topk || cand_names(p.cand_blocks + (int64_t)(t0 + k) * p.cand_topk, p.cand_topk,
                                                   j0 >> lg)))
        incm |= 1u << k;
    }
    if (incm == 0u) return;  // block-uniform
  }

  float* q_s = smem;                         // [qps][Ih][d]
  float* w_s = q_s + qps * Ih * d;           // [qps][Ih]
  const int ld = IX_TILE + 1;
  float* kt_s = w_s + qps * Ih;              // [d + 1][IX_TILE + 1] transposed keys, then row scales

  for (int x = jj; x < qps * Ih * d; x += IX_TILE) {
    const int64_t g = (int64_t)t0 * Ih * d + x;
    q_s[x] = (p.q_dtype == DSV4_F32) ? reinterpret_cast<const float*>(p.q)[g]
                                     : bf16_bits_to_float(reinterpret_cast<const uint16_t*>(p.q)[g]);
  }
  for (int x = jj; x < qps * Ih; x += IX_TILE) w_s[x] = p.weights[(int64_t)t0 * Ih + x];

  // keys: warp w loads keys w, w+4, ... with its 32 lanes spread over the row
  const int warp = jj >> 5, lane = jj & 31;
  const int64_t rb = row_bytes(p.k_dtype, d);
  for (int kk = warp; kk < IX_TILE; kk += IX_TILE / 32) {
    const int j = j0 + kk;
    const uint8_t* row = nullptr;
    if (j < nc_last) {
      const int lp = j / p.page_size;
      const int page = (lp < p.max_pages_per_seq) ? p.block_table[(int64_t)b * p.max_pages_per_seq + lp] : -1;
      if (page >= 0 && page < p.num_pages)
        row = reinterpret_cast<const uint8_t*>(p.k_cache) + ((int64_t)page * p.page_size + j % p.page_size) * rb;
      else if (lane == 0)
        atomicOr(&g_flags_ix, FLAG_PAGE);
    }
    float scale = 1.f;
    if (row != nullptr && p.k_dtype == DSV4_I8_ROWSCALE) scale = *reinterpret_cast<const float*>(row + d);
    for (int e = lane; e < d; e += 32) {
      float v = 0.f;
      if (row != nullptr) {
        if (p.k_dtype == DSV4_F32) v = reinterpret_cast<const float*>(row)[e];
        else if (p.k_dtype == DSV4_BF16) v = bf16_bits_to_float(reinterpret_cast<const uint16_t*>(row)[e]);
        else if (p.k_dtype == DSV4_MXFP4)
          v = e2m1_value((row[e >> 1] >> ((e & 1) * 4)) & 0xFu) * ue8m0_scale(row[d / 2 + e / 32]);
        else v = (float)reinterpret_cast<const int8_t*>(row)[e];
      }
      kt_s[e * ld + kk] = v;
    }
    if (lane == 0) kt_s[d * ld + kk] = scale;
  }
  __syncthreads();

  const int j = j0 + jj;
  const float kscale = kt_s[d * ld + jj];
  for (int k = 0; k < qps; ++k) {
    const int t = t0 + k;
    const int nc = visible_entries(p, t);
    float s = 0.f;
    const float* qk = q_s + k * Ih * d;
    for (int h = 0; h < Ih; ++h) {
      float acc = 0.f;
      const float* qh = qk + h * d;
      for (int e = 0; e < d; ++e) acc = fmaf(qh[e], kt_s[e * ld + jj], acc);
      acc *= kscale;  // int8 keys: code . q, then the row scale
      s = fmaf(w_s[k * Ih + h], fmaxf(acc, 0.f), s);
    }
    const bool on = j < nc && ((incm >> k) & 1u);
    if (on) bufs.scores[(int64_t)t * bufs.nc_stride + j] = s;
    hist_add_warp(bufs.hist + (int64_t)t * HIST_BINS, order_key(s) >> HIST_SHIFT, on);
  }
}

// ------------------------------------------------------------------------------------------------
// Tensor-core score kernel (bf16 queries; bf16 keys, or int8 row-scale keys expanded to bf16 in
// shared memory): D[128 keys x N] = K_tile[128 x d] * Q[N x d]^T with N = q_per_seq * n_heads
// (every query head of the sequence), then per key s_k = sum_h w[k][h] * ReLU(D[key][k*n_heads + h])
// (times the key's row scale for int8 keys).
//
// Persistent CTAs (one per SM), each owning a contiguous range of (sequence, 128-key tile) items: an
// even share of the work, counted as the valid tiles plus a few tiles' worth for every sequence a CTA
// starts on.  Warp 8 streams key tiles with TMA (two 64-row pages x d/64
// K-blocks of 128 B, 128-byte swizzle) into a ring of stages (int8 keys: the two record pages by
// bulk copy into a ring of raw stages, which warps 10-13 expand into the stages), and each
// sequence's Q block into one of two Q slots (one when shared memory is short); its 32 lanes look
// up the block-table pages of 32 items at a time.  One thread of warp 9 issues the tcgen05 MMAs
// (M = 128, K = 16 steps) into a ring of TMEM accumulators.  Warps 0-7 are two epilogue groups of
// four that take alternate tiles: each warp reads its 32 TMEM lanes (one key per thread), applies
// ReLU and the head weights, stores the scores and counts them into its group's shared-memory
// histogram, which is added to the global one when the group leaves a sequence.  The group then
// adds the tiles it scored to the sequence's counter; the group that completes the count records
// the sequence, and after its tiles the CTA runs the top-k of that sequence's tokens itself.
// Every wait is bounded; a timeout raises FLAG_TIMEOUT and all roles drain out.
// ------------------------------------------------------------------------------------------------
namespace ixtc {
constexpr int TILE = 128;
constexpr int KB_BYTES = TILE * 128;         // one 64-dim K-block of a key tile (128 rows x 128 B)
constexpr int NEXP = 4;  // warps expanding raw records (int8, MXFP4 keys), one record row a thread: with 14
                         // warps two SM sub-partitions hold 4 of them, so these instances keep to 128
                         // registers a thread (4 x 32 x 128 = the 16K of a sub-partition)
constexpr int THREADS_BF16 = 320;              // bf16 keys: warps 0-7 epilogue, 8 loads, 9 MMA
constexpr int THREADS = THREADS_BF16 + NEXP * 32;  // raw records: warps 10 .. 9 + NEXP expand
static_assert(THREADS_BF16 / 32 >= tk::SCAN_WARPS_MIN, "the top-k scan covers a chunk with this many warps");
constexpr int W_LOAD = 8, W_MMA = 9;  // warps 10 .. 9 + NEXP expand raw records (int8, MXFP4 caches)
constexpr int SCALE_RING = 16;        // int8 keys: row scales of the last 16 tiles (> stages + accumulators)
constexpr int MAX_STAGES = 8;
constexpr int MAX_RAW = 8;            // raw record pages in flight (int8 keys 2, MXFP4 keys up to 8)
constexpr int KF_BF16 = 0, KF_I8 = 1, KF_MX = 2;  // key formats of the tensor-core kernel
constexpr int FIN_MAX = 64;  // sequences whose top-k one CTA may have to run
constexpr int WSEQ = 8;      // sequences whose head weights and entry counts are loaded up front
constexpr int PRE_MAX = 1024;  // batches up to this size split the key tiles evenly over the CTAs
constexpr int SEQ_START_UNITS = 5;  // tiles' worth of time a CTA spends moving on to another sequence
                                    // (traced: CTAs that do end about 4.5 us, 5 tiles, later)

struct Args {
  const int32_t* positions;
  const int32_t* block_table;
  const float* weights;
  TopkBufs bufs;
  int32_t* topk_idx;
  float* topk_score;
  int64_t num_pages;
  int T, B, qps, Ih, d, ratio, max_pages, tiles_max, max_context, K;
  int fuse_topk;  // the CTA completing a sequence runs its top-k (else a separate sliced launch)
  int bt_div;     // block-table row of item sequence b: b / bt_div (q_per_seq when each query token is
                  // taken as its own sequence, else 1)
  int kf;         // key format: KF_BF16 (TMA tiles), KF_I8 (d int8 + fp32 scale) or KF_MX (MXFP4 records);
                  // int8 and MXFP4 records arrive as bulk-copied pages and are expanded in shared memory
  int rec;        // bytes of one raw record (int8 and MXFP4 keys)
  int nraw;       // raw pages ring depth (pairs of 64-record pages)
  int nqs;        // query slots (2, or 1 when shared memory is short)
  const uint8_t* k_raw;  // int8 key cache
  int N, kblk, stages, tmem_cols, nacc;
  // candidate filtering: lists [T][cM] of blocks of 2^clg entries (2^csh tiles)
  int32_t* cand;
  int cM, clg, csh;
  int cskip;   // consumer with one token a sequence: only the tiles of named blocks are scored
  int cmask;   // consumer with more tokens a sequence: every tile scored, each token's named blocks counted
  int cwrite;  // the source: publishes each token's best blocks after its top-k
};

struct Smem {
  uint64_t full[MAX_STAGES], empty[MAX_STAGES], dfull[4], dempty[4], qfull[2], qempty[2], done, ebar[2];
  uint64_t raw_full[MAX_RAW], raw_empty[MAX_RAW], sready[SCALE_RING];  // raw records; int8 row scales
  int fin[FIN_MAX];
  int nc_tab[WSEQ][DSV4_MAX_Q_PER_SEQ];
  int pre[PRE_MAX];  // exclusive prefix of the sequences' key tiles (balanced item ranges)
  int range[2];      // this CTA's [lo, hi) of the (sequence, tile) grid
  uint32_t nfin;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ int seq_entries(const Args& a, int b) {
  return visible_entries(a.positions, b * a.qps + a.qps - 1, a.max_context, a.ratio);
}

__device__ __forceinline__ int page_of(const Args& a, int b, int lp) {
  if (lp >= a.max_pages) return -1;
  const int pg = a.block_table[(int64_t)(b / a.bt_div) * a.max_pages + lp];
  if (pg < 0 || pg >= a.num_pages) {
    atomicOr(&g_flags_ix, FLAG_PAGE);
    return -1;
  }
  return pg;
}

// Key tiles of sequence b (nc entries) that the kernel scores: every tile, or for a candidate consumer
// with one token a sequence and nc > K, the tiles of the named blocks that hold entries (the named
// blocks increase, so only the last of them can be partial).
__device__ int live_tiles(const Args& a, int b, int nc) {
  const int nt = (nc + TILE - 1) / TILE;
  if (!a.cskip || nc <= a.K) return nt;
  const int32_t* row = a.cand + (int64_t)b * a.cM;
  const int last = (nt - 1) >> a.csh;  // the block holding the last entry
  int prev = -1, tiles = 0;
  for (int i0 = 0; i0 < a.cM; i0 += 8) {
    int blk[8];  // eight list entries loaded together
#pragma unroll
    for (int u = 0; u < 8; ++u) blk[u] = i0 + u < a.cM ? __ldg(row + i0 + u) : -1;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (blk[u] <= prev || blk[u] > last) return tiles;  // the run ends, or the block lies past the entries
      tiles += min(1 << a.csh, nt - (blk[u] << a.csh));
      prev = blk[u];
    }
  }
  return tiles;
}

// Tile of slot v of sequence b: the slot itself, or slot v of the concatenated named blocks.
__device__ __forceinline__ int slot_tile(const Args& a, const int32_t* row, int v) {
  return row ? (__ldg(row + (v >> a.csh)) << a.csh) | (v & ((1 << a.csh) - 1)) : v;
}
__device__ __forceinline__ const int32_t* slot_row(const Args& a, int b, int nc) {
  return (a.cskip && nc > a.K) ? a.cand + (int64_t)b * a.cM : nullptr;
}

// Walks the items of the flat range [lo, hi) of the (sequence, slot) grid in order without divisions;
// slot v < live_tiles of sequence b is its v-th scored tile.
struct ItemIter {
  int it, hi, b, v, nt, nc, tile;
  __device__ __forceinline__ void enter(const Args& a) {
    nc = seq_entries(a, b);
    nt = live_tiles(a, b, nc);
  }
  __device__ __forceinline__ void init(const Args& a, int lo, int hi_) {
    it = lo;
    hi = hi_;
    b = lo / a.tiles_max;
    v = lo % a.tiles_max;
    nt = 0;
    if (it < hi) enter(a);
    skip(a);
  }
  // moves past slots beyond the end of the current sequence (nt <= tiles_max)
  __device__ __forceinline__ void skip(const Args& a) {
    while (it < hi && v >= nt) {
      it += a.tiles_max - v;
      ++b;
      v = 0;
      if (it < hi) enter(a);
    }
    if (it < hi) tile = slot_tile(a, slot_row(a, b, nc), v);
  }
  __device__ __forceinline__ void next(const Args& a) {
    ++it;
    ++v;
    skip(a);
  }
  __device__ __forceinline__ bool valid() const { return it < hi; }
};

// An epilogue group leaves sequence b after scoring `ntile` of its tiles: its shared histogram is
// added to the global one and cleared, its writes are made visible device-wide, and its tiles are
// added to the sequence's counter; the group that completes it records b for the CTA's top-k.
// Called by the group's four warps, with bounded group barriers.
__device__ __forceinline__ bool finish_seq(const Args& a, Smem* sm, uint32_t* hist_g, int b, int ntile, int g, int row,
                                           uint32_t* ephase, volatile int* abort) {
  uint32_t tiles = 0;
  if (row == 0) tiles = (uint32_t)live_tiles(a, b, seq_entries(a, b));  // its load overlaps the flush
  if (!tc::group_sync(&sm->ebar[g], ephase, abort)) return false;
  // 4 bins at a time (the histograms are 16-byte aligned, qps x HIST_BINS a multiple of 512)
  uint4* h4 = reinterpret_cast<uint4*>(hist_g);
#pragma unroll 4
  for (int x4 = row; x4 < a.qps * (HIST_BINS / 4); x4 += 128) {
    const uint4 v = h4[x4];
    if (v.x | v.y | v.z | v.w) {
      const int x = 4 * x4;
      uint32_t* dst = a.bufs.hist + (int64_t)(b * a.qps + x / HIST_BINS) * HIST_BINS + (x % HIST_BINS);
      if (v.x) atomicAdd(dst, v.x);
      if (v.y) atomicAdd(dst + 1, v.y);
      if (v.z) atomicAdd(dst + 2, v.z);
      if (v.w) atomicAdd(dst + 3, v.w);
      h4[x4] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  __threadfence();  // this thread's scores and histogram counts before the counter below
  if (!tc::group_sync(&sm->ebar[g], ephase, abort)) return false;
  if (row == 0) {
    const uint32_t prev = atomicAdd(&a.bufs.seq_done[b], (uint32_t)ntile);
    if (prev + (uint32_t)ntile == tiles) {
      a.bufs.seq_done[b] = 0u;  // complete: no CTA adds to it again in this call; cleared for the next
      // the other CTAs' scores and counts (each fenced before its own counter update) are visible to
      // this CTA's top-k, which reads them after a CTA barrier
      __threadfence();
      const uint32_t i = atomicAdd(&sm->nfin, 1u);
      if (i < FIN_MAX) sm->fin[i] = b;
      else atomicOr(&g_flags_ix, FLAG_TOPK);
    }
  }
  return true;
}

// The MMAs of one key tile: K-block kb, 16-dim step s of the keys (A: 128 rows of 128 B a K-block)
// against the queries (B: N rows of 128 B a K-block), accumulating from the second on.
template <int KBLK>
__device__ __forceinline__ void issue_tile(uint32_t d_tmem, uint64_t ad, uint64_t bd, uint32_t idesc, int N) {
#pragma unroll
  for (int kb = 0; kb < KBLK; ++kb)
#pragma unroll
    for (int s = 0; s < 4; ++s)
      tc::mma_bf16(d_tmem, ad + (uint64_t)((kb * KB_BYTES + s * 32) >> 4), bd + (uint64_t)((kb * N * 128 + s * 32) >> 4),
                   idesc, (kb | s) != 0);
}

// One instance per key format: the bf16 one has no expanding warps (320 threads, at most three warps
// on a sub-partition: 168 registers a thread) and none of the raw-record branches; the raw-record
// ones run 14 warps at 128 registers a thread (the 512-thread bound sets that cap).
template <int KF>
__global__ void __launch_bounds__(KF == 0 ? THREADS_BF16 : 512, 1)
    indexer_score_tc(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap, Args a) {
  constexpr bool RAW = KF != KF_BF16;  // records bulk-copied as pages and expanded to bf16 by warps 10-13
  constexpr bool I8 = KF == KF_I8;     // int8 records: row scales applied to the finished score
  extern __shared__ __align__(1024) uint8_t dsm[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  const int q_bytes = a.kblk * a.N * 128;
  const int stage_bytes = a.kblk * KB_BYTES;
  uint8_t* stage_mem = base;                                               // stages x stage_bytes
  uint8_t* q_mem = base + a.stages * stage_bytes;                          // nqs slots x q_bytes
  const int raw_page = 64 * a.rec, raw_stage = 2 * raw_page;             // raw records: 64 a page, 2 pages a tile
  uint8_t* raw_mem = q_mem + a.nqs * q_bytes;                              // raw records: nraw stages
  float* scale_s = reinterpret_cast<float*>(raw_mem + (RAW ? a.nraw * raw_stage : 0));  // int8: SCALE_RING x 128
  float* w_s = scale_s + (I8 ? SCALE_RING * TILE : 0);                  // 2 groups x 256 floats
  float* w_tab = w_s + 2 * 256;                                            // WSEQ x 128 floats
  uint32_t* hist_s = reinterpret_cast<uint32_t*>(w_tab + WSEQ * 128);      // 2 groups x qps x HIST_BINS
  Smem* sm = reinterpret_cast<Smem*>(hist_s + 2 * a.qps * HIST_BINS);
  volatile int* abort = &sm->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = a.B * a.tiles_max;
  // Set-up that reads nothing in global memory runs before the dependency wait, while the kernel
  // ahead finishes (the launch lets this grid start early): the loading warp initialises the
  // mbarriers and prefetches the tensor maps, the MMA warp allocates TMEM, the epilogue warps clear
  // their histograms.  After the wait the loading warp works out the CTA's range [lo, hi) of the
  // (sequence, tile) grid (an even share of the work, from a prefix over the sequences' tile counts),
  // announces it on named barrier BAR_SETUP and goes straight on to loading; the MMA warp announces
  // TMEM on BAR_TMEM to the epilogue warps, which meanwhile load the head weights and entry counts of
  // the CTA's sequences.
  constexpr uint32_t BAR_SETUP = 1, BAR_TMEM = 2, BAR_EPI = 3;
  if (warp == W_LOAD) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&kmap);
      tc::tma_prefetch_desc(&qmap);
      // L2 hints while the kernel ahead finishes (they hand no value over): the positions, and for the
      // first two sequences of the CTA's share of an even split (its range proper needs the positions)
      // their block-table rows, queries and head weights
      tc::prefetch_l2(a.positions, (size_t)a.T * 4);
      const int g0 = (int)((int64_t)blockIdx.x * total / gridDim.x);
      for (int b = g0 / a.tiles_max; b < min(a.B, g0 / a.tiles_max + 2); ++b) {
        tc::prefetch_l2(a.block_table + (int64_t)(b / a.bt_div) * a.max_pages, (size_t)a.max_pages * 4);
        tc::prefetch_l2(a.weights + (int64_t)b * a.qps * a.Ih, (size_t)a.N * 4);
        for (int kb = 0; kb < a.kblk; ++kb) tc::tma_prefetch_2d(&qmap, kb * 64, b * a.qps * a.Ih);
      }
      for (int s = 0; s < a.stages; ++s) {
        tc::mbar_init(&sm->full[s], RAW ? NEXP : 1);  // raw records: the expanding warps; else the loader (+ bytes)
        tc::mbar_init(&sm->empty[s], 1);
      }
      for (int i = 0; i < MAX_RAW; ++i) {
        tc::mbar_init(&sm->raw_full[i], 1);
        tc::mbar_init(&sm->raw_empty[i], NEXP);
      }
      for (int i = 0; i < SCALE_RING; ++i) tc::mbar_init(&sm->sready[i], NEXP);
      for (int i = 0; i < 4; ++i) {
        tc::mbar_init(&sm->dfull[i], 1);
        tc::mbar_init(&sm->dempty[i], 4);
      }
      for (int i = 0; i < 2; ++i) {
        tc::mbar_init(&sm->qfull[i], 1);
        tc::mbar_init(&sm->qempty[i], 1);
      }
      tc::mbar_init(&sm->done, 1);
      tc::mbar_init(&sm->ebar[0], 4);
      tc::mbar_init(&sm->ebar[1], 4);
      sm->nfin = 0;
      sm->abort = 0;
      tc::fence_barrier_init();
    }
    pdl_wait();  // nothing below runs before the kernels ahead of this one have finished
    int r0 = (int)((int64_t)blockIdx.x * total / gridDim.x), r1 = (int)((int64_t)(blockIdx.x + 1) * total / gridDim.x);
    if (a.B <= 32) {
      // the same as below with one sequence a lane, in registers: the prefix by shuffles, and the
      // sequence a work unit falls in by one ballot (the last lane whose prefix is not above it)
      const int nt = lane < a.B ? live_tiles(a, lane, seq_entries(a, lane)) : 0;
      const int v = nt > 0 ? nt + SEQ_START_UNITS : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      const int running = __shfl_sync(0xffffffffu, incl, 31), pre_b = incl - v;
      auto dense = [&](int x) {
        const unsigned m = __ballot_sync(0xffffffffu, lane < a.B && pre_b <= x);  // bit 0 always set
        const int l = 31 - __clz(m);
        const int pl = __shfl_sync(0xffffffffu, pre_b, l);
        return x >= running ? total : l * a.tiles_max + max(0, x - pl - SEQ_START_UNITS);
      };
      r0 = dense((int)((int64_t)blockIdx.x * running / gridDim.x));
      r1 = dense((int)((int64_t)(blockIdx.x + 1) * running / gridDim.x));
    } else if (a.B <= PRE_MAX) {
      // the work of each sequence in tile units (its tiles, plus SEQ_START_UNITS for starting on it:
      // the histogram flush and counter update of the sequence left and the next queries), all loaded
      // first (independent loads, all in flight together), then the scan
#pragma unroll 4
      for (int b = lane; b < a.B; b += 32) {
        const int nt = live_tiles(a, b, seq_entries(a, b));
        sm->pre[b] = nt > 0 ? nt + SEQ_START_UNITS : 0;
      }
      __syncwarp();
      int running = 0;
      for (int b0 = 0; b0 < a.B; b0 += 32) {
        const int b = b0 + lane;
        const int v = b < a.B ? sm->pre[b] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += u;
        }
        if (b < a.B) sm->pre[b] = running + incl - v;
        running += __shfl_sync(0xffffffffu, incl, 31);
      }
      __syncwarp();
      auto dense = [&](int x) {  // grid position of work unit x (a sequence's start units: its first tile)
        if (x >= running) return total;
        int l = 0, r = a.B - 1;  // last b with pre[b] <= x (it has a tile, since x < pre[b + 1])
        while (l < r) {
          const int m = (l + r + 1) >> 1;
          if (sm->pre[m] <= x) l = m;
          else r = m - 1;
        }
        return l * a.tiles_max + max(0, x - sm->pre[l] - SEQ_START_UNITS);
      };
      r0 = dense((int)((int64_t)blockIdx.x * running / gridDim.x));
      r1 = dense((int)((int64_t)(blockIdx.x + 1) * running / gridDim.x));
    }
    if (lane == 0) {
      sm->range[0] = r0;
      sm->range[1] = r1;
    }
    __syncwarp();
    tc::named_bar_arrive(BAR_SETUP, blockDim.x);
  } else if (warp == W_MMA) {
    tc::tmem_alloc(&sm->tmem_base, a.tmem_cols);
    tc::tmem_relinquish();
    tc::tc_fence_before();
    pdl_wait();
    tc::named_bar_arrive(BAR_TMEM, 32 + 256);
    tc::named_bar_sync(BAR_SETUP, blockDim.x);
  } else if (warp < W_LOAD) {
    const int g = warp >> 2;
    for (int x = threadIdx.x & 127; x < a.qps * HIST_BINS; x += 128) hist_s[g * a.qps * HIST_BINS + x] = 0;
    pdl_wait();
    tc::named_bar_sync(BAR_SETUP, blockDim.x);
  } else {
    pdl_wait();
    tc::named_bar_sync(BAR_SETUP, blockDim.x);
  }
  const int lo = sm->range[0], hi = sm->range[1];
  // every thread is past its dependency wait: the kernels after this one may start from here on (so
  // when one of them starts, everything before this kernel has finished)
  pdl_launch_dependents();
  // head weights and per-token entry counts of the CTA's sequences, when there are few of them
  // (epilogue warps only)
  const int b_first = lo / a.tiles_max;
  const int nseq_rng = hi > lo ? (hi - 1) / a.tiles_max - b_first + 1 : 0;
  const bool pre = nseq_rng <= WSEQ;
  if (warp < W_LOAD) {
    if (pre) {
      for (int x = threadIdx.x; x < nseq_rng * a.N; x += 256) w_tab[x] = a.weights[(int64_t)b_first * a.qps * a.Ih + x];
      for (int x = threadIdx.x; x < nseq_rng * a.qps; x += 256)
        sm->nc_tab[x / a.qps][x % a.qps] =
            visible_entries(a.positions, (b_first + x / a.qps) * a.qps + x % a.qps, a.max_context, a.ratio);
    }
    tc::named_bar_sync(BAR_EPI, 256);
    tc::named_bar_sync(BAR_TMEM, 32 + 256);
  }
  tc::tc_fence_after();
  const uint32_t tmem = sm->tmem_base;  // read by the MMA and epilogue warps only

  if (warp == W_LOAD) {
    // ---------------- TMA producer (lane 0 issues; all lanes look up pages 32 items at a time)
    int stage = 0, cur_b = -1, qn = 0, rn = 0;
    uint32_t phase = 0;
    bool stop = false;
    const uint64_t pol = tc::l2_policy_evict_first();
    ItemIter cur;  // every lane walks the same items; lane i keeps the i-th of each group of 32
    cur.init(a, lo, hi);
    // the first group is only as large as the stages, so that the first copies go out after a few steps
    // of the walk (each step is a short dependent chain; a whole group of 32 took about 3 us)
    int group = a.stages;
    while (cur.valid() && !stop) {
      int vb = -1, pg0 = -1, pg1 = -1, j0 = 0, nc = 0;
      for (int i = 0; i < group && cur.valid(); ++i) {
        if (lane == i) {
          vb = cur.b;
          j0 = cur.tile * TILE;
          nc = cur.nc;
        }
        cur.next(a);
      }
      if (vb >= 0) {  // the block-table pages of the 32 items, looked up together
        pg0 = page_of(a, vb, j0 / 64);
        pg1 = (j0 + 64 < nc) ? page_of(a, vb, j0 / 64 + 1) : -1;
      }
      for (int i = 0; i < group; ++i) {
        const int b = __shfl_sync(0xffffffffu, vb, i);
        const int p0 = __shfl_sync(0xffffffffu, pg0, i);
        const int p1 = __shfl_sync(0xffffffffu, pg1, i);
        if (b < 0) continue;
        int ok = 1;
        if (lane == 0) {
          if (b != cur_b) {
            const int slot = qn % a.nqs;
            ok = tc::mbar_wait_bounded(&sm->qempty[slot], ((qn / a.nqs) & 1) ^ 1, abort);
            if (ok) {
              tc::mbar_arrive_expect_tx(&sm->qfull[slot], q_bytes);
              for (int kb = 0; kb < a.kblk; ++kb)
                tc::tma_load_2d(q_mem + slot * q_bytes + kb * a.N * 128, &qmap, kb * 64, b * a.qps * a.Ih,
                                &sm->qfull[slot]);
              ++qn;
              cur_b = b;
            }
          }
          if (ok && RAW) {
            // raw record pages (whole records, untiled bulk copies) into raw stage rn % nraw
            const int rs = rn % a.nraw;
            ok = tc::mbar_wait_bounded(&sm->raw_empty[rs], ((rn / a.nraw) & 1) ^ 1, abort);
            if (ok) {
              tc::mbar_arrive_expect_tx(&sm->raw_full[rs], (uint32_t)((p0 >= 0) + (p1 >= 0)) * (uint32_t)raw_page);
              if (p0 >= 0)
                tc::bulk_load(raw_mem + rs * raw_stage, a.k_raw + (int64_t)p0 * raw_page, raw_page, &sm->raw_full[rs]);
              if (p1 >= 0)
                tc::bulk_load(raw_mem + rs * raw_stage + raw_page, a.k_raw + (int64_t)p1 * raw_page, raw_page,
                              &sm->raw_full[rs]);
              ++rn;
            }
          } else if (ok) ok = tc::mbar_wait_bounded(&sm->empty[stage], phase ^ 1, abort);
          if (ok && !RAW) {
            const uint32_t bytes = (uint32_t)((p0 >= 0) + (p1 >= 0)) * a.kblk * (KB_BYTES / 2);
            uint8_t* st = stage_mem + stage * stage_bytes;
            tc::mbar_arrive_expect_tx(&sm->full[stage], bytes);
            for (int kb = 0; kb < a.kblk; ++kb) {  // keys are read once: evicted from L2 first
              if (p0 >= 0) tc::tma_load_2d_hint(st + kb * KB_BYTES, &kmap, kb * 64, p0 * 64, &sm->full[stage], pol);
              if (p1 >= 0)
                tc::tma_load_2d_hint(st + kb * KB_BYTES + KB_BYTES / 2, &kmap, kb * 64, p1 * 64, &sm->full[stage],
                                     pol);
            }
            if (++stage == a.stages) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          stop = true;
          break;
        }
      }
      group = 32;
    }
    if (lane == 0) {
      // drain: every issued load must land before the CTA may exit (a completed phase returns at once)
      if (RAW) {
        for (int r = (rn > a.nraw ? rn - a.nraw : 0); r < rn; ++r)
          tc::mbar_wait_bounded(&sm->raw_full[r % a.nraw], (r / a.nraw) & 1, abort, 100000000ull);
      } else {
        for (int s = 0; s < a.stages; ++s) {
          const int parity = (s < stage) ? (int)phase : (int)(phase ^ 1);
          tc::mbar_wait_bounded(&sm->full[s], parity, abort, 100000000ull);
        }
      }
      for (int q = (qn > a.nqs ? qn - a.nqs : 0); q < qn; ++q)  // the last load into each query slot
        tc::mbar_wait_bounded(&sm->qfull[q % a.nqs], (q / a.nqs) & 1, abort, 100000000ull);
    }
  } else if (warp == W_MMA) {
    if (lane == 0) {
      // ---------------- MMA issuer (one thread; its instruction issue sets the pace of the key
      // stream, so the descriptors are built once and advanced by constant offsets: a descriptor's
      // start address is its low 14 bits in 16-byte units, and every shared address here is below
      // 256 KB)
      const uint32_t idesc = tc::idesc_bf16_f32(TILE, a.N);
      const uint64_t adesc0 = tc::sdesc_k_sw128(tc::smem_addr(stage_mem));
      const uint64_t qdesc0 = tc::sdesc_k_sw128(tc::smem_addr(q_mem));
      int stage = 0, acc = 0, cur_b = -1, qn = 0, slot = 0;
      uint32_t phase = 0, aphase = 0;
      ItemIter cur;
      cur.init(a, lo, hi);
      while (cur.valid()) {
        if (cur.b != cur_b) {
          slot = qn % a.nqs;
          if (!tc::mbar_wait_bounded(&sm->qfull[slot], (qn / a.nqs) & 1, abort)) break;
          ++qn;
          cur_b = cur.b;
        }
        if (!tc::mbar_wait_bounded(&sm->full[stage], phase, abort)) break;
        if (!tc::mbar_wait_bounded(&sm->dempty[acc], aphase ^ 1, abort)) break;
        tc::tc_fence_after();
        const uint64_t ad = adesc0 + (uint64_t)((stage * stage_bytes) >> 4);
        const uint64_t bd = qdesc0 + (uint64_t)((slot * q_bytes) >> 4);
        const uint32_t d_tmem = tmem + (uint32_t)(acc * a.N);
        if (a.kblk == 2)
          issue_tile<2>(d_tmem, ad, bd, idesc, a.N);
        else
          issue_tile<1>(d_tmem, ad, bd, idesc, a.N);
        tc::mma_commit(&sm->empty[stage]);
        tc::mma_commit(&sm->dfull[acc]);
        const int b_now = cur.b;
        cur.next(a);
        if (!cur.valid() || cur.b != b_now) tc::mma_commit(&sm->qempty[slot]);
        if (++stage == a.stages) {
          stage = 0;
          phase ^= 1;
        }
        if (++acc == a.nacc) {
          acc = 0;
          aphase ^= 1;
        }
      }
      tc::mma_commit(&sm->done);
      tc::mbar_wait_bounded(&sm->done, 0, abort, 100000000ull);
    }
  } else if (warp > W_MMA) {
    // ---------------- raw records: warps 10 .. 9 + NEXP expand each tile's records into the bf16 stage
    // (K-major, 128-byte swizzle, as TMA would write it), thread x taking rows x, x + 32 NEXP, ... of the
    // tile.  int8 keys:
    // a code is exact in bf16 and the row scales are kept for the epilogue (s = scale * sum_h w_h
    // ReLU(q_h . code), since ReLU(c x) = c ReLU(x) for c > 0).  MXFP4 keys: each E2M1 code's sign, 2
    // exponent bits and mantissa bit are placed into a bf16's sign, lowest exponent bits and top
    // mantissa bit, which is the bf16 code x 2^-126 (exponent-0 codes land on bf16 subnormals), and two
    // bf16x2 multiplies by powers of two, 2^min(e - 1, 127) and 2^max(e - 128, 0), give code x 2^(e - 127)
    // exactly for block exponent bytes e up to 252.
    if (RAW) {
      const int x = threadIdx.x - (W_MMA + 1) * 32;  // 0 .. 32 NEXP - 1
      const int rec = a.rec;
      ItemIter cur;
      cur.init(a, lo, hi);
      for (int k = 0; cur.valid(); cur.next(a), ++k) {
        const int rs = k % a.nraw, st = k % a.stages;
        if (!tc::mbar_wait_bounded(&sm->raw_full[rs], (k / a.nraw) & 1, abort) ||
            !tc::mbar_wait_bounded(&sm->empty[st], ((k / a.stages) & 1) ^ 1, abort))
          break;
        const int j0 = cur.tile * TILE;
        uint8_t* stg = stage_mem + st * stage_bytes;
        float* sc = scale_s + (k % SCALE_RING) * TILE;
        for (int r = x; r < TILE; r += NEXP * 32) {
          if (j0 + r >= cur.nc) break;  // no key from here on: those D rows are never used
          const uint8_t* src = raw_mem + rs * raw_stage + (r >> 6) * raw_page + (r & 63) * rec;
          uint8_t* dstrow = stg + (r >> 3) * 1024 + (r & 7) * 128;
          if (I8) {
            for (int g8 = 0; g8 < a.d / 8; ++g8) {  // 8 codes -> one 16-byte chunk of 8 bf16
              uint32_t o[4];
#pragma unroll
              for (int h4 = 0; h4 < 2; ++h4) {
                const uint32_t w = *reinterpret_cast<const uint32_t*>(src + 8 * g8 + 4 * h4) ^ 0x80808080u;
                // code c as the float 2^23 + (c + 128), minus 2^23 + 128: exact; a small integer's bf16
                // bits are the top half of its fp32 bits
                float f[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  f[q] = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u | (uint32_t)q)) - 8388736.0f;
                o[2 * h4] = __byte_perm(__float_as_uint(f[0]), __float_as_uint(f[1]), 0x7632u);
                o[2 * h4 + 1] = __byte_perm(__float_as_uint(f[2]), __float_as_uint(f[3]), 0x7632u);
              }
              const int kb = g8 >> 3, ch = g8 & 7;
              *reinterpret_cast<uint4*>(dstrow + kb * KB_BYTES + ((ch ^ (r & 7)) << 4)) =
                  make_uint4(o[0], o[1], o[2], o[3]);
            }
            sc[r] = *reinterpret_cast<const float*>(src + a.d);
          } else {
            const uint32_t* code_w = reinterpret_cast<const uint32_t*>(src);  // d / 8 words of 8 codes
            for (int blk = 0; blk < a.d / 32; ++blk) {
              const uint32_t e = src[a.d / 2 + blk];
              const uint32_t e1 = e <= 128u ? e - 1u : 127u, e2 = e <= 128u ? 0u : e - 128u;
              const uint32_t s1b = ((e1 + 127u) << 7) * 0x00010001u, s2b = ((e2 + 127u) << 7) * 0x00010001u;
              const __nv_bfloat162 s1 = *reinterpret_cast<const __nv_bfloat162*>(&s1b);
              const __nv_bfloat162 s2 = *reinterpret_cast<const __nv_bfloat162*>(&s2b);
              uint32_t wv[4];
#pragma unroll
              for (int w4 = 0; w4 < 4; ++w4) wv[w4] = code_w[blk * 4 + w4];
#pragma unroll
              for (int w4 = 0; w4 < 4; ++w4) {  // 8 codes -> one 16-byte chunk of 8 bf16
                uint32_t o[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  const uint32_t b = (wv[w4] >> (8 * q)) & 0xFFu;
                  uint32_t v = ((b & 0x07u) << 6) | ((b & 0x08u) << 12) | ((b & 0x70u) << 18) | ((b & 0x80u) << 24);
                  __nv_bfloat162 bv = *reinterpret_cast<__nv_bfloat162*>(&v);
                  bv = __hmul2(__hmul2(bv, s1), s2);
                  o[q] = *reinterpret_cast<uint32_t*>(&bv);
                }
                const int g8 = blk * 4 + w4, kb = g8 >> 3, ch = g8 & 7;
                *reinterpret_cast<uint4*>(dstrow + kb * KB_BYTES + ((ch ^ (r & 7)) << 4)) =
                    make_uint4(o[0], o[1], o[2], o[3]);
              }
            }
          }
        }
        tc::fence_proxy_async_smem();  // the expanded tile is read by the tensor cores
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(&sm->raw_empty[rs]);
          tc::mbar_arrive(&sm->full[st]);
          if (I8) tc::mbar_arrive(&sm->sready[k % SCALE_RING]);
        }
      }
    }
  } else {
    // ---------------- epilogue: warps 0-7 in two groups of four; group g takes the CTA's items
    // g, g + 2, ...; thread = key row (TMEM lane)
    const int g = warp >> 2, row = (warp & 3) * 32 + lane;
    const float* w_g = w_s + g * 256;
    uint32_t* hist_g = hist_s + g * a.qps * HIST_BINS;
    int cur_b = -1, ntile = 0;
    uint32_t ephase = 0;
    bool ok = true;
    int nc_tok[DSV4_MAX_Q_PER_SEQ] = {0, 0, 0, 0};
    ItemIter cur;
    cur.init(a, lo, hi);
    for (int k = 0; cur.valid(); cur.next(a), ++k) {
      if ((k & 1) != g) continue;
      const int b = cur.b;
      if (b != cur_b) {
        if (cur_b >= 0 && !finish_seq(a, sm, hist_g, cur_b, ntile, g, row, &ephase, abort)) {
          ok = false;
          break;
        }
        if (pre) {
          w_g = w_tab + (b - b_first) * a.N;
#pragma unroll
          for (int q = 0; q < DSV4_MAX_Q_PER_SEQ; ++q) nc_tok[q] = q < a.qps ? sm->nc_tab[b - b_first][q] : 0;
        } else {
          float* wl = w_s + g * 256;
          for (int x = row; x < a.N; x += 128) wl[x] = a.weights[(int64_t)b * a.qps * a.Ih + x];
#pragma unroll
          for (int q = 0; q < DSV4_MAX_Q_PER_SEQ; ++q)
            nc_tok[q] = q < a.qps ? visible_entries(a.positions, b * a.qps + q, a.max_context, a.ratio) : 0;
          if (!tc::group_sync(&sm->ebar[g], &ephase, abort)) {
            ok = false;
            break;
          }
        }
        cur_b = b;
        ntile = 0;
      }
      const int acc = k % a.nacc;
      const uint32_t aphase = (uint32_t)((k / a.nacc) & 1);
      if (!tc::mbar_wait_bounded(&sm->dfull[acc], aphase, abort)) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      float kscale = 1.f;
      if (I8) {
        if (!tc::mbar_wait_bounded(&sm->sready[k % SCALE_RING], (k / SCALE_RING) & 1, abort)) {
          ok = false;
          break;
        }
        kscale = scale_s[(k % SCALE_RING) * TILE + row];
      }
      float sk[DSV4_MAX_Q_PER_SEQ] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(acc * a.N);
      // raw-record instances read 32 columns at a time (one token's heads: n_heads is a multiple of
      // 32) to keep to their 128 registers
      for (int c0 = 0; c0 < a.N && RAW; c0 += 32) {
        uint32_t r[32];
        tc::tmem_ld32_nowait(lane_addr + c0, r);
        tc::tmem_wait_ld_regs<32>(r);
        const float4* w4 = reinterpret_cast<const float4*>(w_g + c0);
        float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 w = w4[i];
          p[0] = fmaf(w.x, fmaxf(__uint_as_float(r[4 * i + 0]), 0.f), p[0]);
          p[1] = fmaf(w.y, fmaxf(__uint_as_float(r[4 * i + 1]), 0.f), p[1]);
          p[2] = fmaf(w.z, fmaxf(__uint_as_float(r[4 * i + 2]), 0.f), p[2]);
          p[3] = fmaf(w.w, fmaxf(__uint_as_float(r[4 * i + 3]), 0.f), p[3]);
        }
        const int k0 = c0 / a.Ih;
#pragma unroll
        for (int q = 0; q < DSV4_MAX_Q_PER_SEQ; ++q)
          if (q == k0) sk[q] += (p[0] + p[1]) + (p[2] + p[3]);
      }
      for (int c0 = 0; c0 < a.N && !RAW; c0 += 64) {
        uint32_t r[64];
        tc::tmem_ld32_nowait(lane_addr + c0, r);
        tc::tmem_ld32_nowait(lane_addr + c0 + 32, r + 32);
        tc::tmem_wait_ld_regs<64>(r);
        const float4* w4 = reinterpret_cast<const float4*>(w_g + c0);
        float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float4 w = w4[i];
          p[0] = fmaf(w.x, fmaxf(__uint_as_float(r[4 * i + 0]), 0.f), p[0]);
          p[1] = fmaf(w.y, fmaxf(__uint_as_float(r[4 * i + 1]), 0.f), p[1]);
          p[2] = fmaf(w.z, fmaxf(__uint_as_float(r[4 * i + 2]), 0.f), p[2]);
          p[3] = fmaf(w.w, fmaxf(__uint_as_float(r[4 * i + 3]), 0.f), p[3]);
        }
        // n_heads is a multiple of 32: the two 32-column halves may belong to different tokens
        const int k0 = c0 / a.Ih, k1 = (c0 + 32) / a.Ih;
        if (k0 == k1) {
#pragma unroll
          for (int q = 0; q < DSV4_MAX_Q_PER_SEQ; ++q)
            if (q == k0) sk[q] += (p[0] + p[1]) + (p[2] + p[3]);
        } else {
          // recompute the halves separately (only when a token boundary falls mid-chunk)
          float h0 = 0.f, h1 = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) h0 = fmaf(w_g[c0 + i], fmaxf(__uint_as_float(r[i]), 0.f), h0);
#pragma unroll
          for (int i = 32; i < 64; ++i) h1 = fmaf(w_g[c0 + i], fmaxf(__uint_as_float(r[i]), 0.f), h1);
#pragma unroll
          for (int q = 0; q < DSV4_MAX_Q_PER_SEQ; ++q) {
            if (q == k0) sk[q] += h0;
            if (q == k1) sk[q] += h1;
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm->dempty[acc]);
      const int j = cur.tile * TILE + row;
      uint32_t incm = 0xFu;  // tokens that count this tile (a consumer: those whose list names its block)
      if (a.cmask) {
        incm = 0u;
#pragma unroll
        for (int q = 0; q < DSV4_MAX_Q_PER_SEQ; ++q)
          if (q < a.qps && (nc_tok[q] <= a.K ||
                            cand_names(a.cand + (int64_t)(b * a.qps + q) * a.cM, a.cM, cur.tile >> a.csh)))
            incm |= 1u << q;
      }
#pragma unroll
      for (int q = 0; q < DSV4_MAX_Q_PER_SEQ; ++q) {
        if (q < a.qps) {
          sk[q] *= kscale;  // 1 for bf16 keys
          const int t = b * a.qps + q;
          const bool on = j < nc_tok[q] && ((incm >> q) & 1u);
          if (on) a.bufs.scores[(int64_t)t * a.bufs.nc_stride + j] = sk[q];
          hist_add_warp(hist_g + q * HIST_BINS, order_key(sk[q]) >> HIST_SHIFT, on);
        }
      }
      ++ntile;
    }
    if (ok && cur_b >= 0) finish_seq(a, sm, hist_g, cur_b, ntile, g, row, &ephase, abort);
  }
  __syncthreads();
  if (threadIdx.x == 0 && sm->abort) atomicOr(&g_flags_ix, FLAG_TIMEOUT);
  if (warp == W_MMA) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, a.tmem_cols);
  }
  if (sm->abort || !a.fuse_topk) return;  // block-uniform
  // ---------------- top-k of the sequences this CTA completed, in the now idle shared memory (the
  // thread that completed a sequence fenced after seeing its count; the barrier above orders the
  // other threads after it)
  uint8_t* tbuf = base;
  const size_t tbytes = (size_t)(reinterpret_cast<uint8_t*>(sm) - base);
  const int nfin = min((int)sm->nfin, FIN_MAX);
  for (int f = 0; f < nfin; ++f) {
    const int b = sm->fin[f];
    for (int q = 0; q < a.qps; ++q) {
      const int t = b * a.qps + q;
      const int n = (pre && b - b_first < WSEQ) ? sm->nc_tab[b - b_first][q]
                                                 : visible_entries(a.positions, t, a.max_context, a.ratio);
      const float* srow = a.bufs.scores + (int64_t)t * a.bufs.nc_stride;
      if (!tk::topk_token(srow, a.bufs.hist + (int64_t)t * HIST_BINS, n, a.K, a.topk_idx + (int64_t)t * a.K,
                          a.topk_score ? a.topk_score + (int64_t)t * a.K : nullptr,
                          a.bufs.cand + (int64_t)t * a.bufs.nc_stride, tbuf, tbytes, abort,
                          (a.cskip || a.cmask) ? a.cand + (int64_t)t * a.cM : nullptr, a.cM, a.clg)) {
        if (threadIdx.x == 0) atomicOr(&g_flags_ix, FLAG_TIMEOUT);
        return;
      }
      if (a.cwrite) tk::publish_blocks(srow, n, a.clg, a.cM, a.cand + (int64_t)t * a.cM, tbuf);
    }
  }
  // sequences without a scored tile (no visible entry, or a consumer's list naming none) are completed
  // by nobody: all -1 (the source publishes no block)
  for (int b = blockIdx.x; b < a.B; b += gridDim.x) {
    if (live_tiles(a, b, seq_entries(a, b)) != 0) continue;
    for (int q = 0; q < a.qps; ++q) {
      const int t = b * a.qps + q;
      for (int x = threadIdx.x; x < a.K; x += blockDim.x) {
        a.topk_idx[(int64_t)t * a.K + x] = -1;
        if (a.topk_score) a.topk_score[(int64_t)t * a.K + x] = -INFINITY;
      }
      if (a.cwrite)
        for (int x = threadIdx.x; x < a.cM; x += blockDim.x) a.cand[(int64_t)t * a.cM + x] = -1;
    }
  }
}

}  // namespace ixtc

// The tensor-core kernel multiplies each key tile by the queries of all of a sequence's tokens (N =
// q_per_seq x n_heads columns, 64 or 128).  With more columns it takes every query token as its own
// sequence (N = n_heads; the tokens of a sequence then read its keys once each).
static bool tc_per_token(const dsv4_indexer_topk_params& p) {
  return p.q_per_seq * p.n_heads > 128 && (p.n_heads == 64 || p.n_heads == 128);
}

static bool use_tc_indexer(const dsv4_indexer_topk_params& p) {
  const int N = tc_per_token(p) ? p.n_heads : p.q_per_seq * p.n_heads;
  return (p.k_dtype == DSV4_BF16 || p.k_dtype == DSV4_I8_ROWSCALE || p.k_dtype == DSV4_MXFP4) &&
         p.q_dtype == DSV4_BF16 &&
         (p.head_dim == 64 || p.head_dim == 128) && p.n_heads % 32 == 0 && N >= 64 && N <= 128 && N % 64 == 0 &&
         p.page_size == 64;
}

static cudaError_t launch_indexer_score_tc(const dsv4_indexer_topk_params& p, const TopkBufs& bufs,
                                           cudaStream_t st) {
  using namespace ixtc;
  const int max_nc = p.max_context / p.ratio;
  Args a;
  a.positions = p.positions;
  a.block_table = p.block_table;
  a.weights = p.weights;
  a.bufs = bufs;
  a.num_pages = p.num_pages;
  const bool per_token = tc_per_token(p);
  a.T = p.T;
  a.B = per_token ? p.T : p.B;
  a.qps = per_token ? 1 : p.q_per_seq;
  a.bt_div = per_token ? p.q_per_seq : 1;
  a.Ih = p.n_heads;
  a.d = p.head_dim;
  a.ratio = p.ratio;
  a.max_pages = p.max_pages_per_seq;
  a.tiles_max = (max_nc + TILE - 1) / TILE;
  a.max_context = p.max_context;
  a.K = p.topk;
  a.fuse_topk = max_nc <= TOPK_FUSED_MAX;
  a.topk_idx = p.topk_idx;
  a.topk_score = p.topk_score;
  a.N = a.qps * p.n_heads;
  a.kblk = p.head_dim / 64;
  a.nacc = 4 * a.N <= 512 ? 4 : 2;  // TMEM accumulators (512 columns available)
  a.kf = p.k_dtype == DSV4_I8_ROWSCALE ? KF_I8 : (p.k_dtype == DSV4_MXFP4 ? KF_MX : KF_BF16);
  a.rec = (int)row_bytes(p.k_dtype, p.head_dim);
  a.nraw = 0;
  a.k_raw = reinterpret_cast<const uint8_t*>(p.k_cache);
  a.tmem_cols = a.nacc * a.N <= 64 ? 64 : (a.nacc * a.N <= 128 ? 128 : (a.nacc * a.N <= 256 ? 256 : 512));
  const CandArgs ca = cand_args(p);
  a.cand = ca.blocks;
  a.cM = ca.M;
  a.clg = ca.lg;
  a.csh = ca.blocks ? ca.lg - 7 : 0;
  a.cskip = ca.blocks && !ca.write && a.qps == 1;
  a.cmask = ca.blocks && !ca.write && a.qps > 1;
  a.cwrite = ca.blocks && ca.write;
  const size_t budget = 227 * 1024;
  auto fixed_for = [&](int nqs, int nraw) {
    return 1024 + (size_t)nqs * a.kblk * a.N * 128 + (size_t)nraw * 2 * 64 * (size_t)a.rec +
           (a.kf == KF_I8 ? (size_t)SCALE_RING * TILE * 4 : 0) +
           (2 * 256 + WSEQ * 128) * 4 + 2 * (size_t)a.qps * HIST_BINS * 4 + sizeof(Smem);
  };
  // the first (query slots, raw pages in flight) that leaves at least two bf16 stages: a second query
  // slot lets the next sequence's queries load early; MXFP4 records (a quarter of a bf16 tile) need a
  // deep raw ring to keep enough bytes in flight
  static const int kOrder[3][7][2] = {{{2, 0}, {1, 0}},
                                      {{2, 2}, {1, 2}},
                                      {{2, 8}, {2, 6}, {1, 8}, {1, 6}, {2, 4}, {1, 4}, {1, 2}}};
  const int nopt = a.kf == KF_MX ? 7 : 2;
  size_t fixed = 0;
  int stages = 0;
  for (int o = 0; o < nopt; ++o) {
    a.nqs = kOrder[a.kf][o][0];
    a.nraw = kOrder[a.kf][o][1];
    fixed = fixed_for(a.nqs, a.nraw);
    stages = fixed < budget ? (int)((budget - fixed) / ((size_t)a.kblk * KB_BYTES)) : 0;
    if (stages >= 2) break;
  }
  a.stages = stages > MAX_STAGES ? MAX_STAGES : stages;
  if (a.stages < 2) return cudaErrorInvalidConfiguration;
  const size_t smem = fixed + (size_t)a.stages * a.kblk * KB_BYTES;
  CUtensorMap kmap, qmap;
  cudaError_t e = make_tmap_2d_bf16(&qmap, p.q, (uint64_t)p.head_dim, (uint64_t)p.T * p.n_heads, 64, (uint32_t)a.N);
  if (e != cudaSuccess) return e;
  if (a.kf != KF_BF16) {
    kmap = qmap;  // raw records are bulk-copied: the key map is not used
  } else {
    e = make_tmap_2d_bf16(&kmap, p.k_cache, (uint64_t)p.head_dim, (uint64_t)p.num_pages * 64, 64, 64);
    if (e != cudaSuccess) return e;
  }
  e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(indexer_score_tc<KF_BF16>), (int)budget);
  if (e == cudaSuccess) e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(indexer_score_tc<KF_I8>), (int)budget);
  if (e == cudaSuccess) e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(indexer_score_tc<KF_MX>), (int)budget);
  if (e != cudaSuccess) return e;
  const int total = a.B * a.tiles_max;
  int grid = num_sms();
  if (grid > total) grid = total;
  if (grid < (total + FIN_MAX - 1) / FIN_MAX) grid = (total + FIN_MAX - 1) / FIN_MAX;  // <= FIN_MAX items per CTA
  if (grid <= 0) return cudaSuccess;
  // the expanding warps exist only for raw records
  if (a.kf == KF_I8)
    return launch_pdl(indexer_score_tc<KF_I8>, dim3(grid), dim3(THREADS), smem, st, /*pdl=*/true, kmap, qmap, a);
  if (a.kf == KF_MX)
    return launch_pdl(indexer_score_tc<KF_MX>, dim3(grid), dim3(THREADS), smem, st, /*pdl=*/true, kmap, qmap, a);
  return launch_pdl(indexer_score_tc<KF_BF16>, dim3(grid), dim3(THREADS_BF16), smem, st, /*pdl=*/true, kmap, qmap,
                    a);
}

// ------------------------------------------------------------------------------------------------
// Top-k after the CUDA-core score kernel: one CTA per token.
// ------------------------------------------------------------------------------------------------
constexpr int TK_THREADS = 320;
static_assert(TK_THREADS / 32 >= tk::SCAN_WARPS_MIN, "the top-k scan covers a chunk with this many warps");
constexpr size_t TK_SMEM = 220 * 1024;

__global__ void __launch_bounds__(TK_THREADS) topk_kernel(dsv4_indexer_topk_params p, TopkBufs bufs) {
  extern __shared__ __align__(128) uint8_t tsm[];
  __shared__ int abort_s;
  pdl_launch_dependents();
  pdl_wait();
  if (threadIdx.x == 0) abort_s = 0;
  __syncthreads();
  const int t = blockIdx.x;
  const int n = visible_entries(p, t);
  const bool has_cand = p.cand_block_size > 0;
  const int lg = has_cand ? __ffs(p.cand_block_size) - 1 : 0;
  int32_t* crow = has_cand ? p.cand_blocks + (int64_t)t * p.cand_topk : nullptr;
  const float* srow = bufs.scores + (int64_t)t * bufs.nc_stride;
  if (!tk::topk_token(srow, bufs.hist + (int64_t)t * HIST_BINS, n, p.topk, p.topk_idx + (int64_t)t * p.topk,
                      p.topk_score ? p.topk_score + (int64_t)t * p.topk : nullptr,
                      bufs.cand + (int64_t)t * bufs.nc_stride, tsm, TK_SMEM, &abort_s,
                      has_cand && !p.cand_write ? crow : nullptr, p.cand_topk, lg)) {
    if (threadIdx.x == 0) atomicOr(&g_flags_ix, FLAG_TIMEOUT);
    return;
  }
  if (has_cand && p.cand_write) {
    __syncthreads();
    tk::publish_blocks(srow, n, lg, p.cand_topk, crow, tsm);
  }
}

// ------------------------------------------------------------------------------------------------
// Top-k of long rows, spread over CTAs: CTA (slice, token) takes SLICE scores of the token.  Each
// finds the threshold bin from the complete histogram, writes its words of the token's selection
// bitmap and appends its candidates to the token's list; the CTA that finishes the token's last
// slice chooses among the candidates and writes the selection (no CTA waits for another).
// ------------------------------------------------------------------------------------------------
constexpr int SLICE_CHUNKS = 2;  // 8192-score slices: more CTAs per long row (measured faster than 16384)
constexpr int SLICE = SLICE_CHUNKS * tk::CHUNK;  // 8192 scores

__global__ void __launch_bounds__(TK_THREADS) topk_slice_kernel(dsv4_indexer_topk_params p, TopkBufs bufs) {
  extern __shared__ __align__(128) uint8_t tsm[];
  __shared__ int abort_s;
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.y, sl = blockIdx.x;
  const int n = visible_entries(p, t), K = p.topk;
  const int nsl = n <= K ? 1 : (n + SLICE - 1) / SLICE;  // a short row: slice 0 writes every entry
  if (sl >= nsl) return;  // block-uniform
  if (threadIdx.x == 0) abort_s = 0;
  __syncthreads();
  const bool has_cand = p.cand_block_size > 0;
  const int lg = has_cand ? __ffs(p.cand_block_size) - 1 : 0;
  int32_t* crow = has_cand ? p.cand_blocks + (int64_t)t * p.cand_topk : nullptr;
  const int r = tk::topk_part(bufs.scores + (int64_t)t * bufs.nc_stride, bufs.hist + (int64_t)t * HIST_BINS, n, K,
                              sl * SLICE, (sl + 1) * SLICE, 1u, (uint32_t)nsl, bufs.bits + (int64_t)t * (bufs.nc_stride / 32),
                              bufs.cand + (int64_t)t * bufs.nc_stride, &bufs.tcnt[2 * t], p.topk_idx + (int64_t)t * K,
                              p.topk_score ? p.topk_score + (int64_t)t * K : nullptr, tsm, TK_SMEM, &abort_s,
                              has_cand && !p.cand_write ? crow : nullptr, p.cand_topk, lg,
                              has_cand && p.cand_write ? crow : nullptr, p.cand_topk);
  if (r < 0 && threadIdx.x == 0) atomicOr(&g_flags_ix, FLAG_TIMEOUT);
}

cudaError_t launch_indexer_topk(const dsv4_indexer_topk_params& p, cudaStream_t st) {
  if (p.T == 0) return cudaSuccess;
  IxLayout L = ix_layout(p);
  char* ws = reinterpret_cast<char*>(p.workspace);
  TopkBufs bufs;  // every call clears the histograms and counters it used before it completes
  bufs.scores = reinterpret_cast<float*>(ws + L.scores_off);
  bufs.hist = reinterpret_cast<uint32_t*>(ws + L.hist_off);
  bufs.seq_done = reinterpret_cast<uint32_t*>(ws + L.done_off);
  bufs.tcnt = reinterpret_cast<uint32_t*>(ws + L.tcnt_off);
  bufs.cand = reinterpret_cast<uint64_t*>(ws + L.cand_off);
  bufs.bits = reinterpret_cast<uint32_t*>(ws + L.bits_off);
  bufs.nc_stride = (int)L.nc_stride;
  cudaError_t e = cudaSuccess;
  if (!p.workspace_zeroed) {  // histograms and counters start at zero (every completed call leaves them so)
    e = cudaMemsetAsync(ws + L.hist_off, 0, L.tcnt_off + (size_t)p.T * 2 * sizeof(uint32_t) - L.hist_off, st);
    if (e != cudaSuccess) return e;
  }
  const int max_nc = p.max_context / p.ratio;
  const bool fused = max_nc <= TOPK_FUSED_MAX;
  if (max_nc > 0 && use_tc_indexer(p)) {
    e = launch_indexer_score_tc(p, bufs, st);  // includes the top-k when the rows are short
    if (e != cudaSuccess || fused) return e;
  } else if (max_nc > 0) {
    const int tiles = (max_nc + IX_TILE - 1) / IX_TILE;
    const size_t smem = sizeof(float) * ((size_t)p.q_per_seq * p.n_heads * p.head_dim +
                                         (size_t)p.q_per_seq * p.n_heads + (size_t)(p.head_dim + 1) * (IX_TILE + 1));
    e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(indexer_score_simt), (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(indexer_score_simt, dim3(tiles, p.B), dim3(IX_TILE), smem, st, /*pdl=*/false, p, bufs);
    if (e != cudaSuccess) return e;
  }
  e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(topk_kernel), (int)TK_SMEM);
  if (e != cudaSuccess) return e;
  e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(topk_slice_kernel), (int)TK_SMEM);
  if (e != cudaSuccess) return e;
  if (fused) return launch_pdl(topk_kernel, dim3(p.T), dim3(TK_THREADS), TK_SMEM, st, /*pdl=*/false, p, bufs);
  const int slices = (max_nc + SLICE - 1) / SLICE;
  return launch_pdl(topk_slice_kernel, dim3(slices, p.T), dim3(TK_THREADS), TK_SMEM, st, /*pdl=*/false, p, bufs);
}

cudaError_t read_flags_indexer(uint32_t* f) {
  unsigned int v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_flags_ix, sizeof(v));
  if (e != cudaSuccess) return e;
  *f |= v;
  return cudaMemcpyToSymbol(g_flags_ix, &z, sizeof(z));
}

}  // namespace dsv4
