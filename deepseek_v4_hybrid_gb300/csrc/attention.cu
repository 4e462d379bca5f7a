// Shared-KV sparse MLA decode attention: one softmax per query head over the sliding-window rows,
// the selected (CSA) or all (HCA) compressed rows and an optional sink logit, split over CTAs and
// merged with log-sum-exp weights.
//
// "DeepSeek V4 Attention: Code Reading Map", §Phase 3: forward_mqa() (items 1-6) and
// §Layer-Type Summary; "vllm.models.deepseek_v41.attention", DeepseekV4Attention.__init__
// (attn_sink initialised to -inf = no sink effect; scale is a parameter).
//
// Row list of a query at position p: rows 0..n_swa-1 are the window positions
// p - n_swa + 1 .. p (n_swa = min(window, p + 1)), then the compressed rows: topk_idx[t][i]
// (an index outside [0, n_c(p)) is masked) or j = 0 .. n_c(p) - 1 when no list is given.
#include <cooperative_groups.h>
#include <cstddef>

#include "dsv4_common.cuh"
#include "dsv4_launch.h"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace cg = cooperative_groups;

namespace dsv4 {

static __device__ unsigned int g_flags_at = 0;

constexpr int AT_CH = 64;       // rows per split chunk (SIMT kernel)
constexpr int AT_HG = 16;       // heads per CTA (SIMT kernel)
constexpr int AT_THREADS = 256;
constexpr int MERGE_THREADS = 256;

struct AtLayout {
  int n_chunks, chunk_rows;
  size_t o_off, ml_off, total;
};

static int max_rows(const dsv4_sparse_mla_decode_params& p) {
  int n_swa = p.window < p.max_context ? p.window : p.max_context;
  // the tensor-core kernel reads whole window pages: at most ceil((window - 1) / 64) + 1 of them
  n_swa = ((n_swa + 62) / 64 + 1) * 64;
  int n_cmp = 0;
  if (p.ratio > 0) n_cmp = p.topk_idx ? p.topk : p.max_context / p.ratio;
  return n_swa + (n_cmp + 63) / 64 * 64;
}

static bool use_tc_attention(const dsv4_sparse_mla_decode_params& p);

// Chunks per (token, head group) of the tensor-core kernel: about one wave of CTAs over the SMs.
// Chunk c takes the 64-row halves c, c + n_chunks, c + 2 n_chunks, ... of the token's row list, so
// window pages and gathered rows spread evenly over the chunks.
static int tc_chunks(const dsv4_sparse_mla_decode_params& p) {
  const int units = p.T * (p.H / 64);
  int n = units > 0 ? num_sms() / units : 1;
  if (n < 1) n = 1;
  const int halves = max_rows(p) / 64;
  return n < halves ? n : (halves > 0 ? halves : 1);
}

static AtLayout at_layout(const dsv4_sparse_mla_decode_params& p) {
  AtLayout L;
  if (use_tc_attention(p)) {
    L.n_chunks = tc_chunks(p);
    L.chunk_rows = (max_rows(p) / 64 + L.n_chunks - 1) / L.n_chunks * 64;  // rows of the largest chunk
  } else {
    L.chunk_rows = AT_CH;
    L.n_chunks = (max_rows(p) + L.chunk_rows - 1) / L.chunk_rows;
  }
  if (L.n_chunks < 1) L.n_chunks = 1;
  const size_t parts = (size_t)p.T * L.n_chunks * p.H;
  L.o_off = 0;
  L.ml_off = align_up(parts * DV * sizeof(float), 256);
  L.total = align_up(L.ml_off + parts * sizeof(float2), 256);
  return L;
}

size_t sparse_mla_workspace(const dsv4_sparse_mla_decode_params& p) { return at_layout(p).total; }

// Address of row r of token t's row list, or nullptr when the row is masked.
__device__ __forceinline__ const uint8_t* attn_row(const dsv4_sparse_mla_decode_params& p, int t, int b, int pos,
                                                   int n_swa, int nc, int r, int64_t rb) {
  int64_t slot;
  const uint8_t* base;
  if (r < n_swa) {
    const int q = pos - n_swa + 1 + r;
    const int lp = q / p.page_size;
    const int page = lp < p.swa_max_pages ? p.swa_block_table[(int64_t)b * p.swa_max_pages + lp] : -1;
    if (page < 0 || page >= p.swa_num_pages) {
      atomicOr(&g_flags_at, FLAG_PAGE);
      return nullptr;
    }
    slot = (int64_t)page * p.page_size + q % p.page_size;
    base = reinterpret_cast<const uint8_t*>(p.swa_cache);
  } else {
    const int i = r - n_swa;
    int j = i;
    if (p.topk_idx != nullptr) {
      j = p.topk_idx[(int64_t)t * p.topk + i];
      if (j < 0) return nullptr;
      if (j >= nc) {
        atomicOr(&g_flags_at, FLAG_TOPK);
        return nullptr;
      }
    }
    const int lp = j / p.page_size;
    const int page = lp < p.main_max_pages ? p.main_block_table[(int64_t)b * p.main_max_pages + lp] : -1;
    if (page < 0 || page >= p.main_num_pages) {
      atomicOr(&g_flags_at, FLAG_PAGE);
      return nullptr;
    }
    slot = (int64_t)page * p.page_size + j % p.page_size;
    base = reinterpret_cast<const uint8_t*>(p.main_cache);
  }
  return base + slot * rb;
}

__device__ __forceinline__ void token_rows(const dsv4_sparse_mla_decode_params& p, int& pos, int& n_swa, int& nc,
                                           int& n_cmp) {
  if (pos < 0 || pos >= p.max_context) {  // outside what the grid was sized for: no rows
    atomicOr(&g_flags_at, FLAG_PAGE);
    pos = 0;
    n_swa = nc = n_cmp = 0;
    return;
  }
  n_swa = pos + 1 < p.window ? pos + 1 : p.window;
  nc = p.ratio > 0 ? (pos + 1) / p.ratio : 0;
  n_cmp = p.ratio == 0 ? 0 : (p.topk_idx ? p.topk : nc);
}

// ------------------------------------------------------------------------------------------------
// SIMT partial kernel: CTA (chunk, token, head group); fp32 math on decoded rows in shared memory.
// ------------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(AT_THREADS) mla_partial_simt(dsv4_sparse_mla_decode_params p, float* o_part,
                                                               float2* ml_part, int n_chunks) {
  extern __shared__ float smem[];
  pdl_launch_dependents();
  pdl_wait();
  const int chunk = blockIdx.x, t = blockIdx.y, h0 = blockIdx.z * AT_HG, tid = threadIdx.x;
  const int b = t / p.q_per_seq;
  int pos = p.positions[t];
  int n_swa, nc, n_cmp;
  token_rows(p, pos, n_swa, nc, n_cmp);
  const int r0 = chunk * AT_CH;
  const int nrows = min(AT_CH, n_swa + n_cmp - r0);
  const int nh = min(AT_HG, p.H - h0);
  const int64_t part = ((int64_t)t * n_chunks + chunk) * p.H;

  if (nrows <= 0) {
    for (int h = tid; h < nh; h += AT_THREADS) ml_part[part + h0 + h] = make_float2(-INFINITY, 0.f);
    return;
  }
  const int LDK = D + 1;
  float* q_s = smem;                   // [AT_HG][D]
  float* kv_s = q_s + AT_HG * D;       // [AT_CH][D + 1]
  float* p_s = kv_s + AT_CH * LDK;     // [AT_HG][AT_CH]
  __shared__ int valid_s[AT_CH];

  for (int x = tid; x < AT_HG * (D / 2); x += AT_THREADS) {
    const int h = x / (D / 2), i = x % (D / 2);
    float2 v = make_float2(0.f, 0.f);
    if (h < nh) {
      const int64_t qrow = ((int64_t)t * p.H + h0 + h) * D;
      v = (p.q_dtype == DSV4_F32) ? reinterpret_cast<const float2*>(p.q)[qrow / 2 + i]
                                  : decode_pair(DSV4_BF16, reinterpret_cast<const uint8_t*>(p.q) + qrow * 2, i);
    }
    q_s[h * D + 2 * i] = v.x;
    q_s[h * D + 2 * i + 1] = v.y;
  }
  const int64_t rb = row_bytes(p.cache_dtype, D);
  __shared__ const uint8_t* rows_s[AT_CH];
  if (tid < AT_CH) rows_s[tid] = tid < nrows ? attn_row(p, t, b, pos, n_swa, nc, r0 + tid, rb) : nullptr;
  __syncthreads();
  for (int r = 0; r < AT_CH; ++r) {
    const uint8_t* row = rows_s[r];
    if (tid == 0) valid_s[r] = row != nullptr;
    for (int i = tid; i < D / 2; i += AT_THREADS) {
      float2 v = row ? decode_pair(p.cache_dtype, row, i) : make_float2(0.f, 0.f);
      kv_s[r * LDK + 2 * i] = v.x;
      kv_s[r * LDK + 2 * i + 1] = v.y;
    }
  }
  __syncthreads();

  // logits: thread -> (head tid/16, rows tid%16 + 16k)
  {
    const int h = tid / 16, rr = tid % 16;
    for (int k = 0; k < AT_CH / 16; ++k) {
      const int r = rr + 16 * k;
      float acc = 0.f;
      const float* qh = q_s + h * D;
      const float* kr = kv_s + r * LDK;
      for (int e = 0; e < D; ++e) acc = fmaf(qh[e], kr[e], acc);
      p_s[h * AT_CH + r] = (r < nrows && valid_s[r]) ? acc * p.softmax_scale : -INFINITY;
    }
  }
  __syncthreads();
  // softmax per head: warp w handles heads 2w, 2w+1
  {
    const int w = tid >> 5, lane = tid & 31;
    for (int hh = 0; hh < 2; ++hh) {
      const int h = 2 * w + hh;
      float* ph = p_s + h * AT_CH;
      const float a = ph[lane], c = ph[lane + 32];
      const float m = warp_max(fmaxf(a, c));
      const float ea = (m == -INFINITY) ? 0.f : expf(a - m);
      const float ec = (m == -INFINITY) ? 0.f : expf(c - m);
      const float l = warp_sum(ea + ec);
      __syncwarp();
      ph[lane] = ea;
      ph[lane + 32] = ec;
      if (lane == 0 && h < nh) ml_part[part + h0 + h] = make_float2(m, l);
    }
  }
  __syncthreads();
  // O[h][c], thread owns value columns 2*tid, 2*tid+1
  {
    float acc[AT_HG][2];
#pragma unroll
    for (int h = 0; h < AT_HG; ++h) acc[h][0] = acc[h][1] = 0.f;
    for (int r = 0; r < nrows; ++r) {
      const float v0 = kv_s[r * LDK + 2 * tid], v1 = kv_s[r * LDK + 2 * tid + 1];
#pragma unroll
      for (int h = 0; h < AT_HG; ++h) {
        const float pr = p_s[h * AT_CH + r];
        acc[h][0] = fmaf(pr, v0, acc[h][0]);
        acc[h][1] = fmaf(pr, v1, acc[h][1]);
      }
    }
#pragma unroll
    for (int h = 0; h < AT_HG; ++h)
      if (h < nh)
        reinterpret_cast<float2*>(o_part + (part + h0 + h) * DV)[tid] = make_float2(acc[h][0], acc[h][1]);
  }
}


// ------------------------------------------------------------------------------------------------
// Tensor-core partial kernel (bf16 caches and queries).  CTA = (chunk of rows, token, 64-head
// group).  Both products are computed transposed, so that the attended rows, not the heads, fill
// the 128 lanes of the MMA:
//   S^T[r, h]  = K[r, :] . Q[h, :]        M = 128 rows, N = 64 heads, K = 576 (9 K-blocks of 64)
//   O^T[v, h] += V^T[v, r] P^T[r, h]      M = 128 value dims (4 blocks for 512), N = 64 heads,
//                                         K = the tile's 128 rows
// O^T takes 4 x 64 TMEM columns and S^T 64 more, so one CTA keeps all 512 value dims and computes
// each QK^T once.
//
// Shared memory holds Q (72 KB) and one 128-row tile (9 K-block slots of 16 KB = 144 KB) in the
// 128-byte swizzled layout TMA writes: K-major for QK^T and, read the other way, MN-major for the
// V^T operand of PV.  P^T (bf16, 128 rows x 64 heads) is written by the softmax warps over slot 8
// (the rope dims, which PV does not read) once QK^T is done.  Slots are refilled per group as soon
// as the PV MMAs that read them retire: {0,1} after value block 0, ..., {6,7} and 8 after block 3.
//
// Row list of a token: the window pages (whole 64-row pages of the SWA cache covering positions
// p - n_swa + 1 .. p, rows outside that range masked), then the compressed rows in 64-row halves
// (top-k indices, or dense pages of the main cache).  Warps 8, 10 and 11 load (the TMA issue rate
// is per issuing warp: K-block kb of every tile is loaded by the kb mod 3-th of them): a window
// page or a dense page as TMA boxes, top-k rows with TMA gather4 (4 rows x one K-block each; an
// invalid index loads a row past the end of the tensor, i.e. zeros).  Lane 0 of warp 9 issues the
// MMAs.  Warps 0-7 run
// the online softmax in the log2 domain with a lazy rescale (O^T is rescaled only when a head's
// running max grows by more than 2^8): warp w owns tile rows 32 (w & 3) .. + 31 (its TMEM lane
// quarter) and heads 32 (w >> 2) .. + 31; a tile's per-head maxima are reduced across lanes by a
// shuffle transpose-reduce and across the four row quarters in shared memory.  A masked row of a
// loaded half gets zero V (it may hold anything, and 0 x NaN would poison O); PV skips halves that
// were not loaded.  At the end, when a token's chunks form a cluster (up to 8), the same warps push
// their O^T scaled by the chunk's log-sum-exp weight into the shared memory of the CTA that owns
// each value-dim slice, and every owner sums its slots and writes its slice of the output; with more
// chunks they turn O^T into [head][value] rows in the idle tile buffer and store the unnormalised O
// and the chunk's (max, sum) per head for mla_merge.
//
// fp8_ds_mla caches (656-byte records: 512 e4m3 codes, 64 bf16 rope dims, 8 UE8M0 block exponents)
// run the same kernel with the tile converted in shared memory: the codes of K-block kb < 8 (64 B
// a row) are loaded by TMA, untiled, into the upper 8 KB of slot kb, and softmax warp kb (idle
// between handing over P^T and the next tile's S^T) expands them in place into bf16
// code x 2^(e - 127) in the swizzled K-major layout (exact: an e4m3 value times a power of two has
// at most 4 significant bits).  The rope dims are bf16 already and go by TMA straight into slot 8.
// The tile's block exponents (8 bytes a row) come by cp.async with the first group's loads.
// Everything after the expansion is the bf16 kernel's.
// ------------------------------------------------------------------------------------------------
namespace attc {
constexpr int TILE = 128;                  // rows per tile
constexpr int HALF = 64;                   // rows per load unit (one page)
constexpr int HG = 64;                     // heads per CTA
constexpr int NKB = 9;                     // 64-dim K-blocks of a 576-dim row
constexpr int SLOT_BYTES = TILE * 128;     // one K-block of a tile: 16 KB
constexpr int HALF_BYTES = HALF * 128;     // 8 KB
constexpr int Q_BYTES = NKB * HG * 128;    // 72 KB
constexpr int KV_BYTES = NKB * SLOT_BYTES;  // 144 KB
constexpr int NGROUPS = 5;                 // slot groups {0,1} {2,3} {4,5} {6,7} {8}
constexpr int THREADS = 384;               // warps 0-7 softmax + epilogue, 8, 10, 11 loads, 9 MMA
constexpr int W_LOAD = 8, W_MMA = 9;
constexpr int NPROD = 3;                   // loading warps: K-block kb of every tile is loaded by warp kb % 3
constexpr uint32_t COL_O = 0, COL_S = 256, TMEM_COLS = 512;
constexpr float RESCALE_LOG2 = 8.0f;
constexpr uint32_t FLAG_TIMEOUT = 4u;
constexpr int K_NONE = 0, K_BOX_SWA = 1, K_BOX_MAIN = 2, K_GATHER = 3;
constexpr int MAX_MERGE_CLUSTER = 8;  // up to this many chunks per token merge inside a (portable) cluster
constexpr int RAW_OFF = SLOT_BYTES / 2;  // fp8: the codes of K-block kb (128 rows x 64 B) staged in slot kb from here
constexpr int RAW_HALF = HALF * 64;      // fp8: codes of one K-block of a 64-row half (4 KB)

struct Args {
  dsv4_sparse_mla_decode_params p;
  float* o_part;
  float2* ml_part;
  int n_chunks;             // chunk c takes halves c, c + n_chunks, ... of a token's row list
  int swa_rows, main_rows;  // rows of the two caches (a gather from this row loads zeros)
  float c_log2;             // softmax_scale * log2(e)
  int cluster_merge;        // the chunks of a (token, head group) form one cluster and merge in it
};

struct Smem {
  uint64_t full[NGROUPS], vfree[4], sfull, pfull, pvdone, qfull, odone, xbar[2][2], ebar;
  uint64_t rawb[NPROD][4];  // fp8: codes of loader p's K-blocks in group g have landed
  uint64_t sbar;            // fp8: the tile's block exponents and row masks are in
  uint2 scl[TILE];          // fp8: UE8M0 bytes of the tile's rows (byte kb: K-block kb)
  uint32_t mask[2][4];  // [tile parity][row / 32]: valid rows
  uint32_t loaded[2];   // [tile parity]: bit u = half u was loaded
  float red[2][2][4][32];  // [tile parity][head half][row quarter][lane]: per-warp maxima
  float lred[2][4][32];
  alignas(16) float mrow[8][64];  // per softmax warp: running max and rescale factor of its 32 heads (read as float4)
  float2 cml[HG];                 // the chunk's (max in log2 units, sum) per head, read by the cluster
  uint32_t tmem_base;
  int abort;
};
static_assert(1024 + Q_BYTES + KV_BYTES + sizeof(Smem) <= 232448, "shared memory of one CTA");
static_assert(offsetof(Smem, mrow) % 16 == 0, "mrow is read with 16-byte loads");

struct TokenRows {
  int pos, lo, first_wp, n_wp, nc, n_cmp, n_halves;
};

__device__ __forceinline__ TokenRows token_plan(const dsv4_sparse_mla_decode_params& p, int t) {
  TokenRows r;
  int pos = p.positions[t], n_swa, nc, n_cmp;
  token_rows(p, pos, n_swa, nc, n_cmp);
  r.pos = pos;
  r.nc = nc;
  r.n_cmp = n_cmp;
  if (n_swa > 0) {
    r.lo = pos - n_swa + 1;
    r.first_wp = r.lo / p.page_size;
    r.n_wp = pos / p.page_size - r.first_wp + 1;
  } else {
    r.lo = 0;
    r.first_wp = 0;
    r.n_wp = 0;
  }
  r.n_halves = r.n_wp + (n_cmp + HALF - 1) / HALF;
  return r;
}

struct HalfPlan {
  int kind, ybox, y0, y1;
  bool v0, v1;  // rows lane and lane + 32 of the half are valid
};

// How half `hh` of the token's row list is loaded, and which of its rows are valid (warp-wide).
__device__ __forceinline__ HalfPlan plan_half(const Args& a, int t, int b, const TokenRows& tr, int hh, int lane) {
  const dsv4_sparse_mla_decode_params& p = a.p;
  HalfPlan h;
  h.kind = K_NONE;
  h.ybox = 0;
  h.y0 = h.y1 = a.main_rows;
  h.v0 = h.v1 = false;
  if (hh >= tr.n_halves) return h;
  if (hh < tr.n_wp) {
    const int lp = tr.first_wp + hh;
    const int page = lp < p.swa_max_pages ? p.swa_block_table[(int64_t)b * p.swa_max_pages + lp] : -1;
    if (page < 0 || page >= p.swa_num_pages) {
      if (lane == 0) atomicOr(&g_flags_at, FLAG_PAGE);
      return h;
    }
    const int q0 = lp * p.page_size + lane, q1 = q0 + 32;
    h.v0 = q0 >= tr.lo && q0 <= tr.pos;
    h.v1 = q1 >= tr.lo && q1 <= tr.pos;
    h.kind = K_BOX_SWA;
    h.ybox = page * p.page_size;
    return h;
  }
  const int j0 = (hh - tr.n_wp) * HALF;
  if (p.topk_idx == nullptr) {  // dense: the half is logical page j0 / 64 of the main cache
    const int lp = j0 / p.page_size;
    const int page = lp < p.main_max_pages ? p.main_block_table[(int64_t)b * p.main_max_pages + lp] : -1;
    if (page < 0 || page >= p.main_num_pages) {
      if (lane == 0) atomicOr(&g_flags_at, FLAG_PAGE);
      return h;
    }
    h.v0 = j0 + lane < tr.nc;
    h.v1 = j0 + lane + 32 < tr.nc;
    h.kind = K_BOX_MAIN;
    h.ybox = page * p.page_size;
    return h;
  }
  int y[2];
  bool v[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int i = j0 + lane + 32 * u;
    v[u] = false;
    y[u] = a.main_rows;
    if (i < tr.n_cmp) {
      const int j = p.topk_idx[(int64_t)t * p.topk + i];
      if (j >= tr.nc) atomicOr(&g_flags_at, FLAG_TOPK);
      if (j >= 0 && j < tr.nc) {
        const int lp = j / p.page_size;
        const int page = lp < p.main_max_pages ? p.main_block_table[(int64_t)b * p.main_max_pages + lp] : -1;
        if (page < 0 || page >= p.main_num_pages) {
          atomicOr(&g_flags_at, FLAG_PAGE);
        } else {
          v[u] = true;
          y[u] = page * p.page_size + j % p.page_size;
        }
      }
    }
  }
  h.y0 = y[0];
  h.y1 = y[1];
  h.v0 = v[0];
  h.v1 = v[1];
  h.kind = __any_sync(0xffffffffu, v[0] || v[1]) ? K_GATHER : K_NONE;
  return h;
}

// Max (or sum) over the 32 lanes of 32 per-lane values, transposed: lane l returns the result for
// value l.  Five butterfly steps, each halving the values a lane keeps.
template <bool kMax>
__device__ __forceinline__ float transpose_reduce32(const float (&x)[32], int lane) {
  float v[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const bool up = lane & 16;
    const float send = up ? x[k] : x[k + 16];
    const float keep = up ? x[k + 16] : x[k];
    const float o = __shfl_xor_sync(0xffffffffu, send, 16);
    v[k] = kMax ? fmaxf(keep, o) : keep + o;
  }
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1) {  // 16 -> 8 -> 4 -> 2 -> 1 values, lane bits 3, 2, 1, 0
#pragma unroll
    for (int k = 0; k < w; ++k) {
      const bool up = lane & w;
      const float send = up ? v[k] : v[k + w];
      const float keep = up ? v[k + w] : v[k];
      const float o = __shfl_xor_sync(0xffffffffu, send, w);
      v[k] = kMax ? fmaxf(keep, o) : keep + o;
    }
  }
  return v[0];
}

// Codes b0..b3 of w (b0 the lowest dim) -> bf16 pairs [b0 b1] and [b2 b3] of code x s1 x s2 x 2^-120.
// With a code in the top byte of a 16-bit lane, its sign and its 7 exponent and mantissa bits masked
// into place give the bf16 code x 2^-120 exactly (the 4 exponent bits become the low bits of the bf16
// exponent and the 3 mantissa bits the top of its mantissa; e4m3 subnormals become bf16 subnormals).
// Multiplying by powers of two keeps every value exact while the product stays inside bf16's range,
// which holds for block exponents e in 3 .. 246.  Integer and bf16x2 arithmetic only (measured as
// fast as the e4m3 -> f16 -> fp32 -> bf16 conversion instructions, with no scaled fp32 step).
template <bool TWO>
__device__ __forceinline__ uint2 e4m3x4_to_bf16(uint32_t w, __nv_bfloat162 s1, __nv_bfloat162 s2) {
  uint32_t m01 = __byte_perm(w, 0u, 0x1404u), m23 = __byte_perm(w, 0u, 0x3424u);  // b << 8 in each half
  m01 = ((m01 >> 4) & 0x07F007F0u) | (m01 & 0x80008000u);
  m23 = ((m23 >> 4) & 0x07F007F0u) | (m23 & 0x80008000u);
  __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&m01), b = *reinterpret_cast<__nv_bfloat162*>(&m23);
  if (TWO) {
    a = __hmul2(a, s1);
    b = __hmul2(b, s1);
  }
  a = __hmul2(a, s2);
  b = __hmul2(b, s2);
  return make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
}

// One row of a K-block: v[j] holds the row's codes 16 jr .. 16 jr + 15 (jr = (j + g) & 3), written as
// the bf16 chunks 2 jr and 2 jr + 1 of the swizzled row (r7 = row & 7), the one of index h first.
template <bool TWO>
__device__ __forceinline__ void expand_row16(uint8_t* row, const uint4 (&v)[4], int g, int h, int r7,
                                             __nv_bfloat162 s1, __nv_bfloat162 s2) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int jr = (j + g) & 3;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int half = e ^ h;  // dims 16 jr + 8 half .. + 7: chunk 2 jr + half
      const uint2 o0 = e4m3x4_to_bf16<TWO>(half ? v[j].z : v[j].x, s1, s2);
      const uint2 o1 = e4m3x4_to_bf16<TWO>(half ? v[j].w : v[j].y, s1, s2);
      *reinterpret_cast<uint4*>(row + (((2 * jr + half) ^ r7) << 4)) = make_uint4(o0.x, o0.y, o1.x, o1.y);
    }
  }
}

// fp8: expands K-block kb of the tile's loaded halves (bit u of `ld` = half u), staged as
// [128 rows][64 codes] from RAW_OFF of the slot, into bf16 in the slot's K-major 128-byte-swizzled
// layout, with the rows' UE8M0 bytes in scl.  Lane L owns rows L, 32 + L, 64 + L, 96 + L.  The bf16
// rows 0-63 lie below the staged codes, rows 64-95 over the staged codes of half 0 and rows 96-127
// over those of half 1: so half 0 goes first, then row 64 + L while the codes of row 96 + L are held
// in registers, then row 96 + L.  Reads and writes move 16 bytes; the order in which lane L takes its
// row's four 16-code vectors (offset g) and each vector's two output chunks (first h) depends on
// L & 7 and makes every quarter-warp's reads and writes hit 8 distinct bank groups.  One loop body
// serves the four rows, so the code the warp streams through stays small.
__device__ __forceinline__ void expand_fp8_kblock(uint8_t* slot, uint32_t ld, const uint2* scl, int kb, int lane) {
  const uint4* raw = reinterpret_cast<const uint4*>(slot + RAW_OFF);  // row r: raw[4 r .. 4 r + 3]
  const int l7 = lane & 7;
  const int g = (0x27D8 >> (2 * l7)) & 3, h = (0x66 >> l7) & 1;  // g = 0 2 1 3 3 1 2 0, h = 0 1 1 0 0 1 1 0
  uint4 held[4];
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {
    if (i == 2) {
      if (ld & 2u) {
#pragma unroll
        for (int j = 0; j < 4; ++j) held[j] = raw[4 * (96 + lane) + ((j + g) & 3)];
      }
      __syncwarp();  // half 0's codes are all read
    }
    if (i == 3) __syncwarp();  // the codes of rows 64-95 are all read
    if (!((ld >> (i >> 1)) & 1u)) continue;
    const int r = 32 * i + lane;
    const uint2 b = scl[r];
    const uint32_t e = ((kb < 4 ? b.x : b.y) >> (8 * (kb & 3))) & 0xFFu;
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = i == 3 ? held[j] : raw[4 * r + ((j + g) & 3)];
    uint8_t* row = slot + (r >> 3) * 1024 + l7 * 128;
    if (e <= 134u) {  // 2^(e - 7) is a bf16
      const uint32_t s = ((e + 120u) << 7) * 0x00010001u;
      const __nv_bfloat162 s2 = *reinterpret_cast<const __nv_bfloat162*>(&s);
      expand_row16<false>(row, v, g, h, l7, s2, s2);
    } else {  // 2^120, then 2^(e - 127)
      const uint32_t s1u = (247u << 7) * 0x00010001u, s2u = (e << 7) * 0x00010001u;
      expand_row16<true>(row, v, g, h, l7, *reinterpret_cast<const __nv_bfloat162*>(&s1u),
                         *reinterpret_cast<const __nv_bfloat162*>(&s2u));
    }
  }
}

// FP8: the caches hold fp8_ds_mla records (swamap64 / mainmap / mainmap64 then map their codes as
// bytes, and the rope maps their bf16 rope dims); else bf16 rows (the rope maps are unused).
template <bool FP8>
__global__ void __launch_bounds__(THREADS, 1)
    mla_partial_tc(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap swamap64,
                   const __grid_constant__ CUtensorMap mainmap, const __grid_constant__ CUtensorMap mainmap64,
                   const __grid_constant__ CUtensorMap ropeswa64, const __grid_constant__ CUtensorMap ropemain,
                   const __grid_constant__ CUtensorMap ropemain64, Args a) {
  extern __shared__ __align__(1024) uint8_t dsm[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  uint8_t* q_mem = base;             // Q_BYTES
  uint8_t* kv_mem = base + Q_BYTES;  // KV_BYTES: slot kb at kb * SLOT_BYTES
  Smem* sm = reinterpret_cast<Smem*>(kv_mem + KV_BYTES);
  volatile int* abort = &sm->abort;
  const dsv4_sparse_mla_decode_params& p = a.p;
  const int chunk = blockIdx.x, t = blockIdx.y, hg = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = t / p.q_per_seq;
  const TokenRows tr = token_plan(p, t);
  const int nh = chunk < tr.n_halves ? (tr.n_halves - chunk + a.n_chunks - 1) / a.n_chunks : 0;  // halves of this chunk
  const int64_t part = ((int64_t)t * a.n_chunks + chunk) * p.H + hg * HG;
  pdl_launch_dependents();
  if (nh <= 0 && !a.cluster_merge) {  // block-uniform: an empty chunk contributes nothing
    pdl_wait();
    if (threadIdx.x < HG) a.ml_part[part + threadIdx.x] = make_float2(-INFINITY, 0.f);
    return;
  }
  // (in a merging cluster an empty chunk runs through with no tiles: it joins the cluster's barriers)
  const int ntiles = nh > 0 ? (nh + 1) / 2 : 0;

  if (threadIdx.x == 0) {
    // fp8: groups 0-3 are released by the two softmax warps that expand their K-blocks
    for (int g = 0; g < NGROUPS; ++g) tc::mbar_init(&sm->full[g], FP8 && g < NGROUPS - 1 ? 2 : NPROD);
    for (int x = 0; x < NPROD * 4; ++x) tc::mbar_init(&sm->rawb[x / 4][x % 4], 1);
    tc::mbar_init(&sm->sbar, 33);  // fp8: loader 0's 32 lanes' exponent copies + its row masks
    for (int m = 0; m < 4; ++m) tc::mbar_init(&sm->vfree[m], 1);
    tc::mbar_init(&sm->sfull, 1);
    tc::mbar_init(&sm->pfull, 8);
    tc::mbar_init(&sm->pvdone, 1);
    tc::mbar_init(&sm->qfull, 1);
    tc::mbar_init(&sm->odone, 1);
    for (int x = 0; x < 4; ++x) tc::mbar_init(&sm->xbar[x >> 1][x & 1], 4);
    tc::mbar_init(&sm->ebar, 8);
    sm->abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == W_MMA) {
    tc::tmem_alloc(&sm->tmem_base, TMEM_COLS);
    tc::tmem_relinquish();
    tc::tc_fence_before();
  }
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  const bool loader = warp == W_LOAD || warp > W_MMA;
  const int pidx = warp == W_LOAD ? 0 : warp - W_MMA;  // loader index (warps 8, 10, 11)
  if (!loader) pdl_wait();
  // softmax warps' state, kept past the role split for the epilogue
  const int qd = warp & 3, hf = warp >> 2;
  const int R = qd * 32 + lane;
  const uint32_t lane_base = tmem + ((uint32_t)(qd * 32) << 16);
  float mref = -INFINITY;  // running max (log2 domain) of head 32 hf + lane
  float lsum = 0.f;        // this warp's rows' share of the sum of head 32 hf + lane
  bool have_o = false;     // softmax warps: every PV product has retired

  if (loader) {
    // ---------------- loads: three warps (the TMA issue rate is per issuing warp); loader pidx
    // issues K-blocks kb with kb % 3 == pidx of every tile, and arrives on each group's barrier with
    // the bytes it issued there
    if (pidx == 0 && lane == 0 && ntiles > 0) {
      tc::tma_prefetch_desc(&qmap);
      tc::tma_prefetch_desc(&swamap64);
      tc::tma_prefetch_desc(&mainmap);
      tc::tma_prefetch_desc(&mainmap64);
      if (FP8) {
        tc::tma_prefetch_desc(&ropeswa64);
        tc::tma_prefetch_desc(&ropemain);
        tc::tma_prefetch_desc(&ropemain64);
      }
    }
    pdl_wait();  // the queries, the caches and the top-k list come from earlier kernels
    if (pidx == 0 && lane == 0 && ntiles > 0) {
      tc::mbar_arrive_expect_tx(&sm->qfull, Q_BYTES);
      for (int kb = 0; kb < NKB; ++kb)
        tc::tma_load_2d(q_mem + kb * HG * 128, &qmap, kb * 64, t * p.H + hg * HG, &sm->qfull);
    }
    int armed_tile = -1, armed_groups = 0;
    bool ok = true;
    for (int i = 0; i < ntiles && ok; ++i) {
      HalfPlan hp[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int hh = chunk + (2 * i + u) * a.n_chunks;
        hp[u] = (2 * i + u < nh) ? plan_half(a, t, b, tr, hh, lane) : plan_half(a, t, b, tr, tr.n_halves, lane);
      }
      const uint32_t m0 = __ballot_sync(0xffffffffu, hp[0].v0), m1 = __ballot_sync(0xffffffffu, hp[0].v1);
      const uint32_t m2 = __ballot_sync(0xffffffffu, hp[1].v0), m3 = __ballot_sync(0xffffffffu, hp[1].v1);
      const uint32_t ld = (hp[0].kind != K_NONE ? 1u : 0u) | (hp[1].kind != K_NONE ? 2u : 0u);
      const int nload = __popc(ld);
      // gather rows: lanes 16u .. 16u + 15 load half u, lane g4 rows 4 g4 .. 4 g4 + 3
      const int gu = lane >> 4, g4 = lane & 15, src = (4 * g4) & 31;
      int r4[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int a0 = __shfl_sync(0xffffffffu, hp[0].y0, src + k), a1 = __shfl_sync(0xffffffffu, hp[0].y1, src + k);
        const int b0 = __shfl_sync(0xffffffffu, hp[1].y0, src + k), b1 = __shfl_sync(0xffffffffu, hp[1].y1, src + k);
        r4[k] = gu == 0 ? (g4 < 8 ? a0 : a1) : (g4 < 8 ? b0 : b1);
      }
      const int my_kind = gu == 0 ? hp[0].kind : hp[1].kind;
      for (int g = 0; g < NGROUPS; ++g) {
        if (i > 0) {
          int w = 1;
          if (lane == 0) w = tc::mbar_wait_bounded(&sm->vfree[g < 4 ? g : 3], (i - 1) & 1, abort);
          if (!__shfl_sync(0xffffffffu, w, 0)) {
            ok = false;
            break;
          }
        }
        const int kb0 = 2 * g, nkb = g < 4 ? 2 : 1;
        int mine = 0;  // K-blocks of this group that this loader issues
        for (int kb = kb0; kb < kb0 + nkb; ++kb) mine += kb % NPROD == pidx;
        if (FP8 && g == 0 && pidx == 0) {
          // the tile's block exponents (rows 64 u + 32 v + lane), now that the previous tile's
          // expansion is over (its S^T is done: vfree[0] has passed)
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const bool swa = hp[u].kind == K_BOX_SWA;
            const uint8_t* cache = reinterpret_cast<const uint8_t*>(swa ? p.swa_cache : p.main_cache);
            const int rows = swa ? a.swa_rows : a.main_rows;
#pragma unroll
            for (int v = 0; v < 2; ++v) {
              const int y = hp[u].kind == K_GATHER ? (v ? hp[u].y1 : hp[u].y0) : hp[u].ybox + 32 * v + lane;
              const bool in = hp[u].kind != K_NONE && y >= 0 && y < rows;
              // (a row with no record reads nothing and gets zeros; the address is still a valid one)
              const uint8_t* src = in ? cache + (int64_t)y * FP8_REC + FP8_SCALE_OFF
                                      : reinterpret_cast<const uint8_t*>(p.swa_cache);
              tc::cp_async8(&sm->scl[64 * u + 32 * v + lane], src, in ? 8u : 0u);
            }
          }
          tc::cp_async_mbar_arrive(&sm->sbar);
        }
        if (lane == 0) {
          if (g == 0 && pidx == 0) {
            sm->mask[i & 1][0] = m0;
            sm->mask[i & 1][1] = m1;
            sm->mask[i & 1][2] = m2;
            sm->mask[i & 1][3] = m3;
            sm->loaded[i & 1] = ld;
            if (FP8) tc::mbar_arrive(&sm->sbar);
          }
          if (!FP8 || g == NGROUPS - 1)  // bf16 rows (fp8: the rope slot) land on the group's barrier
            tc::mbar_arrive_expect_tx(&sm->full[g], (uint32_t)(nload * mine * HALF_BYTES));
          else if (mine > 0)  // fp8 codes land on the loader's own barrier, to be expanded first
            tc::mbar_arrive_expect_tx(&sm->rawb[pidx][g], (uint32_t)(nload * mine * RAW_HALF));
        }
        armed_tile = i;
        armed_groups = g + 1;
        __syncwarp();
        for (int kb = kb0; kb < kb0 + nkb; ++kb) {
          if (kb % NPROD != pidx) continue;
          const bool codes = FP8 && kb < NKB - 1;  // fp8 code bytes: staged, expanded once they land
          const bool rope = FP8 && !codes;         // fp8 rope dims: bf16 already
          uint8_t* dst = kv_mem + kb * SLOT_BYTES + (codes ? RAW_OFF : 0);
          const int hstride = codes ? RAW_HALF : HALF_BYTES, rstride = codes ? 64 : 128;
          uint64_t* bar = codes ? &sm->rawb[pidx][g] : &sm->full[g];
          const int x = rope ? 0 : kb * 64;
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int kind = hp[u].kind;
            if ((kind == K_BOX_SWA || kind == K_BOX_MAIN) && lane == 0) {
              const CUtensorMap* map = kind == K_BOX_SWA ? (rope ? &ropeswa64 : &swamap64)
                                                         : (rope ? &ropemain64 : &mainmap64);
              tc::tma_load_2d(dst + u * hstride, map, x, hp[u].ybox, bar);
            }
          }
          if (my_kind == K_GATHER)
            tc::tma_gather4(dst + gu * hstride + 4 * g4 * rstride, rope ? &ropemain : &mainmap, x, r4[0], r4[1], r4[2],
                            r4[3], bar);
        }
      }
    }
    if (lane == 0) {
      // every load into this CTA has landed before it may exit (already true unless it aborted)
      if (ntiles > 0 && pidx == 0) tc::mbar_wait_bounded(&sm->qfull, 0, abort, 100000000ull);
      for (int g = 0; g < armed_groups; ++g)
        tc::mbar_wait_bounded(&sm->full[g], armed_tile & 1, abort, 100000000ull);
      if (FP8)
        for (int g = 0; g < armed_groups && g < NGROUPS - 1; ++g)
          if ((2 * g) % NPROD == pidx || (2 * g + 1) % NPROD == pidx)
            tc::mbar_wait_bounded(&sm->rawb[pidx][g], armed_tile & 1, abort, 100000000ull);
    }
  } else if (warp == W_MMA) {
    if (lane == 0) {
      // ---------------- MMA issuer
      const uint32_t idesc_s = tc::idesc_bf16_f32(TILE, HG);
      const uint32_t idesc_o = tc::idesc_bf16_f32_amn_bmn(TILE, HG);
      const uint32_t q_addr = tc::smem_addr(q_mem), kv_addr = tc::smem_addr(kv_mem);
      const uint64_t a1 = tc::sdesc_k_sw128(kv_addr), b1 = tc::sdesc_k_sw128(q_addr);
      const uint64_t a2 = tc::sdesc_mn_sw128(kv_addr, SLOT_BYTES, 1024);
      const uint64_t b2 = tc::sdesc_mn_sw128(kv_addr + 8 * SLOT_BYTES, SLOT_BYTES, 1024);
      bool ok = ntiles == 0 || tc::mbar_wait_bounded(&sm->qfull, 0, abort);
      bool o_started = false;
      for (int i = 0; i < ntiles && ok; ++i) {
        for (int g = 0; g < NGROUPS && ok; ++g) {
          ok = tc::mbar_wait_bounded(&sm->full[g], i & 1, abort);
          if (!ok) break;
          tc::tc_fence_after();
          const int kb0 = 2 * g, nkb = g < 4 ? 2 : 1;
          for (int kb = kb0; kb < kb0 + nkb; ++kb) {
#pragma unroll
            for (int s = 0; s < 4; ++s)  // descriptor start addresses advance in 16-byte units
              tc::mma_bf16(tmem + COL_S, a1 + (uint64_t)((kb * SLOT_BYTES + s * 32) >> 4),
                           b1 + (uint64_t)((kb * HG * 128 + s * 32) >> 4), idesc_s, (kb | s) != 0);
          }
        }
        if (!ok) break;
        tc::mma_commit(&sm->sfull);
        ok = tc::mbar_wait_bounded(&sm->pfull, i & 1, abort);
        if (!ok) break;
        tc::tc_fence_after();
        const uint32_t ld = sm->loaded[i & 1];
        for (int m = 0; m < 4; ++m) {
          bool first = !o_started;
          for (int u = 0; u < 2; ++u) {
            if (!((ld >> u) & 1u)) continue;
#pragma unroll
            for (int s = 4 * u; s < 4 * u + 4; ++s) {
              tc::mma_bf16(tmem + COL_O + 64 * m, a2 + (uint64_t)((2 * m * SLOT_BYTES + s * 2048) >> 4),
                           b2 + (uint64_t)((s * 2048) >> 4), idesc_o, first ? 0u : 1u);
              first = false;
            }
          }
          tc::mma_commit(&sm->vfree[m]);
        }
        tc::mma_commit(&sm->pvdone);
        if (ld) o_started = true;
      }
      tc::mma_commit(&sm->odone);
    }
  } else {
    // ---------------- softmax + epilogue: warps 0-7; warp w owns tile rows R = 32 (w & 3) + lane (TMEM
    // lane R) and heads 32 hf .. 32 hf + 31 (hf = w >> 2)
    float lp[32];  // this thread's share of each of the 32 heads' sums
#pragma unroll
    for (int k = 0; k < 32; ++k) lp[k] = 0.f;
    bool ok = true;
    uint8_t* prow = kv_mem + 8 * SLOT_BYTES + (R >> 3) * 1024 + (R & 7) * 128;  // P^T row R
    float* mrow = sm->mrow[warp];
    for (int i = 0; i < ntiles; ++i) {
      if (FP8) {
        // K-block `warp` of this tile (8 warps, 8 code K-blocks): expanded once its codes and the
        // tile's block exponents are in, then its half of the group is released to the MMAs
        const int kb = warp, g = kb >> 1;
        if (!tc::mbar_wait_bounded(&sm->sbar, i & 1, abort) ||
            !tc::mbar_wait_bounded(&sm->rawb[kb % NPROD][g], i & 1, abort)) {
          ok = false;
          break;
        }
        expand_fp8_kblock(kv_mem + kb * SLOT_BYTES, sm->loaded[i & 1], sm->scl, kb, lane);
        tc::fence_proxy_async_smem();  // the MMAs read the expanded rows
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&sm->full[g]);
      }
      if (!tc::mbar_wait_bounded(&sm->sfull, i & 1, abort) ||
          !tc::mbar_wait_bounded(&sm->full[0], i & 1, abort)) {  // full[0] published the row mask
        ok = false;
        break;
      }
      tc::tc_fence_after();
      uint32_t r[32];
      tc::tmem_ld32_nowait(lane_base + COL_S + 32 * hf, r);
      tc::tmem_wait_ld_regs<32>(r);
      const bool valid = (sm->mask[i & 1][qd] >> lane) & 1u;
      const bool loaded = (sm->loaded[i & 1] >> (qd >> 1)) & 1u;
      float z[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) z[k] = valid ? __uint_as_float(r[k]) * a.c_log2 : -INFINITY;
      sm->red[i & 1][hf][qd][lane] = transpose_reduce32<true>(z, lane);
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm->xbar[i & 1][hf]);
      if (!tc::mbar_wait_bounded(&sm->xbar[i & 1][hf], (i >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      float mt = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; ++w) mt = fmaxf(mt, sm->red[i & 1][hf][w][lane]);
      float f = 1.f;
      if (mref == -INFINITY) {
        mref = mt;
      } else if (mt > mref + RESCALE_LOG2) {
        f = tc::ex2_approx(mref - mt);
        mref = mt;
      }
      // the same decision in the 4 warps of this head half: they computed it from the same maxima
      const bool resc = __any_sync(0xffffffffu, f != 1.f);
      mrow[lane] = mref;
      mrow[32 + lane] = f;
      __syncwarp();
      uint32_t pk[16];
#pragma unroll
      for (int k = 0; k < 32; k += 4) {
        const float4 m4 = *reinterpret_cast<const float4*>(mrow + k);
        const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
        float e[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) e[u] = mm[u] == -INFINITY ? 0.f : tc::ex2_approx(z[k + u] - mm[u]);
        if (resc) {
          const float4 f4 = *reinterpret_cast<const float4*>(mrow + 32 + k);
          lp[k] = fmaf(lp[k], f4.x, e[0]);
          lp[k + 1] = fmaf(lp[k + 1], f4.y, e[1]);
          lp[k + 2] = fmaf(lp[k + 2], f4.z, e[2]);
          lp[k + 3] = fmaf(lp[k + 3], f4.w, e[3]);
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u) lp[k + u] += e[u];
        }
        pk[k >> 1] = float2_to_bf16x2_bits(e[0], e[1]);
        pk[(k >> 1) + 1] = float2_to_bf16x2_bits(e[2], e[3]);
      }
      // P^T row R, heads 32 hf .. 32 hf + 31 = 16-byte chunks 4 hf .. 4 hf + 3, over slot 8 (QK^T of
      // this tile is done with it)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(prow + (((4 * hf + c) ^ (R & 7)) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      if (!valid && loaded) {  // a masked row that was loaded: zero its V so that 0 x garbage stays 0
        uint8_t* vrow = kv_mem + (R >> 3) * 1024 + (R & 7) * 128;
#pragma unroll
        for (int kb = 4 * hf; kb < 4 * hf + 4; ++kb)
#pragma unroll
          for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vrow + kb * SLOT_BYTES + c * 16) = make_uint4(0, 0, 0, 0);
      }
      tc::fence_proxy_async_smem();
      if (resc && i > 0) {
        // O^T must be stable (PV of the previous tile retired) before its columns are rescaled in place
        if (!tc::mbar_wait_bounded(&sm->pvdone, (i - 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        for (int m = 0; m < 4; ++m) {
          uint32_t o[32];
          tc::tmem_ld32_nowait(lane_base + COL_O + 64 * m + 32 * hf, o);
          tc::tmem_wait_ld_regs<32>(o);
#pragma unroll
          for (int k = 0; k < 32; k += 4) {
            const float4 f4 = *reinterpret_cast<const float4*>(mrow + 32 + k);
            o[k] = __float_as_uint(__uint_as_float(o[k]) * f4.x);
            o[k + 1] = __float_as_uint(__uint_as_float(o[k + 1]) * f4.y);
            o[k + 2] = __float_as_uint(__uint_as_float(o[k + 2]) * f4.z);
            o[k + 3] = __float_as_uint(__uint_as_float(o[k + 3]) * f4.w);
          }
          tc::tmem_st32(lane_base + COL_O + 64 * m + 32 * hf, o);
        }
        tc::tmem_wait_st();
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm->pfull);
    }
    lsum = transpose_reduce32<false>(lp, lane);
    have_o = __all_sync(0xffffffffu, ok && tc::mbar_wait_bounded(&sm->odone, 0, abort));
    if (have_o) tc::tc_fence_after();
    if (have_o && !a.cluster_merge) {
      // O^T (lane R = value dim 128 m + R, column = head) is turned into [head][value] rows in the
      // now idle tile buffer, then stored with 16-byte writes
      float* ot = reinterpret_cast<float*>(kv_mem);  // [64 heads][512 values] fp32 = 128 KB
      for (int m = 0; m < 4; ++m) {
        uint32_t o[32];
        tc::tmem_ld32_nowait(lane_base + COL_O + 64 * m + 32 * hf, o);
        tc::tmem_wait_ld_regs<32>(o);
#pragma unroll
        for (int k = 0; k < 32; ++k) ot[(32 * hf + k) * DV + 128 * m + R] = __uint_as_float(o[k]);
      }
      sm->lred[hf][qd][lane] = lsum;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm->ebar);
      if (tc::mbar_wait_bounded(&sm->ebar, 0, abort)) {
        float4* dst = reinterpret_cast<float4*>(a.o_part + part * DV);
        const float4* src = reinterpret_cast<const float4*>(ot);
        for (int x = threadIdx.x; x < HG * DV / 4; x += 256) dst[x] = src[x];
        if (qd == 0) {
          float l = 0.f;
#pragma unroll
          for (int w = 0; w < 4; ++w) l += sm->lred[hf][w][lane];
          a.ml_part[part + 32 * hf + lane] = make_float2(mref * 0.69314718055994531f, l);
        }
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && sm->abort) atomicOr(&g_flags_at, FLAG_TIMEOUT);
  if (a.cluster_merge) {
    // ---------------- merge of the chunks inside the cluster (every thread of every CTA reaches the
    // two cluster barriers, whatever happened before: nothing here waits on a flag).  CTA c owns value
    // dims [c WS, (c + 1) WS) of the 64 x 512 output block; every CTA pushes its scaled partial of each
    // owner's dims into that owner's shared memory (a slot per sender over its idle Q and tile
    // buffers), and each owner sums its slots locally.
    cg::cluster_group cl = cg::this_cluster();
    const int nc = a.n_chunks, crank = (int)cl.block_rank();
    const bool smx = warp < 8;
    const int h = 32 * hf + lane;
    const float sink_l2 = (smx && p.sink) ? p.sink[hg * HG + h] * 1.4426950408889634f : -INFINITY;
    if (smx) sm->lred[hf][qd][lane] = lsum;
    __syncthreads();
    if (smx && qd == 0) {
      float l = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) l += sm->lred[hf][w][lane];
      sm->cml[h] = make_float2(have_o ? mref : -INFINITY, l);
    }
    const int WS = ((DV + nc - 1) / nc + 3) & ~3;  // value dims an owner sums (a multiple of 4)
    float* recv = reinterpret_cast<float*>(q_mem);  // [sender][head][WS] fp32, <= 136 KB of the 216 KB
    cl.sync();  // every chunk's (max, sum) per head is in its shared memory and its buffers are idle
    if (smx) {
      // every chunk's (max, sum) of head h read at once: a remote read's latency is paid once, not nc times
      float2 ml[MAX_MERGE_CLUSTER];
#pragma unroll
      for (int c = 0; c < MAX_MERGE_CLUSTER; ++c)
        ml[c] = c < nc ? cl.map_shared_rank(sm->cml, c)[h] : make_float2(-INFINITY, 0.f);
      float M = sink_l2;
#pragma unroll
      for (int c = 0; c < MAX_MERGE_CLUSTER; ++c) M = fmaxf(M, ml[c].x);
      float L = (M == -INFINITY || p.sink == nullptr) ? 0.f : tc::ex2_approx(sink_l2 - M);
#pragma unroll
      for (int c = 0; c < MAX_MERGE_CLUSTER; ++c)
        if (ml[c].x != -INFINITY) L += ml[c].y * tc::ex2_approx(ml[c].x - M);
      const float mine = sm->cml[h].x;
      sm->mrow[warp][lane] = (mine == -INFINITY || !(L > 0.f)) ? 0.f : tc::ex2_approx(mine - M) / L;
      if (crank == 0 && qd == 0 && p.lse)
        p.lse[(int64_t)t * p.H + hg * HG + h] = L > 0.f ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
      __syncwarp();
      // the weights of the warp's 32 heads (0 for a chunk without output)
      float wgt[32];
#pragma unroll
      for (int k = 0; k < 32; k += 4) {
        const float4 f4 = *reinterpret_cast<const float4*>(&sm->mrow[warp][k]);
        wgt[k] = have_o ? f4.x : 0.f;
        wgt[k + 1] = have_o ? f4.y : 0.f;
        wgt[k + 2] = have_o ? f4.z : 0.f;
        wgt[k + 3] = have_o ? f4.w : 0.f;
      }
      // this chunk's O^T scaled by the weights, value dim d = 128 m + R of heads 32 hf .. + 31, pushed
      // to the owner of d; two TMEM loads in flight at a time
      for (int m = 0; m < 4; m += 2) {
        uint32_t o[64];
        if (have_o) {
          tc::tmem_ld32_nowait(lane_base + COL_O + 64 * m + 32 * hf, o);
          tc::tmem_ld32_nowait(lane_base + COL_O + 64 * (m + 1) + 32 * hf, o + 32);
          tc::tmem_wait_ld_regs<64>(o);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int d = 128 * (m + u) + R, own = d / WS;
          float* dst = cl.map_shared_rank(recv, own) + ((size_t)crank * HG + 32 * hf) * WS + (d - own * WS);
#pragma unroll
          for (int k = 0; k < 32; ++k)  // (a zero weight gives 0 whatever O^T holds, NaN included)
            dst[k * WS] = wgt[k] == 0.f ? 0.f : __uint_as_float(o[32 * u + k]) * wgt[k];
        }
      }
    }
    cl.sync();  // every chunk's partials are in their owners' shared memory (no remote access after this)
    {
      // this CTA sums its dims [d0, d0 + 4 w4) over the senders' slots and writes the output
      const int d0 = min(DV, crank * WS), w4 = (min(DV, d0 + WS) - d0) / 4;
      const int64_t obase = ((int64_t)t * p.H + hg * HG) * DV;
      for (int x = threadIdx.x; x < HG * w4; x += THREADS) {
        const int hh = x / w4, q = x - hh * w4;
        const float4* src = reinterpret_cast<const float4*>(recv + (size_t)hh * WS) + q;
        float4 acc = src[0];
        for (int c = 1; c < nc; ++c) {
          const float4 v = src[(size_t)c * HG * WS / 4];
          acc.x += v.x;
          acc.y += v.y;
          acc.z += v.z;
          acc.w += v.w;
        }
        const int64_t o = obase + (int64_t)hh * DV + d0 + 4 * q;
        if (p.out_dtype == DSV4_F32) {
          reinterpret_cast<float4*>(p.out)[o / 4] = acc;
        } else {
          reinterpret_cast<uint2*>(p.out)[o / 4] =
              make_uint2(float2_to_bf16x2_bits(acc.x, acc.y), float2_to_bf16x2_bits(acc.z, acc.w));
        }
      }
    }
  }
  if (warp == W_MMA) {
    // no MMA may still write TMEM when it is released (already true unless the CTA aborted)
    if (lane == 0) tc::mbar_wait_bounded(&sm->odone, 0, abort, 100000000ull);
    __syncwarp();
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}
}  // namespace attc

static bool use_tc_attention(const dsv4_sparse_mla_decode_params& p) {
  return (p.cache_dtype == DSV4_BF16 || p.cache_dtype == DSV4_FP8_DS_MLA) && p.q_dtype == DSV4_BF16 &&
         p.H % attc::HG == 0 && p.page_size == 64;
}

static cudaError_t launch_mla_partial_tc(const dsv4_sparse_mla_decode_params& p, const AtLayout& L, float* o_part,
                                         float2* ml_part, cudaStream_t st) {
  using namespace attc;
  Args a;
  a.p = p;
  a.o_part = o_part;
  a.ml_part = ml_part;
  a.n_chunks = L.n_chunks;
  a.swa_rows = (int)(p.swa_num_pages * p.page_size);
  a.main_rows = p.ratio > 0 ? (int)(p.main_num_pages * p.page_size) : a.swa_rows;
  a.c_log2 = p.softmax_scale * 1.4426950408889634f;
  a.cluster_merge = L.n_chunks <= MAX_MERGE_CLUSTER ? 1 : 0;
  const bool fp8 = p.cache_dtype == DSV4_FP8_DS_MLA;
  CUtensorMap qmap, swamap64, mainmap, mainmap64, ropeswa64, ropemain, ropemain64;
  cudaError_t e = make_tmap_2d_bf16(&qmap, p.q, (uint64_t)D, (uint64_t)p.T * p.H, 64, HG);
  if (e != cudaSuccess) return e;
  // a cache's maps: bf16 rows (K-blocks of 64 dims, swizzled), or for fp8_ds_mla records their
  // 512 code bytes (64-byte boxes, untiled) and their 64 bf16 rope dims (swizzled)
  auto cache_maps = [&](const void* cache, int rows, uint32_t box_rows, CUtensorMap* codes, CUtensorMap* rope) {
    if (!fp8) {
      *rope = qmap;  // unused
      return make_tmap_2d_bf16(codes, cache, (uint64_t)D, (uint64_t)rows, 64, box_rows);
    }
    cudaError_t r = make_tmap_2d(codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, cache, (uint64_t)DV, (uint64_t)rows,
                                 (uint64_t)FP8_REC, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (r != cudaSuccess) return r;
    return make_tmap_2d(rope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, reinterpret_cast<const uint8_t*>(cache) + FP8_ROPE_OFF,
                        (uint64_t)(D - DV), (uint64_t)rows, (uint64_t)FP8_REC, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
  };
  e = cache_maps(p.swa_cache, a.swa_rows, HALF, &swamap64, &ropeswa64);
  if (e != cudaSuccess) return e;
  if (p.ratio > 0) {
    e = cache_maps(p.main_cache, a.main_rows, 1, &mainmap, &ropemain);
    if (e != cudaSuccess) return e;
    e = cache_maps(p.main_cache, a.main_rows, HALF, &mainmap64, &ropemain64);
    if (e != cudaSuccess) return e;
  } else {  // no compressed rows: the main-cache maps are never used (still valid maps)
    e = cache_maps(p.swa_cache, a.swa_rows, 1, &mainmap, &ropemain);
    if (e != cudaSuccess) return e;
    mainmap64 = swamap64;
    ropemain64 = ropeswa64;
  }
  const size_t smem = 1024 + (size_t)Q_BYTES + (size_t)KV_BYTES + sizeof(Smem);
  e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(mla_partial_tc<false>), (int)smem);
  if (e == cudaSuccess) e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(mla_partial_tc<true>), (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.n_chunks, p.T, p.H / HG);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;  // the chunks of one (token, head group)
  attr[1].val.clusterDim.x = a.cluster_merge ? L.n_chunks : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (fp8)
    return count_launch(cudaLaunchKernelEx(&cfg, mla_partial_tc<true>, qmap, swamap64, mainmap, mainmap64, ropeswa64,
                                           ropemain, ropemain64, a));
  return count_launch(cudaLaunchKernelEx(&cfg, mla_partial_tc<false>, qmap, swamap64, mainmap, mainmap64, ropeswa64,
                                         ropemain, ropemain64, a));
}

// ------------------------------------------------------------------------------------------------
// Merge of the chunk partials (m_c, l_c, unnormalised O_c) with the sink: CTA per (token, head).
// ------------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(MERGE_THREADS) mla_merge(dsv4_sparse_mla_decode_params p, const float* o_part,
                                                           const float2* ml_part, int n_chunks) {
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const float sink = p.sink ? p.sink[h] : -INFINITY;
  float M = sink;
  for (int c = 0; c < n_chunks; ++c) M = fmaxf(M, ml_part[((int64_t)t * n_chunks + c) * p.H + h].x);
  float L = (M == -INFINITY) ? 0.f : expf(sink - M);
  float2 acc = make_float2(0.f, 0.f);
  for (int c = 0; c < n_chunks; ++c) {
    const int64_t part = ((int64_t)t * n_chunks + c) * p.H + h;
    const float2 ml = ml_part[part];
    if (ml.x == -INFINITY) continue;
    const float wgt = expf(ml.x - M);
    L += ml.y * wgt;
    const float2 o = reinterpret_cast<const float2*>(o_part + part * DV)[tid];
    acc.x = fmaf(wgt, o.x, acc.x);
    acc.y = fmaf(wgt, o.y, acc.y);
  }
  const float inv = L > 0.f ? 1.0f / L : 0.f;
  const int64_t orow = ((int64_t)t * p.H + h) * DV;
  if (p.out_dtype == DSV4_F32)
    reinterpret_cast<float2*>(p.out)[orow / 2 + tid] = make_float2(acc.x * inv, acc.y * inv);
  else
    reinterpret_cast<uint32_t*>(p.out)[orow / 2 + tid] = float2_to_bf16x2_bits(acc.x * inv, acc.y * inv);
  if (p.lse && tid == 0) p.lse[(int64_t)t * p.H + h] = (L > 0.f) ? M + logf(L) : -INFINITY;
}

cudaError_t launch_sparse_mla_decode(const dsv4_sparse_mla_decode_params& p, cudaStream_t st) {
  if (p.T == 0) return cudaSuccess;
  AtLayout L = at_layout(p);
  char* ws = reinterpret_cast<char*>(p.workspace);
  float* o_part = reinterpret_cast<float*>(ws + L.o_off);
  float2* ml_part = reinterpret_cast<float2*>(ws + L.ml_off);
  cudaError_t e;
  if (use_tc_attention(p)) {
    e = launch_mla_partial_tc(p, L, o_part, ml_part, st);
    if (e != cudaSuccess) return e;
    if (L.n_chunks <= attc::MAX_MERGE_CLUSTER) return cudaSuccess;  // merged inside the kernel's clusters
  } else {
    const size_t smem = sizeof(float) * ((size_t)AT_HG * D + (size_t)AT_CH * (D + 1) + (size_t)AT_HG * AT_CH);
    e = cudaFuncSetAttribute(mla_partial_simt, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(mla_partial_simt, dim3(L.n_chunks, p.T, (p.H + AT_HG - 1) / AT_HG), dim3(AT_THREADS), smem, st, true, p,
                   o_part, ml_part, L.n_chunks);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(mla_merge, dim3(p.T, p.H), dim3(MERGE_THREADS), 0, st, true, p, (const float*)o_part,
                    (const float2*)ml_part, L.n_chunks);
}

cudaError_t read_flags_attention(uint32_t* f) {
  unsigned int v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_flags_at, sizeof(v));
  if (e != cudaSuccess) return e;
  *f |= v;
  return cudaMemcpyToSymbol(g_flags_at, &z, sizeof(z));
}

}  // namespace dsv4
