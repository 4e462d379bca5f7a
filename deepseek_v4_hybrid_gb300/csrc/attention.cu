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
#include "dsv4_common.cuh"
#include "dsv4_launch.h"
#include "tc_ptx.cuh"
#include "tmap.h"

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
  n_swa = (n_swa + 63) / 64 * 64;  // the tensor-core kernel pads the window part to whole tiles
  int n_cmp = 0;
  if (p.ratio > 0) n_cmp = p.topk_idx ? p.topk : p.max_context / p.ratio;
  return n_swa + n_cmp;
}

static bool use_tc_attention(const dsv4_sparse_mla_decode_params& p);

// Rows per CTA of the tensor-core kernel: about one wave of CTAs over the SMs (each (token, head
// group) has two CTAs, one per value half), in whole 64-row tiles.
static int tc_chunk_rows(const dsv4_sparse_mla_decode_params& p) {
  const int per_chunk = p.T * (p.H / 64) * 2;
  int n = per_chunk > 0 ? num_sms() / per_chunk : 1;
  if (n < 1) n = 1;
  const int rows = max_rows(p);
  int c = (rows + n - 1) / n;
  c = (c + 63) / 64 * 64;
  return c < 64 ? 64 : c;
}

static AtLayout at_layout(const dsv4_sparse_mla_decode_params& p) {
  AtLayout L;
  L.chunk_rows = use_tc_attention(p) ? tc_chunk_rows(p) : AT_CH;
  L.n_chunks = (max_rows(p) + L.chunk_rows - 1) / L.chunk_rows;
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
// group x value half); the two value halves form a 2-CTA cluster and share every load: each CTA
// issues half of the TMA traffic (Q, gathers, page boxes) with multicast to both, and both CTAs'
// P V commits release a stage in both.  Heads are the MMA M dimension (M = 128, lanes 64..127 unused), rows the
// N dimension of S = Q K^T (K = 576 in 9 K-blocks of 64 dims) and the K dimension of
// O[:, half] += P V[:, half] (N = 256 value dims).
//
// Warp 2 gathers 64-row tiles with TMA gather4 loads (4 rows x one 64-dim K-block each) straight
// into the 128-byte swizzled K-major layout the MMA reads, so any row order (window positions,
// top-k indices, dense runs) works; a masked row is loaded from past the end of the tensor (zeros).
// Lane 0 of warp 3 issues the MMAs; S goes to one of two TMEM buffers, P (bf16) is written back
// to TMEM by the softmax warps and read from there as the A operand of the P V product; O stays in
// TMEM for the whole chunk.  Warps 0-1 (one head per thread, TMEM lanes 0-63) run the online
// softmax in the log2 domain with a lazy rescale (O is only rescaled when the running max grows
// by more than 2^8), then write the unnormalised O and (max, sum) of the chunk.
// ------------------------------------------------------------------------------------------------
namespace attc {
constexpr int TILE = 64;
constexpr int HG = 64;
constexpr int DVH = 256;
constexpr int NKB = 9;
constexpr int KB_BYTES = TILE * 128;          // 8 KB
constexpr int STAGE_BYTES = NKB * KB_BYTES;   // 72 KB
constexpr int Q_BYTES = NKB * HG * 128;       // 72 KB
constexpr int STAGES = 2;
constexpr int THREADS = 192;  // warps 0-1 and 4-5 softmax, 2 producer, 3 MMA
constexpr uint32_t COL_O = 0, COL_S = 256, COL_P = 384;  // S: 2 x 64 columns, P: 2 x 32 columns
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_LOG2 = 8.0f;
constexpr uint32_t FLAG_TIMEOUT = 4u;

struct Args {
  dsv4_sparse_mla_decode_params p;
  float* o_part;
  float2* ml_part;
  int n_chunks, chunk_rows;
  int swa_rows, main_rows;  // rows of the two tensor maps (a masked row loads from this index)
  float c_log2;             // softmax_scale * log2(e)
};

struct Smem {
  uint64_t full[STAGES], empty[STAGES], sfull[2], pfull[2], pvdone[2], qfull, odone;
  uint64_t mask[STAGES];
  uint64_t xbar[2], lbar;  // exchanges between the two softmax halves (4 warps arrive)
  float xmax[2][2][HG];  // [tile parity][half][head] row maxima
  float lsum[2][HG];     // [half][head] softmax sums
  uint32_t tmem_base;
  int abort;
};

// Row list of the tensor-core kernel: the window rows, padded with masked rows to a multiple of 64 so
// that every 64-row tile reads a single cache, then the compressed rows.
__device__ __forceinline__ int padded_window(int n_swa) { return (n_swa + TILE - 1) / TILE * TILE; }

// Source row of entry r (row index into the SWA cache if r is a window row, into the main cache
// otherwise); a masked row gets the map's out-of-range row, which loads zeros.
__device__ __forceinline__ int row_source(const Args& a, int t, int b, int pos, int n_swa, int nc, int n_rows, int r,
                                          bool& valid) {
  const dsv4_sparse_mla_decode_params& p = a.p;
  const int n_win = padded_window(n_swa);
  valid = false;
  if (r < n_win) {
    if (r >= n_swa || r >= n_rows) return a.swa_rows;
    const int q = pos - n_swa + 1 + r;
    const int lp = q / p.page_size;
    const int page = lp < p.swa_max_pages ? p.swa_block_table[(int64_t)b * p.swa_max_pages + lp] : -1;
    if (page < 0 || page >= p.swa_num_pages) {
      atomicOr(&g_flags_at, FLAG_PAGE);
      return a.swa_rows;
    }
    valid = true;
    return page * p.page_size + q % p.page_size;
  }
  if (r >= n_rows) return a.main_rows;
  const int i = r - n_win;
  int j = i;
  if (p.topk_idx != nullptr) {
    j = p.topk_idx[(int64_t)t * p.topk + i];
    if (j < 0) return a.main_rows;
    if (j >= nc) {
      atomicOr(&g_flags_at, FLAG_TOPK);
      return a.main_rows;
    }
  }
  const int lp = j / p.page_size;
  const int page = lp < p.main_max_pages ? p.main_block_table[(int64_t)b * p.main_max_pages + lp] : -1;
  if (page < 0 || page >= p.main_num_pages) {
    atomicOr(&g_flags_at, FLAG_PAGE);
    return a.main_rows;
  }
  valid = true;
  return page * p.page_size + j % p.page_size;
}

__global__ void __launch_bounds__(THREADS, 1)
    mla_partial_tc(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap swamap,
                   const __grid_constant__ CUtensorMap mainmap, const __grid_constant__ CUtensorMap mainmap64,
                   Args a) {
  extern __shared__ __align__(1024) uint8_t dsm[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  uint8_t* q_mem = base;                     // Q_BYTES (GEMM1 rows 64..127 read the next 8 KB: still smem)
  uint8_t* stage_mem = base + Q_BYTES;       // STAGES x STAGE_BYTES
  Smem* sm = reinterpret_cast<Smem*>(stage_mem + STAGES * STAGE_BYTES);
  volatile int* abort = &sm->abort;

  const dsv4_sparse_mla_decode_params& p = a.p;
  const int chunk = blockIdx.x, t = blockIdx.y;
  const int hg = blockIdx.z >> 1, dh = blockIdx.z & 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = t / p.q_per_seq;
  int pos = p.positions[t];
  int n_swa, nc, n_cmp;
  token_rows(p, pos, n_swa, nc, n_cmp);
  const int n_rows = padded_window(n_swa) + n_cmp;
  const int r0 = chunk * a.chunk_rows;
  const int rows = min(a.chunk_rows, n_rows - r0);
  const int64_t part = ((int64_t)t * a.n_chunks + chunk) * p.H + hg * HG;
  pdl_launch_dependents();
  if (rows <= 0) {  // block-uniform: an empty chunk contributes nothing
    pdl_wait();
    if (dh == 0 && threadIdx.x < HG) a.ml_part[part + threadIdx.x] = make_float2(-INFINITY, 0.f);
    return;
  }
  const int ntiles = (rows + TILE - 1) / TILE;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&sm->full[s], 1);
      tc::mbar_init(&sm->empty[s], 2);  // both CTAs of the pair release a stage (multicast commit)
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sm->sfull[i], 1);
      tc::mbar_init(&sm->pfull[i], 4);
      tc::mbar_init(&sm->xbar[i], 4);
      tc::mbar_init(&sm->pvdone[i], 1);
    }
    tc::mbar_init(&sm->qfull, 1);
    tc::mbar_init(&sm->odone, 1);
    tc::mbar_init(&sm->lbar, 4);
    sm->abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == 3) {
    tc::tmem_alloc(&sm->tmem_base, TMEM_COLS);
    tc::tmem_relinquish();
    tc::tc_fence_before();
  }
  tc::cluster_sync_all();  // the partner's barriers exist before any multicast targets them
  tc::tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  const uint32_t crank = tc::cluster_rank();  // 0 or 1: which half of every load this CTA issues
  if (warp != 2) pdl_wait();

  if (warp == 2) {
    // ---------------- producer: Q by TMA, then each 64-row tile by 144 TMA gather4 loads (lane g < 16
    // loads rows 4g..4g+3 of all 9 K-blocks); the window part of the list is tile-aligned, so a tile
    // reads one cache
    if (lane == 0) {
      tc::tma_prefetch_desc(&qmap);
      tc::tma_prefetch_desc(&swamap);
      tc::tma_prefetch_desc(&mainmap);
      tc::mbar_arrive_expect_tx(&sm->qfull, Q_BYTES);
      for (int kb = (int)crank; kb < NKB; kb += 2)
        tc::tma_load_2d_mc(q_mem + kb * HG * 128, &qmap, kb * 64, t * p.H + hg * HG, &sm->qfull, 0x3);
    }
    pdl_wait();  // the caches and the top-k list come from earlier kernels
    const int n_win = padded_window(n_swa);
    bool v0, v1;
    int y0 = row_source(a, t, b, pos, n_swa, nc, n_rows, r0 + lane, v0);
    int y1 = row_source(a, t, b, pos, n_swa, nc, n_rows, r0 + lane + 32, v1);
    for (int i = 0; i < ntiles; ++i) {
      const int stage = i % STAGES;
      const int tr0 = r0 + i * TILE;
      const bool in0 = i * TILE + lane < rows, in1 = i * TILE + lane + 32 < rows;
      const bool use_main = tr0 >= n_win;
      const int oob = use_main ? a.main_rows : a.swa_rows;
      if (!(v0 && in0)) y0 = oob;
      if (!(v1 && in1)) y1 = oob;
      const unsigned b0 = __ballot_sync(0xffffffffu, v0 && in0), b1 = __ballot_sync(0xffffffffu, v1 && in1);
      // rows 4g..4g+3 for lane g < 16
      const int g = lane & 15;
      const int src_lane = (4 * g) & 31;
      int r4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int ya = __shfl_sync(0xffffffffu, y0, src_lane + u);
        const int yb = __shfl_sync(0xffffffffu, y1, src_lane + u);
        r4[u] = g < 8 ? ya : yb;
      }
      int ok = 1;
      if (lane == 0) ok = tc::mbar_wait_bounded(&sm->empty[stage], ((i / STAGES) & 1) ^ 1, abort);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      uint8_t* st = stage_mem + stage * STAGE_BYTES;
      if (lane == 0) {
        sm->mask[stage] = (uint64_t)b0 | ((uint64_t)b1 << 32);
        tc::mbar_arrive_expect_tx(&sm->full[stage], (uint32_t)TILE * NKB * 128);
      }
      __syncwarp();
      // a dense (no top-k list) compressed tile whose 64 rows are all valid is one whole page
      const int dense_page = (use_main && p.topk_idx == nullptr && (b0 & b1) == 0xffffffffu)
                                 ? __shfl_sync(0xffffffffu, y0, 0) / p.page_size : -1;
      if (dense_page >= 0) {
        if (lane == 0) {
          for (int kb = (int)crank; kb < NKB; kb += 2)
            tc::tma_load_2d_mc(st + kb * KB_BYTES, &mainmap64, kb * 64, dense_page * p.page_size, &sm->full[stage], 0x3);
        }
      } else if (lane < 16 && (lane >> 3) == (int)crank) {  // CTA 0 gathers rows 0-31, CTA 1 rows 32-63
        const CUtensorMap* map = use_main ? &mainmap : &swamap;
#pragma unroll
        for (int kb = 0; kb < NKB; ++kb)
          tc::tma_gather4_mc(st + kb * KB_BYTES + 4 * g * 128, map, kb * 64, r4[0], r4[1], r4[2], r4[3], &sm->full[stage],
                             0x3);
      }
      if (i + 1 < ntiles) {  // look up the next tile's rows while this one is in flight
        y0 = row_source(a, t, b, pos, n_swa, nc, n_rows, tr0 + TILE + lane, v0);
        y1 = row_source(a, t, b, pos, n_swa, nc, n_rows, tr0 + TILE + lane + 32, v1);
      }
    }
    if (lane == 0) {
      // every load into this CTA has landed, and both CTAs' last stage releases (multicast commits
      // into this CTA) have arrived, before the closing cluster barrier lets the partner exit
      tc::mbar_wait_bounded(&sm->qfull, 0, abort, 100000000ull);
      for (int i = (ntiles > STAGES ? ntiles - STAGES : 0); i < ntiles; ++i) {
        tc::mbar_wait_bounded(&sm->full[i % STAGES], (i / STAGES) & 1, abort, 100000000ull);
        tc::mbar_wait_bounded(&sm->empty[i % STAGES], (i / STAGES) & 1, abort, 100000000ull);
      }
    }
  } else if (warp == 3) {
    if (lane == 0) {
      // ---------------- MMA issuer
      const uint32_t idesc_s = tc::idesc_bf16_f32(128, TILE);
      const uint32_t idesc_o = tc::idesc_bf16_f32_bmn(128, DVH);
      const uint32_t q_addr = tc::smem_addr(q_mem);
      bool ok = tc::mbar_wait_bounded(&sm->qfull, 0, abort);
      // S = Q K^T of tile i needs the tile (full[i]) and a free S buffer (the softmax of tile i - 2
      // done, i.e. P V of tile i - 2 issued); P V of tile j needs P (pfull[j]).  Each is issued as soon
      // as it is ready, so a stage is released right after its P V, not one tile load later.
      int ns = 0, np = 0;  // next S tile, next P V tile
      uint64_t t_start = 0;
      while (ok && np < ntiles) {
        bool progressed = false;
        if (ns < ntiles && ns <= np + 1 && tc::mbar_try_wait(&sm->full[ns % STAGES], (ns / STAGES) & 1)) {
          tc::tc_fence_after();
          const uint32_t k_addr = tc::smem_addr(stage_mem + (ns % STAGES) * STAGE_BYTES);
          for (int kb = 0; kb < NKB; ++kb) {
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              const uint64_t ad = tc::sdesc_k_sw128(q_addr + kb * HG * 128 + s * 32);
              const uint64_t bd = tc::sdesc_k_sw128(k_addr + kb * KB_BYTES + s * 32);
              tc::mma_bf16(tmem + COL_S + (ns & 1) * TILE, ad, bd, idesc_s, (kb | s) != 0);
            }
          }
          tc::mma_commit(&sm->sfull[ns & 1]);
          ++ns;
          progressed = true;
        }
        if (np < ns && tc::mbar_try_wait(&sm->pfull[np & 1], (np >> 1) & 1)) {
          tc::tc_fence_after();
          const uint32_t v_addr = tc::smem_addr(stage_mem + (np % STAGES) * STAGE_BYTES + (4 * dh) * KB_BYTES);
#pragma unroll
          for (int s = 0; s < TILE / 16; ++s) {
            const uint64_t bd = tc::sdesc_mn_sw128(v_addr + s * 2048, KB_BYTES, 1024);
            tc::mma_bf16_ts(tmem + COL_O, tmem + COL_P + (np & 1) * 32 + s * 8, bd, idesc_o,
                            (np > 0 || s > 0) ? 1u : 0u);
          }
          tc::mma_commit_mc(&sm->empty[np % STAGES], 0x3);
          tc::mma_commit(&sm->pvdone[np & 1]);
          ++np;
          progressed = true;
        }
        if (progressed) {
          t_start = 0;
        } else {  // bounded spin, like every other wait
          if (*abort) ok = false;
          const uint64_t now = tc::globaltimer_ns();
          if (t_start == 0) t_start = now;
          else if (now - t_start > 250000000ull) {
            *abort = 1;
            ok = false;
          }
        }
      }
      tc::mma_commit(&sm->odone);
    }
  } else {
    // ---------------- softmax + epilogue: warps 0-1 and 4-5, thread = head (TMEM lane); warps 0-1 own
    // S columns 0-31, O columns 0-127 and P columns 0-15 of the tile, warps 4-5 the other halves
    const int half = warp >> 2;
    const int h = (warp & 3) * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t s_col = COL_S + half * 32, o_col = COL_O + half * (DVH / 2), p_col = COL_P + half * 16;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int i = 0; i < ntiles; ++i) {
      if (!tc::mbar_wait_bounded(&sm->sfull[i & 1], (i >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      // the stage's row mask was published with its full barrier
      tc::mbar_wait_bounded(&sm->full[i % STAGES], (i / STAGES) & 1, abort);
      tc::tc_fence_after();
      uint32_t r[32];
      tc::tmem_ld32_nowait(lane_base + s_col + (i & 1) * TILE, r);
      tc::tmem_wait_ld_regs<32>(r);
      const uint32_t mask = (uint32_t)(sm->mask[i % STAGES] >> (32 * half));
      float z[32];
      float mt = -INFINITY;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        z[k] = ((mask >> k) & 1u) ? __uint_as_float(r[k]) * a.c_log2 : -INFINITY;
        mt = fmaxf(mt, z[k]);
      }
      // row max over both halves (an mbarrier, so the wait is bounded like every other one)
      sm->xmax[i & 1][half][h] = mt;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm->xbar[i & 1]);
      if (!tc::mbar_wait_bounded(&sm->xbar[i & 1], (i >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      mt = fmaxf(mt, sm->xmax[i & 1][half ^ 1][h]);
      const float m_new = fmaxf(m_ref, mt);
      if (m_ref == -INFINITY) {
        m_ref = m_new;  // nothing accumulated yet that is not zero
      } else if (m_new > m_ref + RESCALE_LOG2) {
        // O must be stable (the previous P V done) before it is rescaled in place
        if (!tc::mbar_wait_bounded(&sm->pvdone[(i - 1) & 1], ((i - 1) >> 1) & 1, abort)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        const float f = tc::ex2_approx(m_ref - m_new);
        l *= f;
        for (int c = 0; c < DVH / 2; c += 32) {
          uint32_t o[32];
          tc::tmem_ld32_nowait(lane_base + o_col + c, o);
          tc::tmem_wait_ld_regs<32>(o);
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
          tc::tmem_st32(lane_base + o_col + c, o);
        }
        tc::tmem_wait_st();
        m_ref = m_new;
      }
      uint32_t pk[16];
      float ls = 0.f;
      const bool live = m_ref != -INFINITY;
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float e0 = live ? tc::ex2_approx(z[2 * k] - m_ref) : 0.f;
        const float e1 = live ? tc::ex2_approx(z[2 * k + 1] - m_ref) : 0.f;
        ls += e0 + e1;
        pk[k] = float2_to_bf16x2_bits(e0, e1);
      }
      l += ls;
      // P buffer (i & 1) was last read by the P V product of tile i - 2
      if (i >= 2 && !tc::mbar_wait_bounded(&sm->pvdone[i & 1], ((i - 2) >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      tc::tmem_st16(lane_base + p_col + (i & 1) * 32, pk);
      tc::tmem_wait_st();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm->pfull[i & 1]);
    }
    if (ok && tc::mbar_wait_bounded(&sm->odone, 0, abort)) {
      tc::tc_fence_after();
      float* dst = a.o_part + (part + h) * DV + dh * DVH + half * (DVH / 2);
      for (int c = 0; c < DVH / 2; c += 32) {
        uint32_t o[32];
        tc::tmem_ld32_nowait(lane_base + o_col + c, o);
        tc::tmem_wait_ld_regs<32>(o);
#pragma unroll
        for (int k = 0; k < 32; k += 4)
          *reinterpret_cast<float4*>(dst + c + k) = make_float4(__uint_as_float(o[k]), __uint_as_float(o[k + 1]),
                                                                 __uint_as_float(o[k + 2]), __uint_as_float(o[k + 3]));
      }
      sm->lsum[half][h] = l;  // the two halves' sums
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm->lbar);
      if (tc::mbar_wait_bounded(&sm->lbar, 0, abort) && dh == 0 && half == 0)
        a.ml_part[part + h] = make_float2(m_ref * 0.69314718055994531f, l + sm->lsum[1][h]);
    }
  }
  tc::cluster_sync_all();  // the partner no longer loads into or releases through this CTA
  if (threadIdx.x == 0 && sm->abort) atomicOr(&g_flags_at, FLAG_TIMEOUT);
  if (warp == 3) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}
}  // namespace attc

static bool use_tc_attention(const dsv4_sparse_mla_decode_params& p) {
  return p.cache_dtype == DSV4_BF16 && p.q_dtype == DSV4_BF16 && p.H % attc::HG == 0 && p.page_size == 64;
}

static cudaError_t launch_mla_partial_tc(const dsv4_sparse_mla_decode_params& p, const AtLayout& L, float* o_part,
                                         float2* ml_part, cudaStream_t st) {
  using namespace attc;
  Args a;
  a.p = p;
  a.o_part = o_part;
  a.ml_part = ml_part;
  a.n_chunks = L.n_chunks;
  a.chunk_rows = L.chunk_rows;
  a.swa_rows = (int)(p.swa_num_pages * p.page_size);
  a.main_rows = p.ratio > 0 ? (int)(p.main_num_pages * p.page_size) : a.swa_rows;
  a.c_log2 = p.softmax_scale * 1.4426950408889634f;
  CUtensorMap qmap, swamap, mainmap, mainmap64;
  cudaError_t e = make_tmap_2d_bf16(&qmap, p.q, (uint64_t)D, (uint64_t)p.T * p.H, 64, HG);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d_bf16(&swamap, p.swa_cache, (uint64_t)D, (uint64_t)a.swa_rows, 64, 1);
  if (e != cudaSuccess) return e;
  if (p.ratio > 0) {
    e = make_tmap_2d_bf16(&mainmap, p.main_cache, (uint64_t)D, (uint64_t)a.main_rows, 64, 1);
    if (e != cudaSuccess) return e;
    e = make_tmap_2d_bf16(&mainmap64, p.main_cache, (uint64_t)D, (uint64_t)a.main_rows, 64, 64);
    if (e != cudaSuccess) return e;
  } else {
    mainmap = swamap;
    mainmap64 = swamap;
  }
  const size_t smem = 1024 + (size_t)Q_BYTES + (size_t)STAGES * STAGE_BYTES + sizeof(Smem);
  static int attr_done = 0;
  if (!attr_done) {
    e = cudaFuncSetAttribute(mla_partial_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done = 1;
  }
  dim3 grid(L.n_chunks, p.T, (p.H / HG) * 2);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;  // the two value halves of a (chunk, token, head group)
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 2;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, mla_partial_tc, qmap, swamap, mainmap, mainmap64, a);
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
