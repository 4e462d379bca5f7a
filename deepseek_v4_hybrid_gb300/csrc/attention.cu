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
  int n_cmp = 0;
  if (p.ratio > 0) n_cmp = p.topk_idx ? p.topk : p.max_context / p.ratio;
  return n_swa + n_cmp;
}

static bool use_tc_attention(const dsv4_sparse_mla_decode_params& p);
constexpr int TC_CHUNK = 256;   // rows per CTA of the tensor-core kernel

static AtLayout at_layout(const dsv4_sparse_mla_decode_params& p) {
  AtLayout L;
  L.chunk_rows = use_tc_attention(p) ? TC_CHUNK : AT_CH;
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
// Tensor-core partial kernel (bf16 caches and queries).  CTA = (chunk of 256 rows, token, 64-head
// group x value half).  Heads are the MMA M dimension (M = 128, lanes 64..127 unused), rows the
// N dimension of S = Q K^T (K = 576 in 9 K-blocks of 64 dims) and the K dimension of
// O[:, half] += P V[:, half] (N = 256 value dims).
//
// Warps 2 and 3 gather 64-row tiles with 16-byte cp.async copies written straight into the 128-byte
// swizzled K-major layout the MMA reads (one copy instruction = 4 rows x 128 bytes), so any row
// order (window positions, top-k indices, dense runs) works; a masked row is zero-filled.  Q comes
// by TMA.  Lane 0 of warp 4 issues the MMAs; S goes to one of two TMEM buffers, P (bf16) is written back
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
constexpr int THREADS = 160;  // warps 0-1 softmax, 2-3 producers, 4 MMA
constexpr uint32_t COL_O = 0, COL_S = 256, COL_P = 384;  // S: 2 x 64 columns, P: 2 x 32 columns
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_LOG2 = 8.0f;
constexpr uint32_t FLAG_TIMEOUT = 4u;

struct Args {
  dsv4_sparse_mla_decode_params p;
  float* o_part;
  float2* ml_part;
  int n_chunks;
  int swa_rows, main_rows;  // rows of the two tensor maps (a masked row loads from this index)
  float c_log2;             // softmax_scale * log2(e)
};

struct Smem {
  uint64_t full[STAGES], empty[STAGES], sfull[2], pfull[2], pvdone[2], qfull, odone;
  uint64_t mask[STAGES];
  uint32_t tmem_base;
  int abort;
};

// TMA row of entry r of token t's row list: (which map, row index); masked rows get the
// out-of-range row of the map.
__device__ __forceinline__ void row_source(const Args& a, int t, int b, int pos, int n_swa, int nc, int n_rows, int r,
                                           int& use_main, int& y, bool& valid) {
  const dsv4_sparse_mla_decode_params& p = a.p;
  use_main = 0;
  y = a.swa_rows;
  valid = false;
  if (r >= n_rows) return;
  if (r < n_swa) {
    const int q = pos - n_swa + 1 + r;
    const int lp = q / p.page_size;
    const int page = lp < p.swa_max_pages ? p.swa_block_table[(int64_t)b * p.swa_max_pages + lp] : -1;
    if (page < 0 || page >= p.swa_num_pages) {
      atomicOr(&g_flags_at, FLAG_PAGE);
      return;
    }
    y = page * p.page_size + q % p.page_size;
    valid = true;
    return;
  }
  use_main = 1;
  y = a.main_rows;
  const int i = r - n_swa;
  int j = i;
  if (p.topk_idx != nullptr) {
    j = p.topk_idx[(int64_t)t * p.topk + i];
    if (j < 0) return;
    if (j >= nc) {
      atomicOr(&g_flags_at, FLAG_TOPK);
      return;
    }
  }
  const int lp = j / p.page_size;
  const int page = lp < p.main_max_pages ? p.main_block_table[(int64_t)b * p.main_max_pages + lp] : -1;
  if (page < 0 || page >= p.main_num_pages) {
    atomicOr(&g_flags_at, FLAG_PAGE);
    return;
  }
  y = page * p.page_size + j % p.page_size;
  valid = true;
}

__global__ void __launch_bounds__(THREADS, 1)
    mla_partial_tc(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap swamap,
                   const __grid_constant__ CUtensorMap mainmap, Args a) {
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
  const int n_rows = n_swa + n_cmp;
  const int r0 = chunk * TC_CHUNK;
  const int rows = min(TC_CHUNK, n_rows - r0);
  const int64_t part = ((int64_t)t * a.n_chunks + chunk) * p.H + hg * HG;
  if (rows <= 0) {  // block-uniform: an empty chunk contributes nothing
    if (dh == 0 && threadIdx.x < HG) a.ml_part[part + threadIdx.x] = make_float2(-INFINITY, 0.f);
    return;
  }
  const int ntiles = (rows + TILE - 1) / TILE;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&sm->full[s], 32);  // every producer lane arrives once its copies have landed
      tc::mbar_init(&sm->empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sm->sfull[i], 1);
      tc::mbar_init(&sm->pfull[i], 2);
      tc::mbar_init(&sm->pvdone[i], 1);
    }
    tc::mbar_init(&sm->qfull, 1);
    tc::mbar_init(&sm->odone, 1);
    sm->abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == 4) {
    tc::tmem_alloc(&sm->tmem_base, TMEM_COLS);
    tc::tmem_relinquish();
    tc::tc_fence_before();
  }
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm->tmem_base;

  if (warp == 2 || warp == 3) {
    // ---------------- producers: warp 2 loads Q by TMA and the even tiles, warp 3 the odd tiles
    // (tile i always uses stage i % 2), each tile by 16-byte cp.async copies; a warp publishes its
    // tile as soon as the copies have landed, so no tile's issue waits on another's publication.
    const int wp = warp - 2;
    if (wp == 0 && lane == 0) {
      tc::tma_prefetch_desc(&qmap);
      tc::mbar_arrive_expect_tx(&sm->qfull, Q_BYTES);
      for (int kb = 0; kb < NKB; ++kb)
        tc::tma_load_2d(q_mem + kb * HG * 128, &qmap, kb * 64, t * p.H + hg * HG, &sm->qfull);
    }
    const uint8_t* swa_base = reinterpret_cast<const uint8_t*>(p.swa_cache);
    const uint8_t* main_base = p.ratio > 0 ? reinterpret_cast<const uint8_t*>(p.main_cache) : swa_base;
    // lane l owns rows l and l + 32 of a tile; source row pointers (nullptr = masked row)
    auto row_ptr = [&](int r) -> const uint8_t* {
      int um, y;
      bool v;
      row_source(a, t, b, pos, n_swa, nc, n_rows, r, um, y, v);
      if (!v || r >= r0 + rows) return nullptr;
      return (um ? main_base : swa_base) + (int64_t)y * (D * 2);
    };
    const int sub = lane >> 3, chunk16 = lane & 7;  // a copy instruction covers 4 rows x 128 bytes
    const uint8_t* ptr0 = nullptr;
    const uint8_t* ptr1 = nullptr;
    if (wp < ntiles) {
      ptr0 = row_ptr(r0 + wp * TILE + lane);
      ptr1 = row_ptr(r0 + wp * TILE + lane + 32);
    }
    for (int i = wp; i < ntiles; i += STAGES) {
      const int stage = i % STAGES;
      int ok = 1;
      if (lane == 0) ok = tc::mbar_wait_bounded(&sm->empty[stage], ((i / STAGES) & 1) ^ 1, abort);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const unsigned b0 = __ballot_sync(0xffffffffu, ptr0 != nullptr);
      const unsigned b1 = __ballot_sync(0xffffffffu, ptr1 != nullptr);
      if (lane == 0) sm->mask[stage] = (uint64_t)b0 | ((uint64_t)b1 << 32);
      uint8_t* st = stage_mem + stage * STAGE_BYTES;
#pragma unroll 4
      for (int rg = 0; rg < TILE / 4; ++rg) {
        const int row = rg * 4 + sub;
        const uint8_t* lo = reinterpret_cast<const uint8_t*>(__shfl_sync(0xffffffffu, (unsigned long long)ptr0, row & 31));
        const uint8_t* hi = reinterpret_cast<const uint8_t*>(__shfl_sync(0xffffffffu, (unsigned long long)ptr1, row & 31));
        const uint8_t* src = row < 32 ? lo : hi;
        const uint32_t nbytes = src != nullptr ? 16u : 0u;
        if (src == nullptr) src = swa_base;  // any valid address; nothing is read
        uint8_t* dst = st + row * 128 + ((chunk16 ^ (row & 7)) << 4);
#pragma unroll
        for (int kb = 0; kb < NKB; ++kb)
          tc::cp_async16(dst + kb * KB_BYTES, src + (nbytes ? kb * 128 + chunk16 * 16 : 0), nbytes);
      }
      tc::cp_async_commit();
      if (i + STAGES < ntiles) {  // look up this warp's next tile while the copies are in flight
        ptr0 = row_ptr(r0 + (i + STAGES) * TILE + lane);
        ptr1 = row_ptr(r0 + (i + STAGES) * TILE + lane + 32);
      }
      tc::cp_async_wait<0>();
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&sm->full[stage]);
    }
    tc::cp_async_wait<0>();
    if (wp == 0 && lane == 0) tc::mbar_wait_bounded(&sm->qfull, 0, abort, 100000000ull);  // Q landed before exit
  } else if (warp == 4) {
    if (lane == 0) {
      // ---------------- MMA issuer
      const uint32_t idesc_s = tc::idesc_bf16_f32(128, TILE);
      const uint32_t idesc_o = tc::idesc_bf16_f32_bmn(128, DVH);
      const uint32_t q_addr = tc::smem_addr(q_mem);
      bool ok = tc::mbar_wait_bounded(&sm->qfull, 0, abort);
      auto pv = [&](int j) -> bool {
        if (!tc::mbar_wait_bounded(&sm->pfull[j & 1], (j >> 1) & 1, abort)) return false;
        tc::tc_fence_after();
        const uint32_t v_addr = tc::smem_addr(stage_mem + (j % STAGES) * STAGE_BYTES + (4 * dh) * KB_BYTES);
#pragma unroll
        for (int s = 0; s < TILE / 16; ++s) {
          const uint64_t bd = tc::sdesc_mn_sw128(v_addr + s * 2048, KB_BYTES, 1024);
          tc::mma_bf16_ts(tmem + COL_O, tmem + COL_P + (j & 1) * 32 + s * 8, bd, idesc_o, (j > 0 || s > 0) ? 1u : 0u);
        }
        tc::mma_commit(&sm->empty[j % STAGES]);
        tc::mma_commit(&sm->pvdone[j & 1]);
        return true;
      };
      for (int i = 0; ok && i < ntiles; ++i) {
        const int stage = i % STAGES;
        if (!tc::mbar_wait_bounded(&sm->full[stage], (i / STAGES) & 1, abort)) break;
        tc::tc_fence_after();
        const uint32_t k_addr = tc::smem_addr(stage_mem + stage * STAGE_BYTES);
        for (int kb = 0; kb < NKB; ++kb) {
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const uint64_t ad = tc::sdesc_k_sw128(q_addr + kb * HG * 128 + s * 32);
            const uint64_t bd = tc::sdesc_k_sw128(k_addr + kb * KB_BYTES + s * 32);
            tc::mma_bf16(tmem + COL_S + (i & 1) * TILE, ad, bd, idesc_s, (kb | s) != 0);
          }
        }
        tc::mma_commit(&sm->sfull[i & 1]);
        if (i >= 1 && !pv(i - 1)) {
          ok = false;
          break;
        }
      }
      if (ok && !*abort) pv(ntiles - 1);
      tc::mma_commit(&sm->odone);
    }
  } else {
    // ---------------- softmax + epilogue: warps 0-1, thread = head (TMEM lane)
    const int h = warp * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
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
      uint32_t r[64];
      tc::tmem_ld32_nowait(lane_base + COL_S + (i & 1) * TILE, r);
      tc::tmem_ld32_nowait(lane_base + COL_S + (i & 1) * TILE + 32, r + 32);
      tc::tmem_wait_ld_regs<64>(r);
      const uint64_t mask = sm->mask[i % STAGES];
      float z[64];
      float mt = -INFINITY;
#pragma unroll
      for (int k = 0; k < 64; ++k) {
        z[k] = ((mask >> k) & 1ull) ? __uint_as_float(r[k]) * a.c_log2 : -INFINITY;
        mt = fmaxf(mt, z[k]);
      }
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
        const float f = exp2f(m_ref - m_new);
        l *= f;
        for (int c = 0; c < DVH; c += 32) {
          uint32_t o[32];
          tc::tmem_ld32_nowait(lane_base + COL_O + c, o);
          tc::tmem_wait_ld_regs<32>(o);
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
          tc::tmem_st32(lane_base + COL_O + c, o);
        }
        tc::tmem_wait_st();
        m_ref = m_new;
      }
      uint32_t pk[32];
      float ls = 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float e0 = (m_ref == -INFINITY) ? 0.f : exp2f(z[2 * k] - m_ref);
        const float e1 = (m_ref == -INFINITY) ? 0.f : exp2f(z[2 * k + 1] - m_ref);
        ls += e0 + e1;
        pk[k] = float2_to_bf16x2_bits(e0, e1);
      }
      l += ls;
      // P buffer (i & 1) was last read by the P V product of tile i - 2
      if (i >= 2 && !tc::mbar_wait_bounded(&sm->pvdone[i & 1], ((i - 2) >> 1) & 1, abort)) {
        ok = false;
        break;
      }
      tc::tmem_st32(lane_base + COL_P + (i & 1) * 32, pk);
      tc::tmem_wait_st();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm->pfull[i & 1]);
    }
    if (ok && tc::mbar_wait_bounded(&sm->odone, 0, abort)) {
      tc::tc_fence_after();
      float* dst = a.o_part + (part + h) * DV + dh * DVH;
      for (int c = 0; c < DVH; c += 32) {
        uint32_t o[32];
        tc::tmem_ld32_nowait(lane_base + COL_O + c, o);
        tc::tmem_wait_ld_regs<32>(o);
#pragma unroll
        for (int k = 0; k < 32; k += 4)
          *reinterpret_cast<float4*>(dst + c + k) = make_float4(__uint_as_float(o[k]), __uint_as_float(o[k + 1]),
                                                                 __uint_as_float(o[k + 2]), __uint_as_float(o[k + 3]));
      }
      if (dh == 0) a.ml_part[part + h] = make_float2(m_ref * 0.69314718055994531f, l);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && sm->abort) atomicOr(&g_flags_at, FLAG_TIMEOUT);
  if (warp == 4) {
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
  a.swa_rows = (int)(p.swa_num_pages * p.page_size);
  a.main_rows = p.ratio > 0 ? (int)(p.main_num_pages * p.page_size) : a.swa_rows;
  a.c_log2 = p.softmax_scale * 1.4426950408889634f;
  CUtensorMap qmap, swamap, mainmap;
  cudaError_t e = make_tmap_2d_bf16(&qmap, p.q, (uint64_t)D, (uint64_t)p.T * p.H, 64, HG);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d_bf16(&swamap, p.swa_cache, (uint64_t)D, (uint64_t)a.swa_rows, 64, 1);
  if (e != cudaSuccess) return e;
  if (p.ratio > 0) {
    e = make_tmap_2d_bf16(&mainmap, p.main_cache, (uint64_t)D, (uint64_t)a.main_rows, 64, 1);
    if (e != cudaSuccess) return e;
  } else {
    mainmap = swamap;
  }
  const size_t smem = 1024 + (size_t)Q_BYTES + (size_t)STAGES * STAGE_BYTES + sizeof(Smem);
  static int attr_done = 0;
  if (!attr_done) {
    e = cudaFuncSetAttribute(mla_partial_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done = 1;
  }
  dim3 grid(L.n_chunks, p.T, (p.H / HG) * 2);
  mla_partial_tc<<<grid, THREADS, smem, st>>>(qmap, swamap, mainmap, a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------------
// Merge of the chunk partials (m_c, l_c, unnormalised O_c) with the sink: CTA per (token, head).
// ------------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(MERGE_THREADS) mla_merge(dsv4_sparse_mla_decode_params p, const float* o_part,
                                                           const float2* ml_part, int n_chunks) {
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
    mla_partial_simt<<<dim3(L.n_chunks, p.T, (p.H + AT_HG - 1) / AT_HG), AT_THREADS, smem, st>>>(p, o_part, ml_part,
                                                                                                   L.n_chunks);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  mla_merge<<<dim3(p.T, p.H), MERGE_THREADS, 0, st>>>(p, o_part, ml_part, L.n_chunks);
  return cudaGetLastError();
}

cudaError_t read_flags_attention(uint32_t* f) {
  unsigned int v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_flags_at, sizeof(v));
  if (e != cudaSuccess) return e;
  *f |= v;
  return cudaMemcpyToSymbol(g_flags_at, &z, sizeof(z));
}

}  // namespace dsv4
