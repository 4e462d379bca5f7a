// Lightning-Indexer scoring and per-query top-k.
//
// "DeepSeek V4 Attention: Code Reading Map", §Phase 2 (indexer stream, item 4: scores between the
// indexer queries and the compressed indexer keys, then the top-k compressed blocks) and
// §Concrete Trace (top-1024 of ~125,000); "vllm.models.deepseek_v41.attention",
// DeepseekV4Indexer.forward (when the candidates fit in top-k, every candidate is selected).
// Score: s[t][j] = sum_h w[t][h] * ReLU(q[t][h] . k_j) in fp32.
//
// Work split: the score kernel gives a CTA one tile of 128 keys of one sequence and scores them
// for all of that sequence's query tokens, so each key row leaves HBM once per step.  Scores go
// to the workspace; the top-k kernel then runs an exact 4-pass 8-bit radix select per token on
// order-preserving uint32 keys and compacts the selection in increasing j.
#include "dsv4_common.cuh"
#include "dsv4_launch.h"
#include "tc_ptx.cuh"
#include "tmap.h"

namespace dsv4 {

static __device__ unsigned int g_flags_ix = 0;

constexpr int IX_TILE = 128;

// n_c of token t, clamped to what the workspace and grid were sized for (max_context); a position
// outside [0, max_context) is flagged.
__device__ __forceinline__ int visible_entries(const dsv4_indexer_topk_params& p, int t) {
  const int pos = p.positions[t];
  if (pos < 0 || pos >= p.max_context) {
    atomicOr(&g_flags_ix, FLAG_PAGE);
    return pos < 0 ? 0 : p.max_context / p.ratio;
  }
  return (pos + 1) / p.ratio;
}

struct IxLayout {
  size_t scores_off, nc_stride;
};

static IxLayout ix_layout(const dsv4_indexer_topk_params& p) {
  IxLayout L;
  const int64_t max_nc = (int64_t)p.max_context / p.ratio;
  L.nc_stride = align_up((size_t)(max_nc > 0 ? max_nc : 1), 64);
  L.scores_off = 0;
  return L;
}

size_t indexer_topk_workspace(const dsv4_indexer_topk_params& p) {
  IxLayout L = ix_layout(p);
  return align_up((size_t)p.T * L.nc_stride * sizeof(float), 256);
}

// ------------------------------------------------------------------------------------------------
// SIMT score kernel (all key dtypes): thread jj of the CTA owns key tile*128 + jj.
// ------------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(IX_TILE) indexer_score_simt(dsv4_indexer_topk_params p, float* scores,
                                                              int nc_stride) {
  extern __shared__ float smem[];
  const int b = blockIdx.y, tile = blockIdx.x, jj = threadIdx.x;
  const int Ih = p.n_heads, d = p.head_dim, qps = p.q_per_seq;
  const int t0 = b * qps;
  const int nc_last = visible_entries(p, t0 + qps - 1);  // largest n_c among the seq's tokens
  const int j0 = tile * IX_TILE;
  if (j0 >= nc_last) return;

  float* q_s = smem;                         // [qps][Ih][d]
  float* w_s = q_s + qps * Ih * d;           // [qps][Ih]
  const int ld = IX_TILE + 1;
  float* kt_s = w_s + qps * Ih;              // [d][IX_TILE + 1] transposed keys

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
        else v = (float)reinterpret_cast<const int8_t*>(row)[e];
      }
      kt_s[e * ld + kk] = v;
    }
    if (lane == 0) kt_s[d * ld + kk] = scale;  // scale row after the d key rows
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
      acc *= kscale;
      s = fmaf(w_s[k * Ih + h], fmaxf(acc, 0.f), s);
    }
    if (j < nc) scores[(int64_t)t * nc_stride + j] = s;
  }
}

// ------------------------------------------------------------------------------------------------
// Tensor-core score kernel (bf16 keys and queries): D[128 keys x N] = K_tile[128 x d] * Q[N x d]^T
// with N = q_per_seq * n_heads (every query head of the sequence), then per key
// s_k = sum_h w[k][h] * ReLU(D[key][k*n_heads + h]).
//
// Persistent CTAs (one per SM), each owning a contiguous range of (sequence, 128-key tile) items.
// Warp 4 streams key tiles with TMA (two 64-row pages x two 64-dim K-blocks, 128-byte swizzle)
// into a ring of stages and the sequence's Q block into its own buffer; one thread of warp 5 issues
// the tcgen05 MMAs (M = 128, K = 16 steps) into one of two TMEM accumulators; warps 0-3 read
// their 32 TMEM lanes each (one key per thread), apply ReLU and the head weights and store the
// scores.  Every wait is bounded; a timeout raises FLAG_TIMEOUT and all roles drain out.
// ------------------------------------------------------------------------------------------------
namespace ixtc {
constexpr int TILE = 128;
constexpr int KB_BYTES = TILE * 128;         // one 64-dim K-block of a key tile (128 rows x 128 B)
constexpr int STAGE_BYTES = 2 * KB_BYTES;    // d <= 128
constexpr int THREADS = 192;
constexpr uint32_t FLAG_TIMEOUT = 4u;

struct Args {
  const int32_t* positions;
  const int32_t* block_table;
  const float* weights;
  float* scores;
  int64_t num_pages;
  int T, B, qps, Ih, d, ratio, max_pages, nc_stride, tiles_max, max_context;
  int N, kblk, stages, tmem_cols;
};

struct Smem {
  uint64_t full[8], empty[8], dfull[2], dempty[2], qfull, qempty, done;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ int seq_entries(const Args& a, int b) {
  const int pos = a.positions[b * a.qps + a.qps - 1];
  if (pos < 0 || pos >= a.max_context) return pos < 0 ? 0 : a.max_context / a.ratio;
  return (pos + 1) / a.ratio;
}

__device__ __forceinline__ int tok_entries(const Args& a, int t) {
  const int pos = a.positions[t];
  if (pos < 0 || pos >= a.max_context) return pos < 0 ? 0 : a.max_context / a.ratio;
  return (pos + 1) / a.ratio;
}

__device__ __forceinline__ int page_of(const Args& a, int b, int lp) {
  if (lp >= a.max_pages) return -1;
  const int pg = a.block_table[(int64_t)b * a.max_pages + lp];
  if (pg < 0 || pg >= a.num_pages) {
    atomicOr(&g_flags_ix, FLAG_PAGE);
    return -1;
  }
  return pg;
}

// next valid item at or after `it` in [it, hi), or hi
__device__ __forceinline__ int next_item(const Args& a, int it, int hi, int& b, int& tile) {
  for (; it < hi; ++it) {
    b = it / a.tiles_max;
    tile = it % a.tiles_max;
    if (tile * TILE < seq_entries(a, b)) return it;
  }
  return hi;
}

__global__ void __launch_bounds__(THREADS, 1)
    indexer_score_tc(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap, Args a) {
  extern __shared__ __align__(1024) uint8_t dsm[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_mem = base;                                      // stages x STAGE_BYTES
  uint8_t* q_mem = base + a.stages * STAGE_BYTES;                 // kblk x N x 128 B
  float* w_s = reinterpret_cast<float*>(q_mem + a.kblk * a.N * 128);  // N floats
  Smem* sm = reinterpret_cast<Smem*>(w_s + 256);
  volatile int* abort = &sm->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = a.B * a.tiles_max;
  const int lo = (int)((int64_t)blockIdx.x * total / gridDim.x);
  const int hi = (int)((int64_t)(blockIdx.x + 1) * total / gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < a.stages; ++s) {
      tc::mbar_init(&sm->full[s], 1);
      tc::mbar_init(&sm->empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sm->dfull[i], 1);
      tc::mbar_init(&sm->dempty[i], 4);
    }
    tc::mbar_init(&sm->qfull, 1);
    tc::mbar_init(&sm->qempty, 1);
    tc::mbar_init(&sm->done, 1);
    sm->abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == 5) {
    tc::tmem_alloc(&sm->tmem_base, a.tmem_cols);
    tc::tmem_relinquish();
    tc::tc_fence_before();
  }
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm->tmem_base;

  if (warp == 4) {
    if (lane == 0) {
      // ---------------- TMA producer
      tc::tma_prefetch_desc(&kmap);
      tc::tma_prefetch_desc(&qmap);
      int stage = 0, cur_b = -1;
      uint32_t phase = 0, qphase = 0;
      int b, tile;
      for (int it = next_item(a, lo, hi, b, tile); it < hi; it = next_item(a, it + 1, hi, b, tile)) {
        if (b != cur_b) {
          if (cur_b >= 0) {
            if (!tc::mbar_wait_bounded(&sm->qempty, qphase, abort)) break;
            qphase ^= 1;
          }
          tc::mbar_arrive_expect_tx(&sm->qfull, a.kblk * a.N * 128);
          for (int kb = 0; kb < a.kblk; ++kb)
            tc::tma_load_2d(q_mem + kb * a.N * 128, &qmap, kb * 64, b * a.qps * a.Ih, &sm->qfull);
          cur_b = b;
        }
        if (!tc::mbar_wait_bounded(&sm->empty[stage], phase ^ 1, abort)) break;
        const int nc = seq_entries(a, b);
        const int j0 = tile * TILE;
        const int pg0 = page_of(a, b, j0 / 64);
        const int pg1 = (j0 + 64 < nc) ? page_of(a, b, j0 / 64 + 1) : -1;
        const uint32_t bytes = (uint32_t)((pg0 >= 0) + (pg1 >= 0)) * a.kblk * (KB_BYTES / 2);
        uint8_t* st = stage_mem + stage * STAGE_BYTES;
        tc::mbar_arrive_expect_tx(&sm->full[stage], bytes);
        for (int kb = 0; kb < a.kblk; ++kb) {
          if (pg0 >= 0) tc::tma_load_2d(st + kb * KB_BYTES, &kmap, kb * 64, pg0 * 64, &sm->full[stage]);
          if (pg1 >= 0) tc::tma_load_2d(st + kb * KB_BYTES + KB_BYTES / 2, &kmap, kb * 64, pg1 * 64, &sm->full[stage]);
        }
        if (++stage == a.stages) {
          stage = 0;
          phase ^= 1;
        }
      }
      // drain: every issued load must land before the CTA may exit
      for (int s = 0; s < a.stages; ++s) {
        // the most recent use of stage s completed phase `ph`; waiting on it returns at once when consumed
        int uses_parity = (s < stage) ? (int)phase : (int)(phase ^ 1);
        tc::mbar_wait_bounded(&sm->full[s], uses_parity, abort, 100000000ull);
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      // ---------------- MMA issuer
      const uint32_t idesc = tc::idesc_bf16_f32(TILE, a.N);
      const uint32_t q_addr = tc::smem_addr(q_mem);
      int stage = 0, acc = 0, cur_b = -1;
      uint32_t phase = 0, aphase = 0, qphase = 0;
      int b, tile;
      for (int it = next_item(a, lo, hi, b, tile); it < hi;) {
        if (b != cur_b) {
          if (!tc::mbar_wait_bounded(&sm->qfull, qphase, abort)) break;
          qphase ^= 1;
          cur_b = b;
        }
        if (!tc::mbar_wait_bounded(&sm->full[stage], phase, abort)) break;
        if (!tc::mbar_wait_bounded(&sm->dempty[acc], aphase ^ 1, abort)) break;
        tc::tc_fence_after();
        const uint32_t a_addr = tc::smem_addr(stage_mem + stage * STAGE_BYTES);
        const uint32_t d_tmem = tmem + (uint32_t)(acc * a.N);
        for (int kb = 0; kb < a.kblk; ++kb) {
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            const uint64_t ad = tc::sdesc_k_sw128(a_addr + kb * KB_BYTES + s * 32);
            const uint64_t bd = tc::sdesc_k_sw128(q_addr + kb * a.N * 128 + s * 32);
            tc::mma_bf16(d_tmem, ad, bd, idesc, (kb | s) != 0);
          }
        }
        tc::mma_commit(&sm->empty[stage]);
        tc::mma_commit(&sm->dfull[acc]);
        int nb, ntile;
        const int nx = next_item(a, it + 1, hi, nb, ntile);
        if (nx >= hi || nb != b) tc::mma_commit(&sm->qempty);
        if (++stage == a.stages) {
          stage = 0;
          phase ^= 1;
        }
        if (++acc == 2) {
          acc = 0;
          aphase ^= 1;
        }
        it = nx;
        b = nb;
        tile = ntile;
      }
      tc::mma_commit(&sm->done);
      tc::mbar_wait_bounded(&sm->done, 0, abort, 100000000ull);
    }
  } else {
    // ---------------- epilogue: warps 0-3, thread = key row (TMEM lane)
    const int row = warp * 32 + lane;
    int acc = 0, cur_b = -1;
    uint32_t aphase = 0;
    int b, tile;
    for (int it = next_item(a, lo, hi, b, tile); it < hi; it = next_item(a, it + 1, hi, b, tile)) {
      if (b != cur_b) {
        asm volatile("bar.sync 1, 128;" ::: "memory");
        for (int x = row; x < a.N; x += 128) w_s[x] = a.weights[(int64_t)b * a.qps * a.Ih + x];
        asm volatile("bar.sync 1, 128;" ::: "memory");
        cur_b = b;
      }
      if (!tc::mbar_wait_bounded(&sm->dfull[acc], aphase, abort)) break;
      tc::tc_fence_after();
      float sk[DSV4_MAX_Q_PER_SEQ] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(acc * a.N);
      for (int c0 = 0; c0 < a.N; c0 += 32) {
        float v[32];
        tc::tmem_ld32(lane_addr + c0, v);
        float part = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) part = fmaf(w_s[c0 + i], fmaxf(v[i], 0.f), part);
        const int k = c0 / a.Ih;
#pragma unroll
        for (int q = 0; q < DSV4_MAX_Q_PER_SEQ; ++q)
          if (q == k) sk[q] += part;
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&sm->dempty[acc]);
      const int j = tile * TILE + row;
#pragma unroll
      for (int q = 0; q < DSV4_MAX_Q_PER_SEQ; ++q) {
        if (q < a.qps) {
          const int t = b * a.qps + q;
          if (j < tok_entries(a, t)) a.scores[(int64_t)t * a.nc_stride + j] = sk[q];
        }
      }
      if (++acc == 2) {
        acc = 0;
        aphase ^= 1;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && sm->abort) atomicOr(&g_flags_ix, FLAG_TIMEOUT);
  if (warp == 5) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, a.tmem_cols);
  }
}

}  // namespace ixtc

static bool use_tc_indexer(const dsv4_indexer_topk_params& p) {
  const int N = p.q_per_seq * p.n_heads;
  return p.k_dtype == DSV4_BF16 && p.q_dtype == DSV4_BF16 && (p.head_dim == 64 || p.head_dim == 128) &&
         p.n_heads % 32 == 0 && N >= 32 && N <= 256 && p.page_size == 64;
}

static cudaError_t launch_indexer_score_tc(const dsv4_indexer_topk_params& p, float* scores, int nc_stride,
                                           cudaStream_t st) {
  using namespace ixtc;
  const int max_nc = p.max_context / p.ratio;
  Args a;
  a.positions = p.positions;
  a.block_table = p.block_table;
  a.weights = p.weights;
  a.scores = scores;
  a.num_pages = p.num_pages;
  a.T = p.T;
  a.B = p.B;
  a.qps = p.q_per_seq;
  a.Ih = p.n_heads;
  a.d = p.head_dim;
  a.ratio = p.ratio;
  a.max_pages = p.max_pages_per_seq;
  a.nc_stride = nc_stride;
  a.tiles_max = (max_nc + TILE - 1) / TILE;
  a.max_context = p.max_context;
  a.N = p.q_per_seq * p.n_heads;
  a.kblk = p.head_dim / 64;
  a.stages = a.N > 128 ? 4 : 5;
  a.tmem_cols = a.N <= 16 ? 32 : (2 * a.N <= 64 ? 64 : (2 * a.N <= 128 ? 128 : (2 * a.N <= 256 ? 256 : 512)));
  CUtensorMap kmap, qmap;
  cudaError_t e = make_tmap_2d_bf16(&kmap, p.k_cache, (uint64_t)p.head_dim, (uint64_t)p.num_pages * 64, 64, 64);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d_bf16(&qmap, p.q, (uint64_t)p.head_dim, (uint64_t)p.T * p.n_heads, 64, (uint32_t)a.N);
  if (e != cudaSuccess) return e;
  const size_t smem = 1024 + (size_t)a.stages * STAGE_BYTES + (size_t)a.kblk * a.N * 128 + 256 * 4 + sizeof(Smem);
  static int attr_done = 0;
  if (!attr_done) {
    e = cudaFuncSetAttribute(indexer_score_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_done = 1;
  }
  const int total = a.B * a.tiles_max;
  int grid = num_sms();
  if (grid > total) grid = total;
  if (grid <= 0) return cudaSuccess;
  indexer_score_tc<<<grid, THREADS, smem, st>>>(kmap, qmap, a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------------
// Top-k: exact radix select, one CTA per token.
// ------------------------------------------------------------------------------------------------
constexpr int TK_THREADS = 1024;

__device__ __forceinline__ uint32_t order_key(float s) {
  uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive prefix of a 0/1 flag over the CTA (thread order); returns the total in *total.
__device__ __forceinline__ int block_excl_scan_flag(bool f, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, f);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) warp_tot[warp] = __popc(bal);
  __syncthreads();
  if (warp == 0) {
    int v = lane < nw ? warp_tot[lane] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    if (lane < nw) warp_tot[lane] = incl - v;  // exclusive warp offsets
    if (lane == 31) warp_tot[32] = incl;
  }
  __syncthreads();
  const int r = warp_tot[warp] + in_warp;
  *total = warp_tot[32];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(TK_THREADS) topk_radix_kernel(dsv4_indexer_topk_params p, const float* scores,
                                                                int nc_stride) {
  const int t = blockIdx.x, tid = threadIdx.x;
  const int K = p.topk;
  const int n = visible_entries(p, t);
  int32_t* out = p.topk_idx + (int64_t)t * K;
  float* out_s = p.topk_score ? p.topk_score + (int64_t)t * K : nullptr;
  const float* s = scores + (int64_t)t * nc_stride;

  if (n <= K) {  // short context: every candidate, in order
    for (int x = tid; x < K; x += TK_THREADS) {
      out[x] = x < n ? x : -1;
      if (out_s) out_s[x] = x < n ? s[x] : -INFINITY;
    }
    return;
  }

  __shared__ unsigned int hist[256];
  __shared__ unsigned int sh_prefix, sh_remaining;
  __shared__ int warp_tot[33];
  uint32_t prefix = 0, mask = 0;
  if (tid == 0) sh_remaining = K;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int x = tid; x < 256; x += TK_THREADS) hist[x] = 0;
    __syncthreads();
    for (int j = tid; j < n; j += TK_THREADS) {
      const uint32_t u = order_key(s[j]);
      if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      unsigned int rem = sh_remaining, cum = 0;
      int dsel = 0;
      for (int dd = 255; dd >= 0; --dd) {
        if (cum + hist[dd] >= rem) {
          dsel = dd;
          break;
        }
        cum += hist[dd];
      }
      sh_remaining = rem - cum;
      sh_prefix = prefix | ((uint32_t)dsel << shift);
    }
    __syncthreads();
    prefix = sh_prefix;
    mask |= 255u << shift;
  }
  const uint32_t kth = prefix;             // key of the k-th largest score
  const int need_eq = (int)sh_remaining;   // how many entries equal to it are taken (lowest j first)

  int base_out = 0, base_eq = 0;
  for (int j0 = 0; j0 < n; j0 += TK_THREADS) {
    const int j = j0 + tid;
    uint32_t u = 0;
    if (j < n) u = order_key(s[j]);
    const bool gt = j < n && u > kth;
    const bool eq = j < n && u == kth;
    int eq_tot;
    const int eq_rank = block_excl_scan_flag(eq, warp_tot, &eq_tot);
    const bool take = gt || (eq && base_eq + eq_rank < need_eq);
    int take_tot;
    const int pos = block_excl_scan_flag(take, warp_tot, &take_tot);
    if (take) {
      out[base_out + pos] = j;
      if (out_s) out_s[base_out + pos] = s[j];
    }
    base_out += take_tot;
    base_eq += eq_tot;
  }
  for (int x = base_out + tid; x < K; x += TK_THREADS) {  // cannot happen when n > K; kept for safety
    out[x] = -1;
    if (out_s) out_s[x] = -INFINITY;
  }
}

cudaError_t launch_indexer_topk(const dsv4_indexer_topk_params& p, cudaStream_t st) {
  if (p.T == 0) return cudaSuccess;
  IxLayout L = ix_layout(p);
  float* scores = reinterpret_cast<float*>(reinterpret_cast<char*>(p.workspace) + L.scores_off);
  const int max_nc = p.max_context / p.ratio;
  if (max_nc > 0 && use_tc_indexer(p)) {
    cudaError_t e = launch_indexer_score_tc(p, scores, (int)L.nc_stride, st);
    if (e != cudaSuccess) return e;
  } else if (max_nc > 0) {
    const int tiles = (max_nc + IX_TILE - 1) / IX_TILE;
    const size_t smem = sizeof(float) * ((size_t)p.q_per_seq * p.n_heads * p.head_dim +
                                         (size_t)p.q_per_seq * p.n_heads + (size_t)(p.head_dim + 1) * (IX_TILE + 1));
    cudaError_t e = cudaFuncSetAttribute(indexer_score_simt, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    indexer_score_simt<<<dim3(tiles, p.B), IX_TILE, smem, st>>>(p, scores, (int)L.nc_stride);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  topk_radix_kernel<<<p.T, TK_THREADS, 0, st>>>(p, scores, (int)L.nc_stride);
  return cudaGetLastError();
}

cudaError_t read_flags_indexer(uint32_t* f) {
  unsigned int v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_flags_ix, sizeof(v));
  if (e != cudaSuccess) return e;
  *f |= v;
  return cudaMemcpyToSymbol(g_flags_ix, &z, sizeof(z));
}

}  // namespace dsv4
