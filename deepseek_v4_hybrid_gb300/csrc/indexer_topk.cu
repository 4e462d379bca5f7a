// Lightning-Indexer scoring and per-query top-k.
//
// "DeepSeek V4 Attention: Code Reading Map", §Phase 2 (indexer stream, item 4: scores between the
// indexer queries and the compressed indexer keys, then the top-k compressed blocks) and
// §Concrete Trace (top-1024 of ~125,000); "vllm.models.deepseek_v41.attention",
// DeepseekV4Indexer.forward (when the candidates fit in top-k, every candidate is selected).
// Score: s[t][j] = sum_h w[t][h] * ReLU(q[t][h] . k_j) in fp32.
//
// Kernels of one call:
//  1. score: a CTA works on 128-key tiles of one sequence for all of that sequence's query tokens,
//     so each key row leaves HBM once per step.  bf16 keys run on the tensor cores (tcgen05 MMA,
//     TMA-fed); fp32 and int8 keys on the CUDA cores.  Besides the score row of each token, the
//     epilogue builds a 4096-bin histogram of the scores' top 12 order-preserving key bits.
//  2. collect: from the histogram, the bin B* holding the k-th best score; every entry above B*
//     is selected outright, every entry inside B* becomes a candidate.
//  3. final: exact choice among the candidates (larger score first, then smaller j), then the
//     selection sorted by j.
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
  size_t scores_off, hist_off, cnt_off, certain_off, maybe_off, total;
};

static IxLayout ix_layout(const dsv4_indexer_topk_params& p) {
  IxLayout L;
  const int64_t max_nc = (int64_t)p.max_context / p.ratio;
  L.nc_stride = align_up((size_t)(max_nc > 0 ? max_nc : 1), 64);
  L.scores_off = 0;
  L.hist_off = align_up(L.scores_off + (size_t)p.T * L.nc_stride * sizeof(float), 256);
  L.cnt_off = L.hist_off + (size_t)p.T * HIST_BINS * sizeof(uint32_t);  // zeroed together with hist
  L.certain_off = align_up(L.cnt_off + (size_t)p.T * 3 * sizeof(uint32_t), 256);
  L.maybe_off = align_up(L.certain_off + (size_t)p.T * p.topk * sizeof(int32_t), 256);
  L.total = align_up(L.maybe_off + (size_t)p.T * L.nc_stride * sizeof(uint64_t), 256);
  return L;
}

size_t indexer_topk_workspace(const dsv4_indexer_topk_params& p) { return ix_layout(p).total; }

struct TopkBufs {
  float* scores;
  uint32_t* hist;      // [T][HIST_BINS]
  uint32_t* cnt;       // [T][3]: selected-outright count, candidate count, finished collect CTAs
  int32_t* certain;    // [T][topk]
  uint64_t* maybe;     // [T][nc_stride] candidates: (low 20 key bits << 32) | ~j
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
    const bool on = j < nc;
    if (on) bufs.scores[(int64_t)t * bufs.nc_stride + j] = s;
    hist_add_warp(bufs.hist + (int64_t)t * HIST_BINS, order_key(s) >> HIST_SHIFT, on);
  }
}

// ------------------------------------------------------------------------------------------------
// Tensor-core score kernel (bf16 keys and queries): D[128 keys x N] = K_tile[128 x d] * Q[N x d]^T
// with N = q_per_seq * n_heads (every query head of the sequence), then per key
// s_k = sum_h w[k][h] * ReLU(D[key][k*n_heads + h]).
//
// Persistent CTAs (one per SM), each owning a contiguous range of (sequence, 128-key tile) items.
// Warp 4 streams key tiles with TMA (two 64-row pages x d/64 K-blocks of 128 B, 128-byte swizzle)
// into a ring of stages, and each sequence's Q block into one of two Q slots; its 32 lanes look up
// the block-table pages of 32 items at a time.  One thread of warp 5 issues the tcgen05 MMAs
// (M = 128, K = 16 steps) into one of two TMEM accumulators; warps 0-3 read their 32 TMEM lanes
// each (one key per thread), apply ReLU and the head weights, store the scores and count them
// into a shared-memory histogram that is added to the global one when the sequence changes.
// Every wait is bounded; a timeout raises FLAG_TIMEOUT and all roles drain out.
// ------------------------------------------------------------------------------------------------
namespace ixtc {
constexpr int TILE = 128;
constexpr int KB_BYTES = TILE * 128;         // one 64-dim K-block of a key tile (128 rows x 128 B)
constexpr int THREADS = 192;
constexpr int MAX_STAGES = 8;

struct Args {
  const int32_t* positions;
  const int32_t* block_table;
  const float* weights;
  TopkBufs bufs;
  int64_t num_pages;
  int T, B, qps, Ih, d, ratio, max_pages, tiles_max, max_context;
  int N, kblk, stages, tmem_cols, nacc;
};

struct Smem {
  uint64_t full[MAX_STAGES], empty[MAX_STAGES], dfull[4], dempty[4], qfull[2], qempty[2], done, ebar;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ int seq_entries(const Args& a, int b) {
  return visible_entries(a.positions, b * a.qps + a.qps - 1, a.max_context, a.ratio);
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

// Walks the valid (sequence, tile) items of the flat range [lo, hi) in order without divisions.
struct ItemIter {
  int it, hi, b, tile, nc;
  __device__ __forceinline__ void init(const Args& a, int lo, int hi_) {
    it = lo;
    hi = hi_;
    b = lo / a.tiles_max;
    tile = lo % a.tiles_max;
    nc = it < hi ? seq_entries(a, b) : 0;
    skip(a);
  }
  // moves past tiles beyond the end of the current sequence
  __device__ __forceinline__ void skip(const Args& a) {
    while (it < hi && tile * TILE >= nc) {
      it += a.tiles_max - tile;
      ++b;
      tile = 0;
      if (it < hi) nc = seq_entries(a, b);
    }
  }
  __device__ __forceinline__ void next(const Args& a) {
    ++it;
    if (++tile == a.tiles_max) {
      ++b;
      tile = 0;
      if (it < hi) nc = seq_entries(a, b);
    }
    skip(a);
  }
  __device__ __forceinline__ bool valid() const { return it < hi; }
};

// Adds the shared histogram of sequence b (if any) to the global one and clears it (the four
// epilogue warps, with bounded group barriers before and after).
__device__ __forceinline__ bool flush_hist(const Args& a, uint32_t* hist_s, int b, int row, uint64_t* ebar,
                                           uint32_t* ephase, volatile int* abort) {
  if (!tc::group_sync(ebar, ephase, abort)) return false;
  if (b >= 0) {
    for (int x = row; x < a.qps * HIST_BINS; x += 128) {
      const uint32_t v = hist_s[x];
      if (v) {
        atomicAdd(&a.bufs.hist[(int64_t)(b * a.qps + x / HIST_BINS) * HIST_BINS + (x % HIST_BINS)], v);
        hist_s[x] = 0;
      }
    }
  }
  return tc::group_sync(ebar, ephase, abort);
}

__global__ void __launch_bounds__(THREADS, 1)
    indexer_score_tc(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap, Args a) {
  extern __shared__ __align__(1024) uint8_t dsm[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm) + 1023) & ~uintptr_t(1023));
  const int q_bytes = a.kblk * a.N * 128;
  const int stage_bytes = a.kblk * KB_BYTES;
  uint8_t* stage_mem = base;                                               // stages x stage_bytes
  uint8_t* q_mem = base + a.stages * stage_bytes;                          // 2 slots x q_bytes
  float* w_s = reinterpret_cast<float*>(q_mem + 2 * q_bytes);              // 256 floats
  uint32_t* hist_s = reinterpret_cast<uint32_t*>(w_s + 256);               // qps x HIST_BINS
  Smem* sm = reinterpret_cast<Smem*>(hist_s + a.qps * HIST_BINS);
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
    for (int i = 0; i < 4; ++i) {
      tc::mbar_init(&sm->dfull[i], 1);
      tc::mbar_init(&sm->dempty[i], 4);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&sm->qfull[i], 1);
      tc::mbar_init(&sm->qempty[i], 1);
    }
    tc::mbar_init(&sm->done, 1);
    tc::mbar_init(&sm->ebar, 4);
    sm->abort = 0;
    tc::fence_barrier_init();
  }
  for (int x = threadIdx.x; x < a.qps * HIST_BINS; x += THREADS) hist_s[x] = 0;
  if (warp == 5) {
    tc::tmem_alloc(&sm->tmem_base, a.tmem_cols);
    tc::tmem_relinquish();
    tc::tc_fence_before();
  }
  pdl_launch_dependents();
  pdl_wait();  // the prologue above overlaps the previous kernel
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = sm->tmem_base;

  if (warp == 4) {
    // ---------------- TMA producer (lane 0 issues; all lanes look up pages 32 items at a time)
    if (lane == 0) {
      tc::tma_prefetch_desc(&kmap);
      tc::tma_prefetch_desc(&qmap);
    }
    int stage = 0, cur_b = -1, qn = 0;
    uint32_t phase = 0;
    bool stop = false;
    for (int base_it = lo; base_it < hi && !stop; base_it += 32) {
      const int it = base_it + lane;
      int vb = -1, pg0 = -1, pg1 = -1;
      if (it < hi) {
        const int b = it / a.tiles_max, tile = it % a.tiles_max;
        const int nc = seq_entries(a, b);
        const int j0 = tile * TILE;
        if (j0 < nc) {
          vb = b;
          pg0 = page_of(a, b, j0 / 64);
          pg1 = (j0 + 64 < nc) ? page_of(a, b, j0 / 64 + 1) : -1;
        }
      }
      for (int i = 0; i < 32; ++i) {
        const int b = __shfl_sync(0xffffffffu, vb, i);
        const int p0 = __shfl_sync(0xffffffffu, pg0, i);
        const int p1 = __shfl_sync(0xffffffffu, pg1, i);
        if (b < 0) continue;
        int ok = 1;
        if (lane == 0) {
          if (b != cur_b) {
            const int slot = qn & 1;
            ok = tc::mbar_wait_bounded(&sm->qempty[slot], ((qn >> 1) & 1) ^ 1, abort);
            if (ok) {
              tc::mbar_arrive_expect_tx(&sm->qfull[slot], q_bytes);
              for (int kb = 0; kb < a.kblk; ++kb)
                tc::tma_load_2d(q_mem + slot * q_bytes + kb * a.N * 128, &qmap, kb * 64, b * a.qps * a.Ih,
                                &sm->qfull[slot]);
              ++qn;
              cur_b = b;
            }
          }
          if (ok) ok = tc::mbar_wait_bounded(&sm->empty[stage], phase ^ 1, abort);
          if (ok) {
            const uint32_t bytes = (uint32_t)((p0 >= 0) + (p1 >= 0)) * a.kblk * (KB_BYTES / 2);
            uint8_t* st = stage_mem + stage * stage_bytes;
            tc::mbar_arrive_expect_tx(&sm->full[stage], bytes);
            for (int kb = 0; kb < a.kblk; ++kb) {
              if (p0 >= 0) tc::tma_load_2d(st + kb * KB_BYTES, &kmap, kb * 64, p0 * 64, &sm->full[stage]);
              if (p1 >= 0)
                tc::tma_load_2d(st + kb * KB_BYTES + KB_BYTES / 2, &kmap, kb * 64, p1 * 64, &sm->full[stage]);
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
    }
    if (lane == 0) {
      // drain: every issued load must land before the CTA may exit (a completed phase returns at once)
      for (int s = 0; s < a.stages; ++s) {
        const int parity = (s < stage) ? (int)phase : (int)(phase ^ 1);
        tc::mbar_wait_bounded(&sm->full[s], parity, abort, 100000000ull);
      }
      for (int slot = 0; slot < 2; ++slot) {
        const int last = (qn - 1 - slot) >= 0 ? (qn - 1) - ((qn - 1 - slot) & 1) : -1;  // last load into slot
        if (last >= 0) tc::mbar_wait_bounded(&sm->qfull[slot], (last >> 1) & 1, abort, 100000000ull);
      }
    }
  } else if (warp == 5) {
    if (lane == 0) {
      // ---------------- MMA issuer
      const uint32_t idesc = tc::idesc_bf16_f32(TILE, a.N);
      int stage = 0, acc = 0, cur_b = -1, qn = 0, slot = 0;
      uint32_t phase = 0, aphase = 0;
      ItemIter cur;
      cur.init(a, lo, hi);
      while (cur.valid()) {
        if (cur.b != cur_b) {
          slot = qn & 1;
          if (!tc::mbar_wait_bounded(&sm->qfull[slot], (qn >> 1) & 1, abort)) break;
          ++qn;
          cur_b = cur.b;
        }
        if (!tc::mbar_wait_bounded(&sm->full[stage], phase, abort)) break;
        if (!tc::mbar_wait_bounded(&sm->dempty[acc], aphase ^ 1, abort)) break;
        tc::tc_fence_after();
        const uint32_t a_addr = tc::smem_addr(stage_mem + stage * stage_bytes);
        const uint32_t q_addr = tc::smem_addr(q_mem + slot * q_bytes);
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
  } else {
    // ---------------- epilogue: warps 0-3, thread = key row (TMEM lane)
    const int row = warp * 32 + lane;
    int acc = 0, cur_b = -1;
    uint32_t aphase = 0, ephase = 0;
    int nc_tok[DSV4_MAX_Q_PER_SEQ] = {0, 0, 0, 0};
    ItemIter cur;
    cur.init(a, lo, hi);
    for (; cur.valid(); cur.next(a)) {
      const int b = cur.b;
      if (b != cur_b) {
        if (!flush_hist(a, hist_s, cur_b, row, &sm->ebar, &ephase, abort)) break;
        for (int x = row; x < a.N; x += 128) w_s[x] = a.weights[(int64_t)b * a.qps * a.Ih + x];
#pragma unroll
        for (int q = 0; q < DSV4_MAX_Q_PER_SEQ; ++q)
          nc_tok[q] = q < a.qps ? visible_entries(a.positions, b * a.qps + q, a.max_context, a.ratio) : 0;
        if (!tc::group_sync(&sm->ebar, &ephase, abort)) break;
        cur_b = b;
      }
      if (!tc::mbar_wait_bounded(&sm->dfull[acc], aphase, abort)) break;
      tc::tc_fence_after();
      float sk[DSV4_MAX_Q_PER_SEQ] = {0.f, 0.f, 0.f, 0.f};
      const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(acc * a.N);
      for (int c0 = 0; c0 < a.N; c0 += 64) {
        uint32_t r[64];
        tc::tmem_ld32_nowait(lane_addr + c0, r);
        tc::tmem_ld32_nowait(lane_addr + c0 + 32, r + 32);
        tc::tmem_wait_ld_regs<64>(r);
        const float4* w4 = reinterpret_cast<const float4*>(w_s + c0);
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
          for (int i = 0; i < 32; ++i) h0 = fmaf(w_s[c0 + i], fmaxf(__uint_as_float(r[i]), 0.f), h0);
#pragma unroll
          for (int i = 32; i < 64; ++i) h1 = fmaf(w_s[c0 + i], fmaxf(__uint_as_float(r[i]), 0.f), h1);
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
#pragma unroll
      for (int q = 0; q < DSV4_MAX_Q_PER_SEQ; ++q) {
        if (q < a.qps) {
          const int t = b * a.qps + q;
          const bool on = j < nc_tok[q];
          if (on) a.bufs.scores[(int64_t)t * a.bufs.nc_stride + j] = sk[q];
          hist_add_warp(hist_s + q * HIST_BINS, order_key(sk[q]) >> HIST_SHIFT, on);
        }
      }
      if (++acc == a.nacc) {
        acc = 0;
        aphase ^= 1;
      }
    }
    flush_hist(a, hist_s, cur_b, row, &sm->ebar, &ephase, abort);
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
         p.n_heads % 32 == 0 && N >= 64 && N <= 128 && N % 64 == 0 && p.page_size == 64;
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
  a.T = p.T;
  a.B = p.B;
  a.qps = p.q_per_seq;
  a.Ih = p.n_heads;
  a.d = p.head_dim;
  a.ratio = p.ratio;
  a.max_pages = p.max_pages_per_seq;
  a.tiles_max = (max_nc + TILE - 1) / TILE;
  a.max_context = p.max_context;
  a.N = p.q_per_seq * p.n_heads;
  a.kblk = p.head_dim / 64;
  a.nacc = 4 * a.N <= 512 ? 4 : 2;  // TMEM accumulators (512 columns available)
  a.tmem_cols = a.nacc * a.N <= 64 ? 64 : (a.nacc * a.N <= 128 ? 128 : (a.nacc * a.N <= 256 ? 256 : 512));
  const size_t fixed = 1024 + 2 * (size_t)a.kblk * a.N * 128 + 256 * 4 + (size_t)a.qps * HIST_BINS * 4 + sizeof(Smem);
  const size_t budget = 227 * 1024;
  const int stages = (int)((budget - fixed) / ((size_t)a.kblk * KB_BYTES));
  a.stages = stages > MAX_STAGES ? MAX_STAGES : stages;
  if (a.stages < 2) return cudaErrorInvalidConfiguration;
  const size_t smem = fixed + (size_t)a.stages * a.kblk * KB_BYTES;
  CUtensorMap kmap, qmap;
  cudaError_t e = make_tmap_2d_bf16(&kmap, p.k_cache, (uint64_t)p.head_dim, (uint64_t)p.num_pages * 64, 64, 64);
  if (e != cudaSuccess) return e;
  e = make_tmap_2d_bf16(&qmap, p.q, (uint64_t)p.head_dim, (uint64_t)p.T * p.n_heads, 64, (uint32_t)a.N);
  if (e != cudaSuccess) return e;
  static int attr_done = 0;
  if (!attr_done) {
    e = cudaFuncSetAttribute(indexer_score_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)budget);
    if (e != cudaSuccess) return e;
    attr_done = 1;
  }
  const int total = a.B * a.tiles_max;
  int grid = num_sms();
  if (grid > total) grid = total;
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(indexer_score_tc, dim3(grid), dim3(THREADS), smem, st, /*pdl=*/false, kmap, qmap, a);
}

// ------------------------------------------------------------------------------------------------
// Top-k selection
// ------------------------------------------------------------------------------------------------
constexpr int COLLECT_THREADS = 256;
constexpr int COLLECT_PER = 32;                                   // scores per thread
constexpr int COLLECT_SLICE = COLLECT_THREADS * COLLECT_PER;      // 8192 scores per CTA
constexpr int CAND_CAP = 4096;                                    // candidates kept in shared memory
constexpr int J_BITS = 20;                                        // n_c <= 2^20 (checked on the host)

// Candidate value: (low 20 order-key bits << 20) | (2^20 - 1 - j); larger = better score, then smaller j.
__device__ __forceinline__ uint64_t cand_value(uint32_t key, int j) {
  return ((uint64_t)(key & ((1u << HIST_SHIFT) - 1u)) << J_BITS) | (uint64_t)((1u << J_BITS) - 1u - (uint32_t)j);
}
__device__ __forceinline__ int cand_j(uint64_t v) { return (int)((1u << J_BITS) - 1u - (uint32_t)(v & ((1u << J_BITS) - 1u))); }

// Bin holding the k-th largest score (from the histogram of one token) and the number of scores in
// the bins above it.  Called by all COLLECT_THREADS threads.
__device__ void threshold_bin(const uint32_t* hist, int K, int* bin_out, int* above_out) {
  __shared__ uint32_t part[COLLECT_THREADS];
  constexpr int PER = HIST_BINS / COLLECT_THREADS;  // thread i owns bins [i*PER, (i+1)*PER)
  const int tid = threadIdx.x;
  uint32_t local[PER];
  uint32_t sum = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    local[i] = hist[tid * PER + i];
    sum += local[i];
  }
  part[tid] = sum;
  __syncthreads();
  // inclusive suffix sums over the threads' groups (from the top bins down)
  for (int off = 1; off < COLLECT_THREADS; off <<= 1) {
    const uint32_t v = (tid + off < COLLECT_THREADS) ? part[tid + off] : 0u;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  const uint32_t incl = part[tid];
  const uint32_t above_group = incl - sum;  // scores in the groups above this thread's
  if (above_group < (uint32_t)K && incl >= (uint32_t)K) {
    uint32_t cum = above_group;
    for (int i = PER - 1; i >= 0; --i) {
      if (cum + local[i] >= (uint32_t)K) {
        *bin_out = tid * PER + i;
        *above_out = (int)cum;
        break;
      }
      cum += local[i];
    }
  }
  __syncthreads();
}

// Appends `val` to a shared-memory list for every lane with `on`, one shared atomic per warp.
template <typename T>
__device__ __forceinline__ void warp_append_smem(unsigned* cnt, T* list, T val, bool on) {
  const unsigned m = __ballot_sync(0xffffffffu, on);
  if (m == 0) return;
  const int lane = threadIdx.x & 31, leader = __ffs(m) - 1;
  unsigned base = 0;
  if (lane == leader) base = atomicAdd(cnt, (unsigned)__popc(m));
  base = __shfl_sync(0xffffffffu, base, leader);
  if (on) list[base + __popc(m & ((1u << lane) - 1u))] = val;
}

// One CTA per (8192-score slice, token): entries above the threshold bin are selected outright,
// entries in it become candidates; both are staged in shared memory and appended to the token's
// global lists with one atomic each.
__device__ void finalize_token(const dsv4_indexer_topk_params& p, const TopkBufs& bufs, int t, int n, uint64_t* dsm);

__global__ void __launch_bounds__(COLLECT_THREADS) topk_collect(dsv4_indexer_topk_params p, TopkBufs bufs) {
  extern __shared__ uint64_t csm[];
  pdl_launch_dependents();
  pdl_wait();
  uint64_t* maybe_s = csm;                                        // COLLECT_SLICE
  int32_t* cert_s = reinterpret_cast<int32_t*>(csm + COLLECT_SLICE);  // COLLECT_SLICE
  __shared__ unsigned n_cert, n_maybe, base_cert, base_maybe;
  __shared__ int sh_bin, sh_above, sh_last;
  const int t = blockIdx.y;
  const int n = visible_entries(p, t);
  const int K = p.topk;
  const int j0 = blockIdx.x * COLLECT_SLICE;
  const float* s = bufs.scores + (int64_t)t * bufs.nc_stride;
  if (n <= K) {  // short context: every candidate, in order (slice 0 writes it)
    if (blockIdx.x == 0) {
      int32_t* out = p.topk_idx + (int64_t)t * K;
      float* out_s = p.topk_score ? p.topk_score + (int64_t)t * K : nullptr;
      for (int x = threadIdx.x; x < K; x += COLLECT_THREADS) {
        out[x] = x < n ? x : -1;
        if (out_s) out_s[x] = x < n ? s[x] : -INFINITY;
      }
    }
    return;
  }
  if (j0 >= n) return;  // block-uniform: this slice holds no entry of the token
  const int j1 = min(n, j0 + COLLECT_SLICE);
  float v[COLLECT_PER];
#pragma unroll
  for (int i = 0; i < COLLECT_PER; ++i) {  // all loads in flight first
    const int j = j0 + i * COLLECT_THREADS + threadIdx.x;
    v[i] = j < j1 ? s[j] : 0.f;
  }
  if (threadIdx.x == 0) {
    sh_bin = HIST_BINS - 1;
    n_cert = n_maybe = 0;
  }
  __syncthreads();
  threshold_bin(bufs.hist + (int64_t)t * HIST_BINS, K, &sh_bin, &sh_above);
  const uint32_t bstar = (uint32_t)sh_bin;
#pragma unroll
  for (int i = 0; i < COLLECT_PER; ++i) {
    const int j = j0 + i * COLLECT_THREADS + threadIdx.x;
    const uint32_t key = order_key(v[i]);
    const uint32_t bin = key >> HIST_SHIFT;
    warp_append_smem<int32_t>(&n_cert, cert_s, j, j < j1 && bin > bstar);
    warp_append_smem<uint64_t>(&n_maybe, maybe_s, cand_value(key, j), j < j1 && bin == bstar);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    base_cert = n_cert ? atomicAdd(&bufs.cnt[3 * t], n_cert) : 0u;
    base_maybe = n_maybe ? atomicAdd(&bufs.cnt[3 * t + 1], n_maybe) : 0u;
  }
  __syncthreads();
  int32_t* certain = bufs.certain + (int64_t)t * K;
  uint64_t* maybe = bufs.maybe + (int64_t)t * bufs.nc_stride;
  for (unsigned x = threadIdx.x; x < n_cert; x += COLLECT_THREADS)
    if (base_cert + x < (unsigned)K) certain[base_cert + x] = cert_s[x];
  for (unsigned x = threadIdx.x; x < n_maybe; x += COLLECT_THREADS)
    if (base_maybe + x < (unsigned)bufs.nc_stride) maybe[base_maybe + x] = maybe_s[x];
  // the CTA that finishes the token's collection last makes the final choice (no CTA waits)
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned slices = (unsigned)((n + COLLECT_SLICE - 1) / COLLECT_SLICE);
    sh_last = atomicAdd(&bufs.cnt[3 * t + 2], 1u) == slices - 1;
  }
  __syncthreads();
  if (!sh_last) return;
  __threadfence();
  finalize_token(p, bufs, t, n, csm);
}

// Digit of the radix bucket holding the rem-th largest element, from a 256-bin histogram: warp 0
// does it with 8 bins per lane and a shuffle scan.  Writes the digit to *digit and the number of
// elements in higher buckets to *above.  Called by the whole CTA.
__device__ __forceinline__ void pick_digit(const unsigned* hist, unsigned rem, int* digit, unsigned* above) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    unsigned c[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      c[i] = hist[255 - 8 * lane - i];  // lane 0 owns the top bins
      sum += c[i];
    }
    unsigned incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    const unsigned excl = incl - sum;
    if (excl < rem && incl >= rem) {
      unsigned cum = excl;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (cum + c[i] >= rem) {
          *digit = 255 - 8 * lane - i;
          *above = cum;
          break;
        }
        cum += c[i];
      }
    }
  }
  __syncthreads();
}

// Exclusive prefix sum of one value per thread over the CTA; *total gets the sum.
__device__ __forceinline__ int block_excl_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < nw ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += u;
    }
    if (lane < nw) warp_tot[lane] = wi - w;
    if (lane == 31) warp_tot[32] = wi;
  }
  __syncthreads();
  const int r = warp_tot[warp] + incl - v;
  *total = warp_tot[32];
  __syncthreads();
  return r;
}

// Exact choice of the remaining entries among the candidates of token t (radix select on the
// candidate values), then the selection written in increasing j through a bitmap over j.  Run by
// the whole CTA that finished the token's collection last; `dsm` holds CAND_CAP candidates followed
// by the bitmap.
__device__ void finalize_token(const dsv4_indexer_topk_params& p, const TopkBufs& bufs, int t, int n, uint64_t* dsm) {
  uint64_t* cand_s = dsm;                                           // CAND_CAP
  uint32_t* bits = reinterpret_cast<uint32_t*>(dsm + CAND_CAP);    // nc_stride / 32 words
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int K = p.topk;
  int32_t* out = p.topk_idx + (int64_t)t * K;
  float* out_s = p.topk_score ? p.topk_score + (int64_t)t * K : nullptr;
  const float* s = bufs.scores + (int64_t)t * bufs.nc_stride;
  __shared__ unsigned hist[256];
  __shared__ unsigned long long sh_prefix;
  __shared__ unsigned sh_rem, sh_above;
  __shared__ int sh_digit;
  __shared__ int warp_tot[33];
  const int words = (n + 31) >> 5;
  for (int x = tid; x < words; x += nthr) bits[x] = 0u;
  const int n_certain = (int)min(bufs.cnt[3 * t], (uint32_t)K);
  const int m = (int)min(bufs.cnt[3 * t + 1], (uint32_t)bufs.nc_stride);
  int need = K - n_certain;
  if (need > m) {  // cannot happen with a complete histogram; keep the output valid
    if (tid == 0) atomicOr(&g_flags_ix, FLAG_TOPK);
    need = m;
  }
  const uint64_t* maybe_g = bufs.maybe + (int64_t)t * bufs.nc_stride;
  const bool in_smem = m <= CAND_CAP;
  if (in_smem)
    for (int i = tid; i < m; i += nthr) cand_s[i] = maybe_g[i];
  const uint64_t* cand = in_smem ? cand_s : maybe_g;
  __syncthreads();
  for (int x = tid; x < n_certain; x += nthr) {
    const int j = bufs.certain[(int64_t)t * K + x];
    if (j >= 0 && j < n) atomicOr(&bits[j >> 5], 1u << (j & 31));
  }
  if (need > 0) {
    // radix select (8-bit digits over the 40-bit values) of the need-th largest candidate
    unsigned long long prefix = 0, mask = 0;
    if (tid == 0) sh_rem = (unsigned)need;
    for (int shift = 32; shift >= 0; shift -= 8) {
      for (int x = tid; x < 256; x += nthr) hist[x] = 0;
      __syncthreads();
      for (int i = tid; i < m; i += nthr) {
        const unsigned long long v = cand[i];
        if ((v & mask) == prefix) atomicAdd(&hist[(v >> shift) & 255ull], 1u);
      }
      __syncthreads();
      const unsigned rem = sh_rem;
      pick_digit(hist, rem, &sh_digit, &sh_above);
      if (tid == 0) {
        sh_rem = rem - sh_above;
        sh_prefix = prefix | ((unsigned long long)sh_digit << shift);
      }
      __syncthreads();
      prefix = sh_prefix;
      mask |= 255ull << shift;
    }
    const unsigned long long kth = prefix;
    for (int i = tid; i < m; i += nthr) {
      const unsigned long long v = cand[i];
      if (v >= kth) {
        const int j = cand_j(v);
        if (j < n) atomicOr(&bits[j >> 5], 1u << (j & 31));
      }
    }
  }
  __syncthreads();
  // compaction of the bitmap in increasing j
  const int per = (words + nthr - 1) / nthr;
  const int w0 = tid * per, w1 = min(words, w0 + per);
  int cnt = 0;
  for (int w = w0; w < w1; ++w) cnt += __popc(bits[w]);
  int total;
  int pos = block_excl_scan(cnt, warp_tot, &total);
  for (int w = w0; w < w1; ++w) {
    uint32_t b = bits[w];
    while (b) {
      const int j = (w << 5) + __ffs(b) - 1;
      b &= b - 1;
      if (pos < K) {
        out[pos] = j;
        if (out_s) out_s[pos] = s[j];
      }
      ++pos;
    }
  }
  for (int x = total + tid; x < K; x += nthr) {
    out[x] = -1;
    if (out_s) out_s[x] = -INFINITY;
  }
}

cudaError_t launch_indexer_topk(const dsv4_indexer_topk_params& p, cudaStream_t st) {
  if (p.T == 0) return cudaSuccess;
  IxLayout L = ix_layout(p);
  char* ws = reinterpret_cast<char*>(p.workspace);
  TopkBufs bufs;
  bufs.scores = reinterpret_cast<float*>(ws + L.scores_off);
  bufs.hist = reinterpret_cast<uint32_t*>(ws + L.hist_off);
  bufs.cnt = reinterpret_cast<uint32_t*>(ws + L.cnt_off);
  bufs.certain = reinterpret_cast<int32_t*>(ws + L.certain_off);
  bufs.maybe = reinterpret_cast<uint64_t*>(ws + L.maybe_off);
  bufs.nc_stride = (int)L.nc_stride;
  cudaError_t e = cudaMemsetAsync(ws + L.hist_off, 0, L.certain_off - L.hist_off, st);
  if (e != cudaSuccess) return e;
  const int max_nc = p.max_context / p.ratio;
  if (max_nc > 0 && use_tc_indexer(p)) {
    e = launch_indexer_score_tc(p, bufs, st);
    if (e != cudaSuccess) return e;
  } else if (max_nc > 0) {
    const int tiles = (max_nc + IX_TILE - 1) / IX_TILE;
    const size_t smem = sizeof(float) * ((size_t)p.q_per_seq * p.n_heads * p.head_dim +
                                         (size_t)p.q_per_seq * p.n_heads + (size_t)(p.head_dim + 1) * (IX_TILE + 1));
    e = cudaFuncSetAttribute(indexer_score_simt, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(indexer_score_simt, dim3(tiles, p.B), dim3(IX_TILE), smem, st, /*pdl=*/false, p, bufs);
    if (e != cudaSuccess) return e;
  }
  static int attr_done = 0;
  const size_t stage_smem = (size_t)COLLECT_SLICE * (sizeof(uint64_t) + sizeof(int32_t));
  const size_t final_smem = (size_t)CAND_CAP * sizeof(uint64_t) + L.nc_stride / 32 * sizeof(uint32_t);
  const size_t csmem = stage_smem > final_smem ? stage_smem : final_smem;
  if (!attr_done) {
    e = cudaFuncSetAttribute(topk_collect, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    attr_done = 1;
  }
  const int slices = max_nc > 0 ? (max_nc + COLLECT_SLICE - 1) / COLLECT_SLICE : 1;
  return launch_pdl(topk_collect, dim3(slices, p.T), dim3(COLLECT_THREADS), csmem, st, /*pdl=*/false, p, bufs);
}

cudaError_t read_flags_indexer(uint32_t* f) {
  unsigned int v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_flags_ix, sizeof(v));
  if (e != cudaSuccess) return e;
  *f |= v;
  return cudaMemcpyToSymbol(g_flags_ix, &z, sizeof(z));
}

}  // namespace dsv4
