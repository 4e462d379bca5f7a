// SWA KV insert and compressor state store + fold.
//
// KV insert: "DeepSeek V4 Attention: Code Reading Map", §4 _fused_qnorm_rope_kv_insert() (KV half);
// "vllm.models.deepseek_v41.attention", DeepseekV4Attention._fused_qnorm_rope_kv_insert.
// Compressor: "DeepSeek V4 Attention: Code Reading Map", §"What Are the Gate Scores?" and
// §"How Does Compression Actually Work?" (steps 1-7, state cache float32, APE, overlap).
//
// Both kernels give one 288-thread CTA (9 warps) to a row: thread i owns latent dims 2i, 2i+1,
// so the 8 no-pe blocks of an fp8_ds_mla record are warps 0..7 (UE8M0 amax by warp max) and the
// rope pairs (GPT-J interleaved) sit whole inside warp 8.
#include <cooperative_groups.h>

#include "dsv4_common.cuh"
#include "dsv4_launch.h"

namespace cg = cooperative_groups;

namespace dsv4 {

static __device__ unsigned int g_flags_ic = 0;

constexpr int ROW_THREADS = 288;

__device__ __forceinline__ void rope_pair(float& x0, float& x1, const float* cs, int pair) {
  const float c = cs[pair], s = cs[32 + pair];
  const float y0 = x0 * c - x1 * s;
  const float y1 = x0 * s + x1 * c;
  x0 = y0;
  x1 = y1;
}

__global__ void __launch_bounds__(ROW_THREADS) kv_insert_kernel(dsv4_kv_insert_params p) {
  pdl_launch_dependents();
  pdl_wait();
  const int t = blockIdx.x, i = threadIdx.x;
  const int64_t slot = p.slot_mapping[t];
  if (slot < 0) return;
  const int64_t page = slot / p.page_size;
  if (page >= p.num_pages) {
    if (i == 0) atomicOr(&g_flags_ic, FLAG_PAGE);
    return;
  }
  float2 x;
  if (p.kv_dtype == DSV4_F32)
    x = reinterpret_cast<const float2*>(p.kv_new)[(int64_t)t * (D / 2) + i];
  else
    x = decode_pair(DSV4_BF16, reinterpret_cast<const uint8_t*>(p.kv_new) + (int64_t)t * D * 2, i);
  if (p.cos_sin != nullptr && i >= 256) {
    int pos = p.positions[t];
    if (pos < 0 || pos >= p.max_pos) {
      atomicOr(&g_flags_ic, FLAG_PAGE);
      pos = 0;
    }
    rope_pair(x.x, x.y, p.cos_sin + (int64_t)pos * 64, i - 256);
  }
  uint8_t* row = reinterpret_cast<uint8_t*>(p.cache) + slot * row_bytes(p.cache_dtype, D);
  encode_pair_store(p.cache_dtype, row, i, x.x, x.y);
}


// RMSNorm * weight of the folded entry j (thread i holds dims 2i, 2i+1), GPT-J RoPE of the rope pairs
// at position j * ratio, and the encoded store into main-cache row j of sequence b.  All 288 threads.
__device__ void finish_entry(const dsv4_compress_update_params& p, int b, int j, int i, float x0, float x1,
                             float* red) {
  float ss = warp_sum(x0 * x0 + x1 * x1);
  if ((i & 31) == 0) red[i >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < ROW_THREADS / 32; ++w) tot += red[w];
  const float inv = 1.0f / sqrtf(tot / (float)D + p.eps);
  const float2 g = reinterpret_cast<const float2*>(p.norm_weight)[i];
  x0 = x0 * inv * g.x;
  x1 = x1 * inv * g.y;
  if (i >= 256) {
    int rp = j * p.ratio;
    if (rp >= p.max_pos) {
      atomicOr(&g_flags_ic, FLAG_PAGE);
      rp = 0;
    }
    rope_pair(x0, x1, p.cos_sin + (int64_t)rp * 64, i - 256);
  }
  const int lp = j / p.page_size;
  const int page = (lp < p.max_pages_per_seq) ? p.block_table[(int64_t)b * p.max_pages_per_seq + lp] : -1;
  if (page < 0 || page >= p.num_pages) {
    if (i == 0) atomicOr(&g_flags_ic, FLAG_PAGE);
  } else {
    uint8_t* row = reinterpret_cast<uint8_t*>(p.main_cache) +
                   ((int64_t)page * p.page_size + j % p.page_size) * row_bytes(p.cache_dtype, D);
    encode_pair_store(p.cache_dtype, row, i, x0, x1);
  }
}

// Stores the fp32 state row of token t (kv half as is, score half + APE); all threads of the CTA.
__device__ __forceinline__ void store_state_row(const dsv4_compress_update_params& p, float* state_b, int t, int pos,
                                                int tid, int nthreads) {
  const int coff = p.coff, r = p.ratio;
  const int state_w = 2 * coff * D, half = coff * D;
  const float2* src = reinterpret_cast<const float2*>(p.kv_score + (int64_t)t * state_w);
  float2* dst = reinterpret_cast<float2*>(state_b + (int64_t)(pos % (coff * r)) * state_w);
  const float2* ape = p.ape ? reinterpret_cast<const float2*>(p.ape + (int64_t)(pos % r) * half) : nullptr;
  for (int c = tid; c < state_w / 2; c += nthreads) {
    float2 v = src[c];
    if (ape != nullptr && c >= half / 2) {
      const float2 a = ape[c - half / 2];
      v.x += a.x;
      v.y += a.y;
    }
    dst[c] = v;
  }
}

// One CTA per sequence; its new tokens are handled in position order so that a fold sees
// exactly the state a token-by-token decode would have (a later token of the same step can
// reuse the ring slot of a row the fold still needs).
__global__ void __launch_bounds__(ROW_THREADS) compress_update_kernel(dsv4_compress_update_params p) {
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.x, i = threadIdx.x;
  const int coff = p.coff, r = p.ratio;
  const int nslots = coff * r;
  const int state_w = 2 * coff * D;  // floats per state row
  const int half = coff * D;         // kv half width = score half width
  float* state_b = p.state + (int64_t)b * nslots * state_w;
  __shared__ float red[ROW_THREADS / 32];

  for (int k = 0; k < p.q_per_seq; ++k) {
    const int t = b * p.q_per_seq + k;
    const int pos = p.positions[t];
    if (pos < 0) {  // block-uniform: every thread skips the token
      if (i == 0) atomicOr(&g_flags_ic, FLAG_PAGE);
      continue;
    }
    store_state_row(p, state_b, t, pos, i, ROW_THREADS);  // kv half as is, score half + APE
    __syncthreads();
    if ((pos + 1) % r == 0) {
      const int j = pos / r;
      // ---- fold: per-channel online softmax over the group's rows
      float m0 = -INFINITY, m1 = -INFINITY, s0 = 0.f, s1 = 0.f, a0 = 0.f, a1 = 0.f;
      const int nser = (coff == 2 && j >= 1) ? 2 : 1;
      for (int ser = 0; ser < nser; ++ser) {
        const int q0 = (j - ser) * r;  // series A: this group; series B: the previous group
        const int kv_off = ser * D, sc_off = half + ser * D;
#pragma unroll 4
        for (int q = q0; q < q0 + r; ++q) {
          const float* rowp = state_b + (int64_t)(q % nslots) * state_w;
          const float2 kv = reinterpret_cast<const float2*>(rowp + kv_off)[i];
          const float2 sc = reinterpret_cast<const float2*>(rowp + sc_off)[i];
          float n0 = fmaxf(m0, sc.x), n1 = fmaxf(m1, sc.y);
          float c0 = expf(m0 - n0), c1 = expf(m1 - n1);
          float e0 = expf(sc.x - n0), e1 = expf(sc.y - n1);
          s0 = s0 * c0 + e0;
          s1 = s1 * c1 + e1;
          a0 = a0 * c0 + e0 * kv.x;
          a1 = a1 * c1 + e1 * kv.y;
          m0 = n0;
          m1 = n1;
        }
      }
      finish_entry(p, b, j, i, a0 / s0, a1 / s1, red);
      __syncthreads();
    }
  }
}


// Ratio-128 groups (coff = 1): one 8-CTA cluster per sequence.  Each CTA folds 16 of the group's
// 128 rows into per-channel partial softmax states (max, sum, weighted kv sum) in its shared memory;
// CTA 0 combines the eight partial states through distributed shared memory and finishes the entry.
// The sequence's tokens are still handled in position order (stores up to the emitting token, the
// fold, then the later tokens' stores).  Cluster barriers are hardware barriers, not flag spins.
constexpr int FOLD_CTAS = 8;
__global__ void __cluster_dims__(FOLD_CTAS, 1, 1) __launch_bounds__(ROW_THREADS)
    compress_fold_cluster_kernel(dsv4_compress_update_params p) {
  pdl_launch_dependents();
  pdl_wait();
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.y, i = threadIdx.x;
  const int r = p.ratio, nslots = r;  // coff == 1
  const int state_w = 2 * D;
  float* state_b = p.state + (int64_t)b * nslots * state_w;
  __shared__ float2 pm[ROW_THREADS], ps[ROW_THREADS], pa[ROW_THREADS];
  __shared__ float red[ROW_THREADS / 32];
  int k_emit = -1;
  for (int k = 0; k < p.q_per_seq; ++k) {
    const int pos = p.positions[b * p.q_per_seq + k];
    if (pos >= 0 && (pos + 1) % r == 0) {
      k_emit = k;
      break;
    }
  }
  const int k_end = k_emit >= 0 ? k_emit + 1 : p.q_per_seq;
  if (rank == 0)
    for (int k = 0; k < k_end; ++k) {
      const int t = b * p.q_per_seq + k, pos = p.positions[t];
      if (pos < 0) {
        if (i == 0) atomicOr(&g_flags_ic, FLAG_PAGE);
        continue;
      }
      store_state_row(p, state_b, t, pos, i, ROW_THREADS);
      __syncthreads();
    }
  if (k_emit >= 0) {  // cluster-uniform
    cluster.sync();   // the stored rows are visible to every CTA of the cluster
    const int pos = p.positions[b * p.q_per_seq + k_emit];
    const int j = pos / r;
    float m0 = -INFINITY, m1 = -INFINITY, s0 = 0.f, s1 = 0.f, a0 = 0.f, a1 = 0.f;
    const int q0 = j * r + rank * (r / FOLD_CTAS);
    float2 kv[16], sc[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {  // all 32 loads in flight
      const float* rowp = state_b + (int64_t)((q0 + u) % nslots) * state_w;
      kv[u] = reinterpret_cast<const float2*>(rowp)[i];
      sc[u] = reinterpret_cast<const float2*>(rowp + D)[i];
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const float n0 = fmaxf(m0, sc[u].x), n1 = fmaxf(m1, sc[u].y);
      const float c0 = expf(m0 - n0), c1 = expf(m1 - n1);
      const float e0 = expf(sc[u].x - n0), e1 = expf(sc[u].y - n1);
      s0 = s0 * c0 + e0;
      s1 = s1 * c1 + e1;
      a0 = a0 * c0 + e0 * kv[u].x;
      a1 = a1 * c1 + e1 * kv[u].y;
      m0 = n0;
      m1 = n1;
    }
    pm[i] = make_float2(m0, m1);
    ps[i] = make_float2(s0, s1);
    pa[i] = make_float2(a0, a1);
    cluster.sync();  // every CTA's partial state is in its shared memory
    if (rank == 0) {
      float M0 = -INFINITY, M1 = -INFINITY;
      float2 qm[FOLD_CTAS], qs[FOLD_CTAS], qa[FOLD_CTAS];
#pragma unroll
      for (int c = 0; c < FOLD_CTAS; ++c) {
        qm[c] = cluster.map_shared_rank(pm, c)[i];
        qs[c] = cluster.map_shared_rank(ps, c)[i];
        qa[c] = cluster.map_shared_rank(pa, c)[i];
        M0 = fmaxf(M0, qm[c].x);
        M1 = fmaxf(M1, qm[c].y);
      }
      float S0 = 0.f, S1 = 0.f, A0 = 0.f, A1 = 0.f;
#pragma unroll
      for (int c = 0; c < FOLD_CTAS; ++c) {
        const float w0 = expf(qm[c].x - M0), w1 = expf(qm[c].y - M1);
        S0 += qs[c].x * w0;
        S1 += qs[c].y * w1;
        A0 += qa[c].x * w0;
        A1 += qa[c].y * w1;
      }
      finish_entry(p, b, j, i, A0 / S0, A1 / S1, red);
    }
    cluster.sync();  // no CTA leaves while CTA 0 still reads its shared memory
  }
  if (rank == 0)
    for (int k = k_end; k < p.q_per_seq; ++k) {
      const int t = b * p.q_per_seq + k, pos = p.positions[t];
      if (pos < 0) continue;
      __syncthreads();
      store_state_row(p, state_b, t, pos, i, ROW_THREADS);
    }
}

cudaError_t launch_kv_insert(const dsv4_kv_insert_params& p, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  return launch_pdl(kv_insert_kernel, dim3(p.T), dim3(ROW_THREADS), 0, s, true, p);
}

cudaError_t launch_compress_update(const dsv4_compress_update_params& p, cudaStream_t s) {
  if (p.B == 0) return cudaSuccess;
  if (p.coff == 1 && p.ratio % (FOLD_CTAS * 16) == 0 && p.ratio / FOLD_CTAS == 16) {
    return launch_pdl(compress_fold_cluster_kernel, dim3(FOLD_CTAS, p.B), dim3(ROW_THREADS), 0, s, true, p);
  }
  return launch_pdl(compress_update_kernel, dim3(p.B), dim3(ROW_THREADS), 0, s, true, p);
}

cudaError_t read_flags_insert_compress(uint32_t* f) {
  unsigned int v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_flags_ic, sizeof(v));
  if (e != cudaSuccess) return e;
  *f |= v;
  return cudaMemcpyToSymbol(g_flags_ic, &z, sizeof(z));
}

}  // namespace dsv4
