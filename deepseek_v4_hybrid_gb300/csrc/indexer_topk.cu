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
  if (max_nc > 0) {
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
