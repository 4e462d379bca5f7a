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

static AtLayout at_layout(const dsv4_sparse_mla_decode_params& p) {
  AtLayout L;
  L.chunk_rows = AT_CH;
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
  const size_t smem = sizeof(float) * ((size_t)AT_HG * D + (size_t)AT_CH * (D + 1) + (size_t)AT_HG * AT_CH);
  cudaError_t e = cudaFuncSetAttribute(mla_partial_simt, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  mla_partial_simt<<<dim3(L.n_chunks, p.T, (p.H + AT_HG - 1) / AT_HG), AT_THREADS, smem, st>>>(p, o_part, ml_part,
                                                                                                 L.n_chunks);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
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
