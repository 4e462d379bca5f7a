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
#include "dsv4_common.cuh"
#include "dsv4_launch.h"

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

// One CTA per sequence; its new tokens are handled in position order so that a fold sees
// exactly the state a token-by-token decode would have (a later token of the same step can
// reuse the ring slot of a row the fold still needs).
__global__ void __launch_bounds__(ROW_THREADS) compress_update_kernel(dsv4_compress_update_params p) {
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
    // ---- store: kv half as is, score half + APE (fp32 add)
    {
      const float2* src = reinterpret_cast<const float2*>(p.kv_score + (int64_t)t * state_w);
      float2* dst = reinterpret_cast<float2*>(state_b + (int64_t)(pos % nslots) * state_w);
      const float2* ape = p.ape ? reinterpret_cast<const float2*>(p.ape + (int64_t)(pos % r) * half) : nullptr;
      for (int c = i; c < state_w / 2; c += ROW_THREADS) {
        float2 v = src[c];
        if (ape != nullptr && c >= half / 2) {
          float2 a = ape[c - half / 2];
          v.x += a.x;
          v.y += a.y;
        }
        dst[c] = v;
      }
    }
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
      float x0 = a0 / s0, x1 = a1 / s1;
      // ---- RMSNorm over the 576 dims
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
      // ---- RoPE of the rope dims at position j * ratio
      if (i >= 256) {
        int rp = j * r;
        if (rp >= p.max_pos) {
          atomicOr(&g_flags_ic, FLAG_PAGE);
          rp = 0;
        }
        rope_pair(x0, x1, p.cos_sin + (int64_t)rp * 64, i - 256);
      }
      // ---- encode into main-cache row j
      const int lp = j / p.page_size;
      int page = (lp < p.max_pages_per_seq) ? p.block_table[(int64_t)b * p.max_pages_per_seq + lp] : -1;
      if (page < 0 || page >= p.num_pages) {
        if (i == 0) atomicOr(&g_flags_ic, FLAG_PAGE);
      } else {
        uint8_t* row = reinterpret_cast<uint8_t*>(p.main_cache) +
                       ((int64_t)page * p.page_size + j % p.page_size) * row_bytes(p.cache_dtype, D);
        encode_pair_store(p.cache_dtype, row, i, x0, x1);
      }
      __syncthreads();
    }
  }
}

cudaError_t launch_kv_insert(const dsv4_kv_insert_params& p, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  kv_insert_kernel<<<p.T, ROW_THREADS, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_compress_update(const dsv4_compress_update_params& p, cudaStream_t s) {
  if (p.B == 0) return cudaSuccess;
  compress_update_kernel<<<p.B, ROW_THREADS, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t read_flags_insert_compress(uint32_t* f) {
  unsigned int v = 0, z = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_flags_ic, sizeof(v));
  if (e != cudaSuccess) return e;
  *f |= v;
  return cudaMemcpyToSymbol(g_flags_ic, &z, sizeof(z));
}

}  // namespace dsv4
