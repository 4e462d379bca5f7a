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
#include "tc_ptx.cuh"

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

__device__ __forceinline__ void kv_insert_body(const dsv4_kv_insert_params& p) {
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

__global__ void __launch_bounds__(ROW_THREADS) kv_insert_kernel(dsv4_kv_insert_params p) {
  pdl_start(p.after_independent != 0);
  kv_insert_body(p);
  if (p.after_independent) pdl_wait();  // completes only after the kernel before it
}

// ------------------------------------------------------------------------------------------------
// Fused query preparation + KV insert.  CTA (t, y): for y < ceil(H_pad / 8) warp w < 8 prepares
// query head 8 y + w of token t; CTA (t, ngroups) stores the token's kv row (kv_insert_body).  A
// warp holds its head in registers: with 16-byte vectors of E elements (8 bf16 or 4 fp32), lane l
// takes no-pe vectors l + 32 v (512 / E / 32 of them) and, when l < 64 / E, rope vector 512 / E + l,
// whose GPT-J pairs lie inside it.  All loads come before any store, so q_out may be q itself.
// ------------------------------------------------------------------------------------------------
constexpr int QP_HEADS = 8;

template <bool BF>
struct QVec {
  static constexpr int E = BF ? 8 : 4;  // elements per 16-byte vector
  static __device__ __forceinline__ void load(const uint8_t* src, int vec, float (&x)[E]) {
    const uint4 u = reinterpret_cast<const uint4*>(src)[vec];
    if (BF) {
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        x[2 * k] = __uint_as_float(w[k] << 16);
        x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
      }
    } else {
      x[0] = __uint_as_float(u.x);
      x[1] = __uint_as_float(u.y);
      x[2] = __uint_as_float(u.z);
      x[3] = __uint_as_float(u.w);
    }
  }
  static __device__ __forceinline__ void store(uint8_t* dst, int vec, const float (&x)[E]) {
    uint4 u;
    if (BF) {
      u = make_uint4(float2_to_bf16x2_bits(x[0], x[1]), float2_to_bf16x2_bits(x[2], x[3]),
                     float2_to_bf16x2_bits(x[4], x[5]), float2_to_bf16x2_bits(x[6], x[7]));
    } else {
      u = make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]), __float_as_uint(x[3]));
    }
    reinterpret_cast<uint4*>(dst)[vec] = u;
  }
};

// One query head (576 elements at src) -> dst, by one warp.  cs: the cos/sin row of the token's
// position, or nullptr for no RoPE; w: the RMSNorm weight or nullptr (= 1).
template <bool BF>
__device__ __forceinline__ void qprep_head(const uint8_t* src, uint8_t* dst, bool norm, const float* w, float eps,
                                           const float* cs, int lane) {
  using V = QVec<BF>;
  constexpr int E = V::E, NV = D_NOPE / E / 32, RV = D_ROPE / E;
  float x[NV][E], r[E];
#pragma unroll
  for (int v = 0; v < NV; ++v) V::load(src, lane + 32 * v, x[v]);
  const bool rl = lane < RV;
  if (rl) V::load(src, D_NOPE / E + lane, r);
  float ss = 0.f;
#pragma unroll
  for (int v = 0; v < NV; ++v)
#pragma unroll
    for (int e = 0; e < E; ++e) ss = fmaf(x[v][e], x[v][e], ss);
  if (rl)
#pragma unroll
    for (int e = 0; e < E; ++e) ss = fmaf(r[e], r[e], ss);
  if (norm) {
    const float inv = 1.0f / sqrtf(warp_sum(ss) / (float)D + eps);
#pragma unroll
    for (int v = 0; v < NV; ++v) {
      const int d0 = (lane + 32 * v) * E;
#pragma unroll
      for (int e = 0; e < E; ++e) x[v][e] *= inv * (w ? __ldg(w + d0 + e) : 1.f);
    }
    if (rl) {
      const int d0 = D_NOPE + lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) r[e] *= inv * (w ? __ldg(w + d0 + e) : 1.f);
    }
  }
  if (rl && cs != nullptr) {
#pragma unroll
    for (int k = 0; k < E / 2; ++k) {
      const int pr = lane * (E / 2) + k;  // GPT-J pair of dims 512 + 2 pr, 512 + 2 pr + 1
      const float c = __ldg(cs + pr), s = __ldg(cs + 32 + pr);
      const float y0 = r[2 * k] * c - r[2 * k + 1] * s;
      const float y1 = r[2 * k] * s + r[2 * k + 1] * c;
      r[2 * k] = y0;
      r[2 * k + 1] = y1;
    }
  }
#pragma unroll
  for (int v = 0; v < NV; ++v) V::store(dst, lane + 32 * v, x[v]);
  if (rl) V::store(dst, D_NOPE / E + lane, r);
}

__global__ void __launch_bounds__(ROW_THREADS) qnorm_rope_kv_insert_kernel(dsv4_qnorm_rope_kv_insert_params p) {
  pdl_start(p.after_independent != 0);
  const int t = blockIdx.x, y = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ngroups = (p.H_pad + QP_HEADS - 1) / QP_HEADS;
  if (y < ngroups) {
    const int h = y * QP_HEADS + warp;
    if (warp < QP_HEADS && h < p.H_pad) {
      const int esz = p.act_dtype == DSV4_F32 ? 4 : 2;
      uint8_t* dst = reinterpret_cast<uint8_t*>(p.q_out) + ((int64_t)t * p.H_pad + h) * D * esz;
      if (h >= p.H) {  // padding head: zeros
        for (int v = lane; v < D * esz / 16; v += 32) reinterpret_cast<uint4*>(dst)[v] = make_uint4(0u, 0u, 0u, 0u);
      } else {
        const uint8_t* src = reinterpret_cast<const uint8_t*>(p.q) + ((int64_t)t * p.H + h) * D * esz;
        const float* cs = nullptr;
        if (p.apply_q_rope) {
          int pos = p.positions[t];
          if (pos < 0 || pos >= p.max_pos) {
            if (lane == 0) atomicOr(&g_flags_ic, FLAG_PAGE);
            pos = 0;
          }
          cs = p.cos_sin + (int64_t)pos * 64;
        }
        if (p.act_dtype == DSV4_F32)
          qprep_head<false>(src, dst, p.apply_q_norm != 0, p.q_norm_weight, p.eps, cs, lane);
        else
          qprep_head<true>(src, dst, p.apply_q_norm != 0, p.q_norm_weight, p.eps, cs, lane);
      }
    }
  } else {
    dsv4_kv_insert_params k;
    k.struct_size = sizeof(k);
    k.kv_new = p.kv_new;
    k.kv_dtype = p.act_dtype;
    k.slot_mapping = p.slot_mapping;
    k.cache = p.cache;
    k.cache_dtype = p.cache_dtype;
    k.T = p.T;
    k.page_size = p.page_size;
    k.num_pages = p.num_pages;
    k.positions = p.positions;
    k.cos_sin = p.apply_kv_rope ? p.cos_sin : nullptr;
    k.max_pos = p.max_pos;
    k.after_independent = p.after_independent;
    kv_insert_body(k);
  }
  if (p.after_independent) pdl_wait();  // completes only after the kernel before it
}

cudaError_t launch_qnorm_rope_kv_insert(const dsv4_qnorm_rope_kv_insert_params& p, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  const int ngroups = (p.H_pad + QP_HEADS - 1) / QP_HEADS;
  return launch_pdl(qnorm_rope_kv_insert_kernel, dim3(p.T, ngroups + 1), dim3(ROW_THREADS), 0, s, true, p);
}

// What finishing entry j of sequence b needs, loaded before the fold so that it costs no extra
// round trip: the RMSNorm weight pair of thread i, its cos/sin pair (rope threads) at position
// j * ratio and the destination row of the main cache.
struct EntryCtx {
  float2 g;
  float c, s;
  uint8_t* row;
};

__device__ __forceinline__ EntryCtx entry_prefetch(const dsv4_compress_update_params& p, int b, int j, int i) {
  EntryCtx e;
  e.g = reinterpret_cast<const float2*>(p.norm_weight)[i];
  e.c = 1.f;
  e.s = 0.f;
  if (i >= 256) {
    int rp = j * p.ratio;
    if (rp >= p.max_pos) {
      atomicOr(&g_flags_ic, FLAG_PAGE);
      rp = 0;
    }
    e.c = p.cos_sin[(int64_t)rp * 64 + (i - 256)];
    e.s = p.cos_sin[(int64_t)rp * 64 + 32 + (i - 256)];
  }
  const int lp = j / p.page_size;
  const int page = (lp < p.max_pages_per_seq) ? p.block_table[(int64_t)b * p.max_pages_per_seq + lp] : -1;
  e.row = (page >= 0 && page < p.num_pages)
              ? reinterpret_cast<uint8_t*>(p.main_cache) +
                    ((int64_t)page * p.page_size + j % p.page_size) * row_bytes(p.cache_dtype, D)
              : nullptr;
  return e;
}

// Index key of entry j (b, j) from its latent in shared memory (lat[576], the entry after its
// RMSNorm and before its RoPE): k = wk lat, RMSNorm over ik_dim dims times ik_norm_weight, GPT-J
// RoPE of the last 64 dims at position j * ratio, encoded into row j of the indexer cache.  All 288
// threads: warp w computes outputs w, w + 9, ... (one 1152-byte wk row a time, read as bf16 pairs);
// then thread i < ik_dim / 2 holds the pair (2i, 2i + 1).
__device__ void index_key_store(const dsv4_compress_update_params& p, int b, int j, const float* lat, float* kk,
                                float* red, int i) {
  const int warp = i >> 5, lane = i & 31, d = p.ik_dim;
  const uint32_t* wk = reinterpret_cast<const uint32_t*>(p.wk);
  const float2* lat2 = reinterpret_cast<const float2*>(lat);
  constexpr int U = D / 2 / 32;  // bf16 pairs of a wk row per lane (9)
  constexpr int RPW = 8;         // wk rows a warp has in flight at once
  float2 x[U];
#pragma unroll
  for (int u = 0; u < U; ++u) x[u] = lat2[lane + 32 * u];
  for (int o0 = warp * RPW; o0 < d; o0 += (ROW_THREADS / 32) * RPW) {
    uint32_t w[RPW][U];
#pragma unroll
    for (int r = 0; r < RPW; ++r)
#pragma unroll
      for (int u = 0; u < U; ++u)
        w[r][u] = o0 + r < d ? __ldg(wk + (int64_t)(o0 + r) * (D / 2) + lane + 32 * u) : 0u;
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        acc = fmaf(__uint_as_float(w[r][u] << 16), x[u].x, acc);
        acc = fmaf(__uint_as_float(w[r][u] & 0xFFFF0000u), x[u].y, acc);
      }
      acc = warp_sum(acc);
      if (lane == 0 && o0 + r < d) kk[o0 + r] = acc;
    }
  }
  __syncthreads();
  const bool own = i < d / 2;
  float k0 = own ? kk[2 * i] : 0.f, k1 = own ? kk[2 * i + 1] : 0.f;
  const float ss = warp_sum(k0 * k0 + k1 * k1);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < ROW_THREADS / 32; ++w) tot += red[w];
  const float inv = 1.0f / sqrtf(tot / (float)d + p.ik_eps);
  const int pr = i - (d - D_ROPE) / 2;  // rope pair of thread i (the key's last 64 dims)
  if (own) {
    k0 = k0 * inv * __ldg(p.ik_norm_weight + 2 * i);
    k1 = k1 * inv * __ldg(p.ik_norm_weight + 2 * i + 1);
    if (pr >= 0) {
      int rp = j * p.ratio;
      if (rp >= p.max_pos) {
        atomicOr(&g_flags_ic, FLAG_PAGE);
        rp = 0;
      }
      const float c = __ldg(p.cos_sin + (int64_t)rp * 64 + pr), s = __ldg(p.cos_sin + (int64_t)rp * 64 + 32 + pr);
      const float y0 = k0 * c - k1 * s;
      const float y1 = k0 * s + k1 * c;
      k0 = y0;
      k1 = y1;
    }
  }
  float amax = 0.f;
  if (p.ik_dtype == DSV4_I8_ROWSCALE) {  // block-uniform
    __syncthreads();                      // red is reused
    const float m = warp_max(own ? fmaxf(fabsf(k0), fabsf(k1)) : 0.f);
    if (lane == 0) red[warp] = m;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < ROW_THREADS / 32; ++w) amax = fmaxf(amax, red[w]);
  }
  if (!own) return;
  const int lp = j / p.page_size;
  const int page = (lp < p.ik_max_pages) ? p.ik_block_table[(int64_t)b * p.ik_max_pages + lp] : -1;
  if (page < 0 || page >= p.ik_num_pages) {
    if (i == 0) atomicOr(&g_flags_ic, FLAG_PAGE);
    return;
  }
  const int64_t slot = (int64_t)page * p.page_size + j % p.page_size;
  uint8_t* dst = reinterpret_cast<uint8_t*>(p.ik_cache) + slot * row_bytes(p.ik_dtype, d);
  if (p.ik_dtype == DSV4_F32) {
    reinterpret_cast<float2*>(dst)[i] = make_float2(k0, k1);
  } else if (p.ik_dtype == DSV4_BF16) {
    reinterpret_cast<uint32_t*>(dst)[i] = float2_to_bf16x2_bits(k0, k1);
  } else if (p.ik_dtype == DSV4_MXFP4) {
    // a 32-element block is one half warp (thread i holds elements 2i, 2i + 1)
    float m = fmaxf(fabsf(k0), fabsf(k1));
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int e = mxfp4_exponent(m);
    const float sc = exp2_neg_int(e);
    dst[i] = (uint8_t)(e2m1_code(k0 * sc) | (e2m1_code(k1 * sc) << 4));
    if ((i & 15) == 0) dst[d / 2 + (i >> 4)] = (uint8_t)(e + 127);
  } else {
    const float scale = amax == 0.f ? 1.f : __fdiv_rn(amax, 127.f);
    const float c0 = fminf(fmaxf(rintf(__fdiv_rn(k0, scale)), -127.f), 127.f);
    const float c1 = fminf(fmaxf(rintf(__fdiv_rn(k1, scale)), -127.f), 127.f);
    reinterpret_cast<uint16_t*>(dst)[i] = (uint16_t)(((uint32_t)(int)c0 & 0xFFu) | (((uint32_t)(int)c1 & 0xFFu) << 8));
    if (i == 0) *reinterpret_cast<float*>(dst + d) = scale;
  }
}

// RMSNorm * weight of the folded entry (thread i holds dims 2i, 2i+1), GPT-J RoPE of the rope pairs
// and the encoded store into the main-cache row; with an index-key projection, also the entry's index
// key (index_key_store, from the latent before the RoPE).  All 288 threads (block reductions).
__device__ void entry_finish(const dsv4_compress_update_params& p, const EntryCtx& e, int i, float x0, float x1,
                             float* red, int b, int j) {
  __shared__ __align__(16) float lat[D];
  __shared__ float kk[128];
  float ss = warp_sum(x0 * x0 + x1 * x1);
  if ((i & 31) == 0) red[i >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < ROW_THREADS / 32; ++w) tot += red[w];
  const float inv = 1.0f / sqrtf(tot / (float)D + p.eps);
  x0 = x0 * inv * e.g.x;
  x1 = x1 * inv * e.g.y;
  if (p.wk != nullptr) reinterpret_cast<float2*>(lat)[i] = make_float2(x0, x1);
  if (i >= 256) {
    const float y0 = x0 * e.c - x1 * e.s;
    const float y1 = x0 * e.s + x1 * e.c;
    x0 = y0;
    x1 = y1;
  }
  if (e.row == nullptr) {
    if (i == 0) atomicOr(&g_flags_ic, FLAG_PAGE);
  } else {
    encode_pair_store(p.cache_dtype, e.row, i, x0, x1);
  }
  if (p.wk != nullptr) {  // block-uniform
    __syncthreads();      // lat is complete; red is free again
    index_key_store(p, b, j, lat, kk, red, i);
  }
}

// Online softmax step of one row of a fold (two channels per thread).
struct FoldAcc {
  float m0 = -INFINITY, m1 = -INFINITY, s0 = 0.f, s1 = 0.f, a0 = 0.f, a1 = 0.f;
  __device__ __forceinline__ void add(float2 kv, float2 sc) {
    const float n0 = fmaxf(m0, sc.x), n1 = fmaxf(m1, sc.y);
    const float c0 = expf(m0 - n0), c1 = expf(m1 - n1);
    const float e0 = expf(sc.x - n0), e1 = expf(sc.y - n1);
    s0 = s0 * c0 + e0;
    s1 = s1 * c1 + e1;
    a0 = a0 * c0 + e0 * kv.x;
    a1 = a1 * c1 + e1 * kv.y;
    m0 = n0;
    m1 = n1;
  }
};

// Channel pair i of token t's new state row: kv series `ser` and score series `ser` (+ APE of its
// position), as stored in the ring.
__device__ __forceinline__ void new_row_pair(const dsv4_compress_update_params& p, int t, int pos, int ser, int i,
                                             float2& kv, float2& sc) {
  const int half = p.coff * D;
  const float2* src = reinterpret_cast<const float2*>(p.kv_score + (int64_t)t * 2 * half);
  kv = src[ser * (D / 2) + i];
  sc = src[half / 2 + ser * (D / 2) + i];
  if (p.ape != nullptr) {
    const float2 a = reinterpret_cast<const float2*>(p.ape + (int64_t)(pos % p.ratio) * half)[ser * (D / 2) + i];
    sc.x += a.x;
    sc.y += a.y;
  }
}

// One CTA per sequence; its new tokens are handled in position order, so a fold sees exactly the
// state a token-by-token decode would have (a later token of the same step may reuse the ring slot
// of a row an earlier fold reads).  Per token, everything it needs is loaded up front (its new row,
// the fold's other rows from the ring, the entry's weights and destination); the token's own row
// enters the fold from registers, so storing it costs no round trip.
constexpr int FOLD_BATCH = 8;
__device__ __forceinline__ void compress_update_body(const dsv4_compress_update_params& p) {
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
    const bool emit = (pos + 1) % r == 0;
    const int j = pos / r;
    float2 kvn[2], scn[2];
    new_row_pair(p, t, pos, 0, i, kvn[0], scn[0]);
    if (coff == 2) new_row_pair(p, t, pos, 1, i, kvn[1], scn[1]);
    EntryCtx ec;
    // fold rows: series A (kv / score block 0) over this group, then for coff == 2 series B (block 1)
    // over the previous group (absent for j = 0)
    const int nser = (coff == 2 && j >= 1) ? 2 : 1;
    const int nrows = emit ? nser * r : 0;
    float2 kvb[FOLD_BATCH], scb[FOLD_BATCH];
    auto load_batch = [&](int base) {
#pragma unroll
      for (int u = 0; u < FOLD_BATCH; ++u) {
        const int idx = base + u;
        if (idx < nrows) {
          const int ser = idx / r, q = (j - ser) * r + idx % r;
          const float* rowp = state_b + (int64_t)(q % nslots) * state_w;
          kvb[u] = reinterpret_cast<const float2*>(rowp + ser * D)[i];
          scb[u] = reinterpret_cast<const float2*>(rowp + half + ser * D)[i];
        }
      }
    };
    if (emit) {
      ec = entry_prefetch(p, b, j, i);
      load_batch(0);
    }
    // this token's row into its ring slot (which holds position pos - nslots, outside the fold)
    float2* dst = reinterpret_cast<float2*>(state_b + (int64_t)(pos % nslots) * state_w);
    dst[i] = kvn[0];
    dst[half / 2 + i] = scn[0];
    if (coff == 2) {
      dst[D / 2 + i] = kvn[1];
      dst[half / 2 + D / 2 + i] = scn[1];
    }
    if (emit) {
      FoldAcc f;
      for (int base = 0; base < nrows; base += FOLD_BATCH) {
        if (base > 0) load_batch(base);
#pragma unroll
        for (int u = 0; u < FOLD_BATCH; ++u) {
          const int idx = base + u;
          if (idx < nrows) {
            const int ser = idx / r, q = (j - ser) * r + idx % r;
            if (q == pos) f.add(ser == 0 ? kvn[0] : kvn[1], ser == 0 ? scn[0] : scn[1]);  // own row
            else f.add(kvb[u], scb[u]);
          }
        }
      }
      entry_finish(p, ec, i, f.a0 / f.s0, f.a1 / f.s1, red, b, j);
    }
    __syncthreads();  // the next token's store may reuse a slot this fold read
  }
}

__global__ void __launch_bounds__(ROW_THREADS) compress_update_kernel(dsv4_compress_update_params p) {
  if (p.after_independent) {
    pdl_launch_dependents();
  } else {
    // while the kernel ahead finishes: the sequence's new rows, its state ring when it folds this step,
    // and a slice of wk (every sequence's index key reads all of it), into L2
    if (threadIdx.x == 0) {
      const int b = blockIdx.x, half = p.coff * D, nslots = p.coff * p.ratio;
      tc::prefetch_l2(p.kv_score + (int64_t)b * p.q_per_seq * 2 * half, (size_t)p.q_per_seq * 2 * half * 4);
      // the ring only when a token of the sequence folds an entry this step (positions read relaxed)
      bool emits = false;
      for (int k = 0; k < p.q_per_seq; ++k) {
        const int pos = tc::ld_relaxed_s32(p.positions + b * p.q_per_seq + k);
        emits |= pos >= 0 && (pos + 1) % p.ratio == 0;
      }
      if (emits) tc::prefetch_l2(p.state + (int64_t)b * nslots * 2 * half, (size_t)nslots * 2 * half * 4);
      if (p.wk != nullptr) {
        const size_t wb = (size_t)p.ik_dim * D * 2, slice = (wb / gridDim.x + 127) / 128 * 128;
        if ((size_t)b * slice < wb)
          tc::prefetch_l2(reinterpret_cast<const uint8_t*>(p.wk) + (size_t)b * slice, min(slice, wb - (size_t)b * slice));
      }
    }
    pdl_wait();
    pdl_launch_dependents();
  }
  compress_update_body(p);
  if (p.after_independent) pdl_wait();  // completes only after the kernel before it
}


// Ratio-128 groups (coff = 1): one 8-CTA cluster per sequence.  Each CTA folds 16 of the group's
// 128 rows into per-channel partial softmax states (max, sum, weighted kv sum) in its shared memory;
// CTA 0 combines the eight partial states through distributed shared memory and finishes the entry.
// Rows of this call's tokens up to the emitting one enter the fold straight from kv_score (+ APE),
// so the fold needs no barrier after CTA 0 stores them; the later tokens' rows, which reuse ring
// slots of the group, are stored after the fold.  Cluster barriers are hardware barriers, not flag
// spins.
constexpr int FOLD_CTAS = 8;
__device__ __forceinline__ void compress_fold_cluster_body(const dsv4_compress_update_params& p) {
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.y, i = threadIdx.x;
  const int r = p.ratio, nslots = r;  // coff == 1
  const int state_w = 2 * D;
  float* state_b = p.state + (int64_t)b * nslots * state_w;
  __shared__ float2 pm[ROW_THREADS], ps[ROW_THREADS], pa[ROW_THREADS];
  __shared__ float red[ROW_THREADS / 32];
  int posk[DSV4_MAX_Q_PER_SEQ];
  int k_emit = -1;
#pragma unroll
  for (int k = 0; k < DSV4_MAX_Q_PER_SEQ; ++k) {
    posk[k] = k < p.q_per_seq ? p.positions[b * p.q_per_seq + k] : -1;
    if (k < p.q_per_seq && k_emit < 0 && posk[k] >= 0 && (posk[k] + 1) % r == 0) k_emit = k;
  }
  const int k_end = k_emit >= 0 ? k_emit + 1 : p.q_per_seq;
  if (k_emit >= 0) {  // cluster-uniform
    const int pos = posk[k_emit];
    const int j = pos / r;
    const int q0 = j * r + rank * (r / FOLD_CTAS);
    EntryCtx ec;
    if (rank == 0) ec = entry_prefetch(p, b, j, i);
    float2 kv[16], sc[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {  // all 32 loads in flight
      const float* rowp = state_b + (int64_t)((q0 + u) % nslots) * state_w;
      kv[u] = reinterpret_cast<const float2*>(rowp)[i];
      sc[u] = reinterpret_cast<const float2*>(rowp + D)[i];
    }
    // rows written by this call's tokens come from kv_score instead of the ring
#pragma unroll
    for (int k = 0; k < DSV4_MAX_Q_PER_SEQ; ++k) {
      const int u = posk[k] - q0;
      if (k <= k_emit && posk[k] >= 0 && u >= 0 && u < 16) {
#pragma unroll
        for (int v = 0; v < 16; ++v)
          if (v == u) new_row_pair(p, b * p.q_per_seq + k, posk[k], 0, i, kv[v], sc[v]);
      }
    }
    if (rank == 0)
      for (int k = 0; k < k_end; ++k) {  // rows of the tokens up to the emitting one, for later calls
        if (posk[k] < 0) {
          if (i == 0) atomicOr(&g_flags_ic, FLAG_PAGE);
          continue;
        }
        float2 a, c;
        new_row_pair(p, b * p.q_per_seq + k, posk[k], 0, i, a, c);
        float2* dst = reinterpret_cast<float2*>(state_b + (int64_t)(posk[k] % nslots) * state_w);
        dst[i] = a;
        dst[D / 2 + i] = c;
      }
    FoldAcc f;
#pragma unroll
    for (int u = 0; u < 16; ++u) f.add(kv[u], sc[u]);
    pm[i] = make_float2(f.m0, f.m1);
    ps[i] = make_float2(f.s0, f.s1);
    pa[i] = make_float2(f.a0, f.a1);
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
      entry_finish(p, ec, i, A0 / S0, A1 / S1, red, b, j);
    }
    cluster.sync();  // the fold has read the ring, and no CTA leaves while CTA 0 reads its shared memory
  } else if (rank == 0) {
    for (int k = 0; k < k_end; ++k) {
      if (posk[k] < 0) {
        if (i == 0) atomicOr(&g_flags_ic, FLAG_PAGE);
        continue;
      }
      float2 a, c;
      new_row_pair(p, b * p.q_per_seq + k, posk[k], 0, i, a, c);
      float2* dst = reinterpret_cast<float2*>(state_b + (int64_t)(posk[k] % nslots) * state_w);
      dst[i] = a;
      dst[D / 2 + i] = c;
    }
  }
  if (rank == 0)
    for (int k = k_end; k < p.q_per_seq; ++k) {  // later tokens (after the fold)
      if (posk[k] < 0) continue;
      float2 a, c;
      new_row_pair(p, b * p.q_per_seq + k, posk[k], 0, i, a, c);
      float2* dst = reinterpret_cast<float2*>(state_b + (int64_t)(posk[k] % nslots) * state_w);
      dst[i] = a;
      dst[D / 2 + i] = c;
    }
}

__global__ void __cluster_dims__(FOLD_CTAS, 1, 1) __launch_bounds__(ROW_THREADS)
    compress_fold_cluster_kernel(dsv4_compress_update_params p) {
  if (p.after_independent) {
    pdl_launch_dependents();
  } else {
    // while the kernel ahead finishes: this CTA's 16 ring rows of the sequence (slots 16 rank .. + 15,
    // whatever the position) when the sequence folds this step, and its new rows, into L2
    if (threadIdx.x == 0) {
      const int b = blockIdx.y, rank = (int)cg::this_cluster().block_rank();
      bool emits = false;  // (positions read relaxed: the ring rows are read only by a fold)
      for (int k = 0; k < p.q_per_seq; ++k) {
        const int pos = tc::ld_relaxed_s32(p.positions + b * p.q_per_seq + k);
        emits |= pos >= 0 && (pos + 1) % p.ratio == 0;
      }
      if (emits)
        tc::prefetch_l2(p.state + ((int64_t)b * p.ratio + rank * (p.ratio / FOLD_CTAS)) * 2 * D,
                        (size_t)(p.ratio / FOLD_CTAS) * 2 * D * 4);
      if (rank == 0) tc::prefetch_l2(p.kv_score + (int64_t)b * p.q_per_seq * 2 * D, (size_t)p.q_per_seq * 2 * D * 4);
    }
    pdl_wait();
    pdl_launch_dependents();
  }
  compress_fold_cluster_body(p);
  if (p.after_independent) pdl_wait();  // completes only after the kernel before it
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
