// C ABI entry points: host-side argument validation, then the kernel launches.
// The declarations, argument meanings and error behaviour are documented in include/dsv4.h.
#include <atomic>
#include <cstdint>
#include <cstring>

#include "dsv4_common.cuh"
#include "dsv4_launch.h"

using namespace dsv4;

namespace {

thread_local int g_last_cuda_error = 0;
std::atomic<unsigned long long> g_kernel_launches{0};

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return DSV4_OK;
  g_last_cuda_error = (int)e;
  return DSV4_ERR_CUDA;
}

bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

bool latent_cache_dtype(int d) { return d == DSV4_F32 || d == DSV4_BF16 || d == DSV4_FP8_DS_MLA; }
bool act_dtype(int d) { return d == DSV4_F32 || d == DSV4_BF16; }

#define CHECK(cond, code) \
  do {                    \
    if (!(cond)) return (code); \
  } while (0)

}  // namespace

void dsv4::record_cuda_error(int e) { g_last_cuda_error = e; }

cudaError_t dsv4::count_launch(cudaError_t e) {
  if (e == cudaSuccess) g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  return e;
}

extern "C" {

int dsv4_abi_version(void) { return DSV4_ABI_VERSION; }

uint64_t dsv4_kernel_launches(void) { return g_kernel_launches.load(std::memory_order_relaxed); }

const char* dsv4_status_string(int s) {
  switch (s) {
    case DSV4_OK: return "ok";
    case DSV4_ERR_INVALID: return "invalid argument";
    case DSV4_ERR_UNSUPPORTED: return "unsupported dtype or shape";
    case DSV4_ERR_CUDA: return "CUDA error";
    case DSV4_ERR_BOUNDS: return "a kernel skipped an out-of-range index";
    case DSV4_ERR_TIMEOUT: return "a kernel gave up a bounded wait (outputs unspecified)";
  }
  return "unknown status";
}

int dsv4_last_cuda_error(void) { return g_last_cuda_error; }

int dsv4_read_device_flags(uint32_t* flags) {
  CHECK(flags != nullptr, DSV4_ERR_INVALID);
  *flags = 0;
  int st = cuda_status(cudaDeviceSynchronize());
  if (st != DSV4_OK) return st;
  st = cuda_status(read_flags_insert_compress(flags));
  if (st != DSV4_OK) return st;
  st = cuda_status(read_flags_indexer(flags));
  if (st != DSV4_OK) return st;
  st = cuda_status(read_flags_attention(flags));
  if (st != DSV4_OK) return st;
  if (*flags & 4u) return DSV4_ERR_TIMEOUT;
  return *flags ? DSV4_ERR_BOUNDS : DSV4_OK;
}

int dsv4_kv_insert(const dsv4_kv_insert_params* p, dsv4_stream_t stream) {
  CHECK(p != nullptr && p->struct_size == sizeof(dsv4_kv_insert_params), DSV4_ERR_INVALID);
  CHECK(p->T >= 0 && p->page_size > 0 && p->num_pages >= 0, DSV4_ERR_INVALID);
  CHECK(act_dtype(p->kv_dtype), DSV4_ERR_UNSUPPORTED);
  CHECK(latent_cache_dtype(p->cache_dtype), DSV4_ERR_UNSUPPORTED);
  if (p->T == 0) return DSV4_OK;
  CHECK(p->kv_new && p->slot_mapping && p->cache, DSV4_ERR_INVALID);
  CHECK(aligned(p->kv_new, 8) && aligned(p->cache, 16) && aligned(p->slot_mapping, 8), DSV4_ERR_INVALID);
  CHECK(p->cos_sin == nullptr || (p->positions != nullptr && p->max_pos > 0), DSV4_ERR_INVALID);
  return cuda_status(launch_kv_insert(*p, (cudaStream_t)stream));
}

int dsv4_qnorm_rope_kv_insert(const dsv4_qnorm_rope_kv_insert_params* p, dsv4_stream_t stream) {
  CHECK(p != nullptr && p->struct_size == sizeof(dsv4_qnorm_rope_kv_insert_params), DSV4_ERR_INVALID);
  CHECK(p->T >= 0 && p->page_size > 0 && p->num_pages >= 0, DSV4_ERR_INVALID);
  CHECK(p->H >= 1 && p->H_pad >= p->H && p->H_pad <= 1024, DSV4_ERR_INVALID);
  CHECK(act_dtype(p->act_dtype), DSV4_ERR_UNSUPPORTED);
  CHECK(latent_cache_dtype(p->cache_dtype), DSV4_ERR_UNSUPPORTED);
  if (p->T == 0) return DSV4_OK;
  CHECK(p->q && p->q_out && p->kv_new && p->slot_mapping && p->cache, DSV4_ERR_INVALID);
  CHECK(aligned(p->q, 16) && aligned(p->q_out, 16) && aligned(p->kv_new, 8) && aligned(p->cache, 16) &&
            aligned(p->slot_mapping, 8) && aligned(p->q_norm_weight, 4),
        DSV4_ERR_INVALID);
  const bool rope = p->apply_q_rope || p->apply_kv_rope;
  CHECK(!rope || (p->positions != nullptr && p->cos_sin != nullptr && p->max_pos > 0), DSV4_ERR_INVALID);
  // q_out is q itself (in place, same head count) or a separate buffer
  const size_t esz = p->act_dtype == DSV4_F32 ? 4 : 2;
  const uintptr_t q0 = reinterpret_cast<uintptr_t>(p->q), q1 = q0 + (size_t)p->T * p->H * D * esz;
  const uintptr_t o0 = reinterpret_cast<uintptr_t>(p->q_out), o1 = o0 + (size_t)p->T * p->H_pad * D * esz;
  CHECK((q0 == o0 && p->H_pad == p->H) || o1 <= q0 || q1 <= o0, DSV4_ERR_INVALID);
  return cuda_status(launch_qnorm_rope_kv_insert(*p, (cudaStream_t)stream));
}

int dsv4_padded_num_q_heads(int H, int cache_dtype) {
  if (H < 1 || !latent_cache_dtype(cache_dtype)) return -1;
  return cache_dtype == DSV4_F32 ? H : (H + 63) / 64 * 64;
}

int dsv4_compress_update(const dsv4_compress_update_params* p, dsv4_stream_t stream) {
  CHECK(p != nullptr && p->struct_size == sizeof(dsv4_compress_update_params), DSV4_ERR_INVALID);
  CHECK(p->B >= 0 && p->q_per_seq >= 1 && p->q_per_seq <= DSV4_MAX_Q_PER_SEQ, DSV4_ERR_INVALID);
  CHECK((int64_t)p->B * p->q_per_seq == p->T, DSV4_ERR_INVALID);
  CHECK((p->ratio == 4 && p->coff == 2) || (p->ratio == 128 && p->coff == 1) || (p->ratio == 4 && p->coff == 1),
        DSV4_ERR_UNSUPPORTED);
  CHECK(p->q_per_seq <= p->ratio, DSV4_ERR_UNSUPPORTED);
  CHECK(latent_cache_dtype(p->cache_dtype), DSV4_ERR_UNSUPPORTED);
  CHECK(p->page_size > 0 && p->num_pages >= 0 && p->max_pages_per_seq > 0 && p->max_pos > 0, DSV4_ERR_INVALID);
  CHECK(p->eps >= 0.f, DSV4_ERR_INVALID);
  if (p->B == 0) return DSV4_OK;
  CHECK(p->kv_score && p->positions && p->state && p->norm_weight && p->cos_sin && p->main_cache && p->block_table,
        DSV4_ERR_INVALID);
  CHECK(aligned(p->kv_score, 8) && aligned(p->state, 8) && aligned(p->norm_weight, 8) &&
            aligned(p->main_cache, 16) && (p->ape == nullptr || aligned(p->ape, 8)),
        DSV4_ERR_INVALID);
  if (p->wk != nullptr) {
    CHECK(p->ik_dim == 64 || p->ik_dim == 128, DSV4_ERR_UNSUPPORTED);
    CHECK(p->ik_dtype == DSV4_F32 || p->ik_dtype == DSV4_BF16 || p->ik_dtype == DSV4_I8_ROWSCALE ||
              p->ik_dtype == DSV4_MXFP4,
          DSV4_ERR_UNSUPPORTED);
    CHECK(p->ik_norm_weight && p->ik_cache && p->ik_block_table && p->ik_max_pages > 0 && p->ik_num_pages >= 0 &&
              p->ik_eps >= 0.f,
          DSV4_ERR_INVALID);
    CHECK(aligned(p->wk, 4) && aligned(p->ik_norm_weight, 4) && aligned(p->ik_cache, 16), DSV4_ERR_INVALID);
  }
  return cuda_status(launch_compress_update(*p, (cudaStream_t)stream));
}

size_t dsv4_indexer_topk_workspace_bytes(const dsv4_indexer_topk_params* p) {
  if (p == nullptr || p->struct_size != sizeof(dsv4_indexer_topk_params) || p->ratio <= 0 || p->T < 0 ||
      p->max_context < 0)
    return 0;
  return indexer_topk_workspace(*p);
}

int dsv4_indexer_topk(const dsv4_indexer_topk_params* p, dsv4_stream_t stream) {
  CHECK(p != nullptr && p->struct_size == sizeof(dsv4_indexer_topk_params), DSV4_ERR_INVALID);
  CHECK(p->B >= 0 && p->q_per_seq >= 1 && p->q_per_seq <= DSV4_MAX_Q_PER_SEQ, DSV4_ERR_INVALID);
  CHECK((int64_t)p->B * p->q_per_seq == p->T, DSV4_ERR_INVALID);
  CHECK(p->ratio > 0 && p->page_size > 0 && p->max_pages_per_seq > 0 && p->num_pages >= 0, DSV4_ERR_INVALID);
  CHECK(p->topk > 0 && p->topk <= 16384 && p->max_context >= 0, DSV4_ERR_INVALID);
  CHECK(act_dtype(p->q_dtype), DSV4_ERR_UNSUPPORTED);
  CHECK(p->k_dtype == DSV4_F32 || p->k_dtype == DSV4_BF16 || p->k_dtype == DSV4_I8_ROWSCALE ||
            (p->k_dtype == DSV4_MXFP4 && p->head_dim % 32 == 0),
        DSV4_ERR_UNSUPPORTED);
  CHECK(p->n_heads >= 1 && p->n_heads <= 128 && p->head_dim >= 16 && p->head_dim <= 256 && p->head_dim % 16 == 0,
        DSV4_ERR_UNSUPPORTED);
  CHECK((int64_t)p->q_per_seq * p->n_heads <= 256, DSV4_ERR_UNSUPPORTED);
  CHECK(p->max_context / p->ratio <= (1 << 20), DSV4_ERR_UNSUPPORTED);
  if (p->cand_block_size != 0) {
    const int cb = p->cand_block_size;
    CHECK(cb >= 128 && cb <= 65536 && (cb & (cb - 1)) == 0, DSV4_ERR_INVALID);
    CHECK(p->cand_topk >= 1 && p->cand_topk <= 64 && (p->cand_write == 0 || p->cand_write == 1), DSV4_ERR_INVALID);
    CHECK(p->T == 0 || (p->cand_blocks != nullptr && aligned(p->cand_blocks, 4)), DSV4_ERR_INVALID);
  }
  if (p->T == 0) return DSV4_OK;
  CHECK(p->q && p->weights && p->k_cache && p->block_table && p->positions && p->topk_idx, DSV4_ERR_INVALID);
  CHECK(aligned(p->q, 16) && aligned(p->k_cache, 16) && aligned(p->weights, 4), DSV4_ERR_INVALID);
  CHECK(p->workspace != nullptr && aligned(p->workspace, 256), DSV4_ERR_INVALID);
  CHECK(p->workspace_bytes >= indexer_topk_workspace(*p), DSV4_ERR_INVALID);
  return cuda_status(launch_indexer_topk(*p, (cudaStream_t)stream));
}

size_t dsv4_sparse_mla_decode_workspace_bytes(const dsv4_sparse_mla_decode_params* p) {
  if (p == nullptr || p->struct_size != sizeof(dsv4_sparse_mla_decode_params) || p->T < 0 || p->H <= 0 ||
      p->max_context < 0 || p->ratio < 0)
    return 0;
  return sparse_mla_workspace(*p);
}

int dsv4_sparse_mla_decode(const dsv4_sparse_mla_decode_params* p, dsv4_stream_t stream) {
  CHECK(p != nullptr && p->struct_size == sizeof(dsv4_sparse_mla_decode_params), DSV4_ERR_INVALID);
  CHECK(p->B >= 0 && p->q_per_seq >= 1 && p->q_per_seq <= DSV4_MAX_Q_PER_SEQ, DSV4_ERR_INVALID);
  CHECK((int64_t)p->B * p->q_per_seq == p->T, DSV4_ERR_INVALID);
  CHECK(p->H >= 1 && p->H <= 128, DSV4_ERR_UNSUPPORTED);
  CHECK(p->page_size > 0 && p->window >= 1 && p->ratio >= 0 && p->max_context >= 0, DSV4_ERR_INVALID);
  CHECK(p->swa_max_pages > 0 && p->swa_num_pages >= 0, DSV4_ERR_INVALID);
  CHECK(act_dtype(p->q_dtype) && act_dtype(p->out_dtype), DSV4_ERR_UNSUPPORTED);
  CHECK(latent_cache_dtype(p->cache_dtype), DSV4_ERR_UNSUPPORTED);
  CHECK(p->topk_idx == nullptr || (p->topk > 0 && p->topk <= 16384), DSV4_ERR_INVALID);
  if (p->T == 0) return DSV4_OK;
  CHECK(p->q && p->positions && p->swa_cache && p->swa_block_table && p->out, DSV4_ERR_INVALID);
  if (p->ratio > 0) CHECK(p->main_cache && p->main_block_table && p->main_max_pages > 0, DSV4_ERR_INVALID);
  CHECK(aligned(p->q, 16) && aligned(p->swa_cache, 16) && aligned(p->out, 16), DSV4_ERR_INVALID);
  if (p->ratio > 0) CHECK(aligned(p->main_cache, 16), DSV4_ERR_INVALID);
  CHECK(p->workspace != nullptr && aligned(p->workspace, 256), DSV4_ERR_INVALID);
  CHECK(p->workspace_bytes >= sparse_mla_workspace(*p), DSV4_ERR_INVALID);
  return cuda_status(launch_sparse_mla_decode(*p, (cudaStream_t)stream));
}

}  // extern "C"
