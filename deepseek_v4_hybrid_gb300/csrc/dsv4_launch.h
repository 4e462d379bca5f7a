// Host-side launchers of the decode-step kernels (called by api.cu after validation).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/dsv4.h"

namespace dsv4 {

cudaError_t launch_kv_insert(const dsv4_kv_insert_params& p, cudaStream_t s);
cudaError_t launch_compress_update(const dsv4_compress_update_params& p, cudaStream_t s);

size_t indexer_topk_workspace(const dsv4_indexer_topk_params& p);
cudaError_t launch_indexer_topk(const dsv4_indexer_topk_params& p, cudaStream_t s);

size_t sparse_mla_workspace(const dsv4_sparse_mla_decode_params& p);
cudaError_t launch_sparse_mla_decode(const dsv4_sparse_mla_decode_params& p, cudaStream_t s);

cudaError_t read_flags_insert_compress(uint32_t* f);
cudaError_t read_flags_indexer(uint32_t* f);
cudaError_t read_flags_attention(uint32_t* f);

// Makes `e` the value dsv4_last_cuda_error() reports on this thread.
void record_cuda_error(int e);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace dsv4
