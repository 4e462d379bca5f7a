// Host-side launchers of the decode-step kernels (called by api.cu after validation).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/dsv4.h"

namespace dsv4 {

cudaError_t launch_kv_insert(const dsv4_kv_insert_params& p, cudaStream_t s);
cudaError_t launch_qnorm_rope_kv_insert(const dsv4_qnorm_rope_kv_insert_params& p, cudaStream_t s);
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

// Counts one kernel enqueued by the library (dsv4_kernel_launches()); `e` is the launch's status.
cudaError_t count_launch(cudaError_t e);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace dsv4

namespace dsv4 {

// Programmatic dependent launch: the next kernel on the stream may start (and run its prologue)
// while this one finishes; it must call pdl_wait() before touching anything an earlier kernel
// writes.  Every kernel of the library calls pdl_wait() before its first dependent access, so the
// order of the stream is kept transitively.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// Start of a kernel that is either after_independent (its work needs nothing from the kernels ahead:
// their dependents may start at once, and it waits for them only before exiting) or not (it waits
// first and lets its own dependents start only then, so that when a kernel after it starts, every
// kernel before this one has finished).
__device__ __forceinline__ void pdl_start(bool after_independent) {
  if (after_independent) {
    pdl_launch_dependents();
  } else {
    pdl_wait();
    pdl_launch_dependents();
  }
}

// `pdl` false launches plainly (the kernel's pdl_wait() then returns at once).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return count_launch(cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...));
}

}  // namespace dsv4
