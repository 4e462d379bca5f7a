// dsv4_indexer_topk_noalloc: the indexer + top-k call for callers that cannot allocate device
// memory, e.g. code running inside another runtime's memory pool or allocator-free plugin hosts
// where a cudaMalloc (or a caching allocator) is not available or not allowed.
//
// The scratch the indexer needs (the per-token score rows) lives in one file-scope device array of
// fixed size, DSV4_NOALLOC_SCRATCH_BYTES, that every GPU loading this library keeps until the
// process exits.  Host code never hands the array's symbol to a kernel: on first use on a device
// (with that device current) the entry point asks the runtime for the array's device address with
// cudaGetSymbolAddress and passes that address on.  All calls on a device share the one array,
// so calls whose kernels overlap on the GPU race on it.
#include <mutex>

#include "dsv4_common.cuh"
#include "dsv4_launch.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[DSV4_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int dsv4_indexer_topk_noalloc(const dsv4_indexer_topk_params* p, dsv4_stream_t stream) {
  if (p == nullptr || p->struct_size != sizeof(dsv4_indexer_topk_params)) return DSV4_ERR_INVALID;
  if (p->ratio <= 0 || p->T < 0 || p->max_context < 0) return DSV4_ERR_INVALID;
  const size_t need = dsv4::indexer_topk_workspace(*p);
  if (need > (size_t)DSV4_NOALLOC_SCRATCH_BYTES) return DSV4_ERR_INVALID;  // problem too large for the array
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    dsv4::record_cuda_error((int)e);
    return DSV4_ERR_CUDA;
  }
  dsv4_indexer_topk_params q = *p;
  q.workspace = scratch;
  q.workspace_bytes = DSV4_NOALLOC_SCRATCH_BYTES;
  q.workspace_zeroed = 0;  // the array is shared by every call: always cleared first
  return dsv4_indexer_topk(&q, stream);
}
