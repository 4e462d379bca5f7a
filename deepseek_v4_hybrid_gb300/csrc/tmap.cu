// TMA tensor-map encoding and device queries shared by the tensor-core kernels.
#include <mutex>

#include "tmap.h"

namespace dsv4 {

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_once;
EncodeTiledFn g_encode = nullptr;
cudaError_t g_encode_err = cudaSuccess;

void load_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (g_encode_err == cudaSuccess && q != cudaDriverEntryPointSuccess) g_encode_err = cudaErrorNotSupported;
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
}
}  // namespace

cudaError_t make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                              uint32_t box_rows) {
  std::call_once(g_once, load_encode);
  if (g_encode_err != cudaSuccess) return g_encode_err;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
                         uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw) {
  std::call_once(g_once, load_encode);
  if (g_encode_err != cudaSuccess) return g_encode_err;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  CUresult r = g_encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {
constexpr int kMaxDevices = 64;
constexpr int kMaxKernels = 16;
std::mutex g_dev_mutex;
int g_sms[kMaxDevices] = {0};
struct SmemAttr {
  const void* fn;
  int bytes;
};
SmemAttr g_smem_attr[kMaxDevices][kMaxKernels] = {};
}  // namespace

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (g_sms[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_sms[dev] = n > 0 ? n : 1;
  }
  return g_sms[dev];
}

cudaError_t ensure_max_dynamic_smem(const void* fn, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  SmemAttr* tab = g_smem_attr[dev];
  int i = 0;
  for (; i < kMaxKernels && tab[i].fn != nullptr; ++i)
    if (tab[i].fn == fn && tab[i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  for (int k = 0; k < kMaxKernels; ++k)
    if (tab[k].fn == fn) {
      tab[k].bytes = bytes;
      return cudaSuccess;
    }
  if (i < kMaxKernels) tab[i] = SmemAttr{fn, bytes};
  return cudaSuccess;
}

}  // namespace dsv4
