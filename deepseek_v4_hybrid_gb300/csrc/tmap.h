// Host helpers for TMA tensor maps (driver entry point fetched through the runtime, so the library
// needs no link-time dependency on libcuda) and the device's SM count.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dsv4 {

// 2-D bf16 tensor [rows, cols] (cols innermost, rows `cols * 2` bytes apart), box
// [box_rows, box_cols] with 128-byte swizzle (box_cols * 2 must be 128).
cudaError_t make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                              uint32_t box_rows);

// 2-D tensor of `rows` rows of `cols` elements of type `dt`, consecutive rows `row_bytes` apart (a
// row may be wider than the mapped columns: a column range of packed records), box
// [box_rows, box_cols], swizzle `sw`.  Out-of-range rows read as zeros.
cudaError_t make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t cols, uint64_t rows,
                         uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw);

// Multiprocessor count of the current device.
int num_sms();

// Sets the maximum dynamic shared memory of kernel `fn` to `bytes` on the current device, once per
// device (function attributes belong to each device's context); thread safe.
cudaError_t ensure_max_dynamic_smem(const void* fn, int bytes);

}  // namespace dsv4
