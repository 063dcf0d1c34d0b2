// Host helpers shared by the TMA kernels' launchers: the driver's tensor-map
// encoder (looked up once through the runtime, so the library links no
// libcuda) and the 3-D map over one layer's paged cache.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

namespace pkv {

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    cudaGetLastError();
  });
  return fn;
}

// 3-D map over one layer's cache viewed as [rows = num_blocks*block_size]
// [num_kv_heads][head_dim]; box = [box_rows][1][128 bytes of one row], 128-byte
// swizzle (the smem tile layout the fragment addressing assumes).  16-bit
// caches take two boxes per row (64 elements each), FP8 caches one.
inline bool make_map(CUtensorMap* m, const void* base, int head_dim, int num_kv_heads, int64_t rows,
              int box_rows, bool fp8) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t esz = fp8 ? 1 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(num_kv_heads),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * esz,
                           static_cast<cuuint64_t>(head_dim) * esz * num_kv_heads};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / esz), 1u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                  const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace pkv
