// host_util.h -- host-side helpers shared by the library's translation units:
// CUDA error mapping and TMA descriptor encoding.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <cstdio>
#include <cstdlib>

#include "../../include/mk.h"

namespace mk {

inline bool log_enabled() {
  const char* e = std::getenv("MK_LOG");
  return e && e[0] == '1';
}

#define MK_CUDA_TRY(expr)                                              \
  do {                                                                 \
    cudaError_t _e = (expr);                                           \
    if (_e != cudaSuccess) {                                           \
      if (::mk::log_enabled())                                         \
        std::fprintf(stderr, "mk: %s failed: %s\n", #expr,             \
                     cudaGetErrorString(_e));                          \
      return _e == cudaErrorMemoryAllocation ? MK_ERR_OOM : MK_ERR_CUDA; \
    }                                                                  \
  } while (0)

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion,
                                    CUtensorMapFloatOOBfill);

inline PFN_encodeTiled get_encode_fn() {
  static PFN_encodeTiled fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled>(p);
  }
  return fn;
}

// 2-D tiled map over a row-major [rows][inner] matrix of `elem_bytes`-byte
// elements; box = box_inner x box_rows, 128-byte swizzle, out-of-range
// elements read as zero.
inline mk_status encode_tmap_2d(CUtensorMap* map, const void* base, int elem_bytes,
                                uint64_t inner, uint64_t rows, uint32_t box_inner,
                                uint32_t box_rows) {
  PFN_encodeTiled fn = get_encode_fn();
  if (!fn) return MK_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0) return MK_ERR_INVALID_ARG;
  if ((inner * elem_bytes) % 16 != 0) return MK_ERR_INVALID_ARG;
  CUtensorMapDataType dt = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                           : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * static_cast<uint64_t>(elem_bytes)};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MK_OK : MK_ERR_INVALID_ARG;
}

}  // namespace mk
