// Host-side construction of TMA tensor maps for the [tokens, heads, d] tensors.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace marble {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// View a row-major [n_tokens, heads, d] tensor as the 3-D TMA tensor (d, token, head) and
// describe a box of (box_d elements of d) x (box_rows tokens) x (1 head).  bf16 boxes use
// 128-byte swizzle (box_d = 64); fp32 boxes use 128-byte swizzle with box_d = 32.
inline bool make_rows_map(CUtensorMap* map, const void* base, CUtensorMapDataType dtype,
                          int elem_bytes, int64_t n_tokens, int heads, int d, int box_d,
                          int box_rows, CUtensorMapSwizzle swizzle) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)n_tokens, (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)heads * d * elem_bytes, (cuuint64_t)d * elem_bytes};
  cuuint32_t box[3] = {(cuuint32_t)box_d, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(map, dtype, 3, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace marble
