// Tensor-map encoding through the driver's cuTensorMapEncodeTiled, resolved
// once through the runtime's entry-point query (no link-time libcuda).
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.h"

namespace moe {

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

CUresult encode_tensor_map_nd(CUtensorMap* m, CUtensorMapDataType dt, void* base, int rank,
                              const uint64_t* dims, const uint64_t* strides_bytes,
                              const uint32_t* box, CUtensorMapSwizzle swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (enc == nullptr) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) { d[i] = dims[i]; b[i] = box[i]; e[i] = 1; }
  for (int i = 0; i + 1 < rank; ++i) st[i] = strides_bytes[i];
  return enc(m, dt, static_cast<cuuint32_t>(rank), base, d, st, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

CUresult encode_gate_up_map(CUtensorMap* m, CUtensorMapDataType dt, const void* w13, int n,
                            int inter, int d, size_t elem_bytes, uint32_t box_k,
                            uint32_t box_mats, uint32_t box_rows) {
  const uint64_t dims[4] = {static_cast<uint64_t>(d), static_cast<uint64_t>(inter), 2,
                            static_cast<uint64_t>(n)};
  const uint64_t row = static_cast<uint64_t>(d) * elem_bytes;
  const uint64_t strides[3] = {row, row * inter, row * inter * 2};
  const uint32_t box[4] = {box_k, box_rows, box_mats, 1};
  return encode_tensor_map_nd(m, dt, const_cast<void*>(w13), 4, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B);
}

CUresult encode_gate_up_map_interleaved(CUtensorMap* m, CUtensorMapDataType dt, const void* w13,
                                        int n, int inter, int d, size_t elem_bytes,
                                        uint32_t box_k) {
  const uint64_t dims[5] = {static_cast<uint64_t>(d), 64, 2, static_cast<uint64_t>(inter / 64),
                            static_cast<uint64_t>(n)};
  const uint64_t row = static_cast<uint64_t>(d) * elem_bytes;
  const uint64_t strides[4] = {row, row * inter, row * 64, row * inter * 2};
  const uint32_t box[5] = {box_k, 64, 2, 2, 1};
  return encode_tensor_map_nd(m, dt, const_cast<void*>(w13), 5, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B);
}

CUresult encode_tensor_map_2d(CUtensorMap* m, CUtensorMapDataType dt, void* base, uint64_t inner,
                              uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                              uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (enc == nullptr) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace moe
