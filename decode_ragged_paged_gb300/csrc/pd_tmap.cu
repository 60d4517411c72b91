// pd_tmap.cu -- host-side construction of TMA tensor maps (CUtensorMap) for the
// query rows and the HND page pools. The driver entry point is looked up once
// through the runtime, so the library links only against libcudart.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "pd_internal.h"

namespace pd {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

CUtensorMapDataType tma_dtype(int32_t dtype) {
  return dtype == PD_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
}

}  // namespace

// HND pool [num_pages][hkv][page_size][head_dim] as a 4-D tensor {head_dim,
// page_size, hkv, num_pages} (innermost first), box {box_cols, box_rows, 1, 1};
// NHD pool [num_pages][page_size][hkv][head_dim] as {head_dim, hkv, page_size,
// num_pages}, box {box_cols, 1, box_rows, 1}. Either way one box is box_rows
// slots x box_cols elements of one (page, head), landing in shared memory as
// box_rows rows of box_cols elements; coordinates follow the tensor's order.
bool make_pool_map(CUtensorMap* map, const void* pool, int32_t dtype, int32_t num_pages, int32_t hkv,
                   int32_t page_size, int32_t head_dim, int32_t box_cols, int32_t box_rows, bool swizzle128,
                   bool nhd) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const int es = dtype == PD_BF16 ? 2 : 4;
  const cuuint64_t row = (cuuint64_t)head_dim * es;
  cuuint64_t dims[4] = {(cuuint64_t)head_dim, (cuuint64_t)page_size, (cuuint64_t)hkv, (cuuint64_t)num_pages};
  cuuint64_t strides[3] = {row, (cuuint64_t)page_size * row, (cuuint64_t)hkv * page_size * row};
  cuuint32_t box[4] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1, 1};
  if (nhd) {
    dims[1] = (cuuint64_t)hkv;
    dims[2] = (cuuint64_t)page_size;
    strides[0] = row;                     // next head
    strides[1] = (cuuint64_t)hkv * row;   // next slot
    box[1] = 1;
    box[2] = (cuuint32_t)box_rows;
  }
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, tma_dtype(dtype), 4, const_cast<void*>(pool), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// q / o rows [total][hq][head_dim] as a 3-D tensor {head_dim, hq, total}; one box
// = box_rows consecutive rows of box_heads consecutive heads, box_cols elements
// wide, laid out (row, head)-major in shared memory.
bool make_rows_map(CUtensorMap* map, const void* base, int32_t dtype, int32_t total, int32_t hq, int32_t head_dim,
                   int32_t box_cols, int32_t box_rows, bool swizzle128, int32_t box_heads) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const int es = dtype == PD_BF16 ? 2 : 4;
  cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)hq, (cuuint64_t)total};
  cuuint64_t strides[2] = {(cuuint64_t)head_dim * es, (cuuint64_t)hq * head_dim * es};
  cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_heads, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, tma_dtype(dtype), 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace pd
