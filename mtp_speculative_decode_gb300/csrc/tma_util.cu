// Tensor-map (TMA descriptor) encoding through the driver entry point, so the
// library needs no link-time dependency on libcuda.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace mtpsd {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
  }
  return fn;
}

bool tma_available() { return encode_fn() != nullptr; }

bool make_tma_2d(void* map, int dtype_u8_or_bf16, const void* base, uint64_t inner_elems, uint64_t rows,
                 uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, bool l2_256) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner_elems, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUtensorMapDataType dt = dtype_u8_or_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r = fn((CUtensorMap*)map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  l2_256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Rows of row_bytes uint8 values as a [rows, row_bytes] tensor map without swizzle, for one-row boxes of
// box_bytes bytes (tile::gather4 loads; box_bytes and row_bytes multiples of 16).
bool make_tma_2d_plain_u8(void* map, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {box_bytes, 1};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn((CUtensorMap*)map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Float32 vector as a [1, n_elems] tensor map without swizzle (rank 2 with a single row, so the
// encoding has a stride to check; box of box_elems x 1, box_elems * 4 a multiple of 16 bytes; a copy's
// start coordinate must be a multiple of 4 elements).  Elements past n_elems read as 0.
bool make_tma_1d_f32(void* map, const void* base, uint64_t n_elems, uint32_t box_elems) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)n_elems, 1};
  cuuint64_t strides[1] = {(cuuint64_t)((n_elems * 4 + 15) / 16 * 16)};
  cuuint32_t box[2] = {box_elems, 1};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn((CUtensorMap*)map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tensor map for TMA stores from shared memory: rank 2 or 3, bf16 or float32, 128-byte swizzle
// (the box's inner extent must be 128 bytes).  dims[0] is the contiguous dimension; strides are the
// byte strides of dims 1.. (multiples of 16).
bool make_tma_store_map(void* map, bool f32, const void* base, int rank, const uint64_t* dims,
                        const uint64_t* strides, const uint32_t* box) {
  auto fn = encode_fn();
  if (!fn || rank < 2 || rank > 3) return false;
  cuuint64_t d[3], st[2];
  cuuint32_t bx[3], estr[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = (cuuint64_t)dims[i];
    bx[i] = (cuuint32_t)box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) st[i] = (cuuint64_t)strides[i];
  CUresult r = fn((CUtensorMap*)map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  (cuuint32_t)rank, const_cast<void*>(base), d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace mtpsd
