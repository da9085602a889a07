// Host-side TMA tensor-map encoding through the driver entry point (no
// link-time dependency on libcuda).
#include <mutex>

#include "tc.cuh"

namespace dsa {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

void resolve() {
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}
}  // namespace

bool make_tmap_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes,
                  uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_cols) {
  std::call_once(g_once, resolve);
  if (!g_encode) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * (cuuint64_t)elem_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_1d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes,
                  uint64_t n, uint32_t box) {
  // encoded as one row of a 2-D tensor (the row stride only has to be a
  // multiple of 16 bytes; with a single row it is never stepped)
  std::call_once(g_once, resolve);
  if (!g_encode) return false;
  cuuint64_t dims[2] = {n, 1};
  cuuint64_t strides[1] = {((n * (cuuint64_t)elem_bytes) + 15) & ~(cuuint64_t)15};
  cuuint32_t boxd[2] = {box, 1};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dtype, 2, const_cast<void *>(base), dims, strides, boxd, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_3d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes,
                  uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box0, uint32_t box1,
                  uint32_t box2) {
  std::call_once(g_once, resolve);
  if (!g_encode) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * (cuuint64_t)elem_bytes, d0 * d1 * (cuuint64_t)elem_bytes};
  cuuint32_t box[3] = {box0, box1, box2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, dtype, 3, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace dsa
