// Host helpers for the tcgen05 GEMM: TMA tensor-map encoding and the SM count.
#include <mutex>

#include "moe_internal.h"

namespace moe {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int encode3d(CUtensorMap* map, const void* base, const cuuint64_t dims[3],
             const cuuint64_t strides[2], const cuuint32_t box[3]) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return MOE_ERR_CUDA;
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

// bf16 tensor [groups][rows][k_extent] read in K-major boxes of 64 (K) x box_rows.
int encode_map_kmajor(CUtensorMap* map, const void* base, uint64_t k_extent, uint64_t rows,
                      uint64_t groups, uint32_t box_rows) {
  const cuuint64_t dims[3] = {k_extent, rows, groups};
  const cuuint64_t strides[2] = {k_extent * 2, k_extent * rows * 2};
  const cuuint32_t box[3] = {64, box_rows, 1};
  return encode3d(map, base, dims, strides, box);
}

// bf16 tensor [groups][k_rows][mn_extent] read in MN-major boxes of 64 (MN) x 64 (K).
int encode_map_mnmajor(CUtensorMap* map, const void* base, uint64_t mn_extent, uint64_t k_rows,
                       uint64_t groups) {
  const cuuint64_t dims[3] = {mn_extent, k_rows, groups};
  const cuuint64_t strides[2] = {mn_extent * 2, mn_extent * k_rows * 2};
  const cuuint32_t box[3] = {64, 64, 1};
  return encode3d(map, base, dims, strides, box);
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  static int cache[64] = {0};
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 1;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev < 64) cache[dev] = n;
  return n;
}

}  // namespace moe
