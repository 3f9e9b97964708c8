// Host-side encoding of the TMA tensor maps over the activations x [M, K]
// (BF16, row-major) and over the units of a blob.  The driver entry point is
// resolved once through the runtime, so libtf needs no link-time dependency
// on libcuda.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/tf.h"
#include "tf_abi.h"

namespace tf {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int encode(const uint16_t* x, int M, int K, unsigned box_k, unsigned box_m, CUtensorMapSwizzle swz,
           CUtensorMap* map) {
  auto enc = encode_fn();
  if (!enc) return TF_ERR_CUDA;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {box_k, box_m};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TF_OK : TF_ERR_CUDA;
}

}  // namespace

int encode_x_map(const uint16_t* x, int M, int K, CUtensorMap* map) {
  return encode(x, M, K, kTileK, (unsigned)M, CU_TENSOR_MAP_SWIZZLE_NONE, map);
}

int encode_y_map(const uint16_t* y, int M, int N, CUtensorMap* map) {
  return encode(y, M, N, 128, 16, CU_TENSOR_MAP_SWIZZLE_NONE, map);
}
int encode_x_map_sw128(const uint16_t* x, int M, int K, int rows, CUtensorMap* map) {
  return encode(x, M, K, 64, (unsigned)rows, CU_TENSOR_MAP_SWIZZLE_128B, map);
}

int encode_units_map(const uint8_t* units, int S, int KT, int unit_bytes, CUtensorMap* map) {
  auto enc = encode_fn();
  if (!enc) return TF_ERR_CUDA;
  const int e = unit_bytes / 8;  // 8-byte elements per unit
  CUresult r;
  if (e <= 256) {
    const cuuint64_t dims[3] = {(cuuint64_t)e, (cuuint64_t)KT, (cuuint64_t)S};
    const cuuint64_t strides[2] = {(cuuint64_t)unit_bytes, (cuuint64_t)KT * unit_bytes};
    const cuuint32_t box[3] = {(cuuint32_t)e, 1, (cuuint32_t)kSlabsPerTile};
    const cuuint32_t estr[3] = {1, 1, 1};
    r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<uint8_t*>(units), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    // INT8 units: two halves of at most 256 elements each
    const cuuint64_t dims[4] = {(cuuint64_t)e / 2, 2, (cuuint64_t)KT, (cuuint64_t)S};
    const cuuint64_t strides[3] = {(cuuint64_t)unit_bytes / 2, (cuuint64_t)unit_bytes,
                                   (cuuint64_t)KT * unit_bytes};
    const cuuint32_t box[4] = {(cuuint32_t)e / 2, 2, 1, (cuuint32_t)kSlabsPerTile};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 4, const_cast<uint8_t*>(units), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS ? TF_OK : TF_ERR_CUDA;
}

}  // namespace tf
