// kda_tma.cu -- host side of the raw-tile tensor maps (kda_tma.cuh): the
// driver's cuTensorMapEncodeTiled, reached through the runtime's entry-point
// query (libkda links only the runtime).
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "kda_tma.cuh"

namespace kda {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    else
      cudaGetLastError();
  });
  return g_encode;
}

}  // namespace

cudaError_t make_raw_map(CUtensorMap* map, const void* base, int64_t T_total, int H) {
  if (T_total < 1 || T_total >= (static_cast<int64_t>(1) << 31) || H < 1) return cudaErrorInvalidValue;
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(T_total)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kDim) * 2,
                                 static_cast<cuuint64_t>(H) * kDim * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(RAW_ROW / 2), 1, kChunk};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_raw_maps(RawMaps* maps, const void* q, const void* k, const void* v,
                          const void* g, int64_t T_total, int H, bool gate_scalar) {
  std::memset(maps, 0, sizeof(RawMaps));
  if (T_total == 0) return cudaSuccess;
  cudaError_t e = make_raw_map(&maps->q, q, T_total, H);
  if (e == cudaSuccess) e = make_raw_map(&maps->k, k, T_total, H);
  if (e == cudaSuccess) e = make_raw_map(&maps->v, v, T_total, H);
  if (e == cudaSuccess && !gate_scalar) e = make_raw_map(&maps->g, g, T_total, H);
  return e;
}

}  // namespace kda
