// kda_prep.cu -- K1, the token-parallel chunk kernel.  One 128-thread CTA
// walks (chunk slot, head) work items with a grid-stride loop and writes one
// record per item (kda_chunk.cuh).  FlashKDA's K1 ("FlashKDA: MoonshotAI's
// High-Performance Kimi Delta Attention Kernels", sec. 2.2) has the same
// parallel axes (N x H x chunks); this one adds the W/U factors and stores
// everything the recurrence kernel reads.
#include "kda_chunk.cuh"

namespace kda {

struct PrepSmem {
  ChunkSmem chunk;
  uint8_t raw[4 * 4096];  // q, k, v, g_raw tiles of the current chunk
};

__global__ void __launch_bounds__(128, 4)
chunk_prep_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                  const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ g,
                  const __nv_bfloat16* __restrict__ beta_raw, float scale, float lb_log2e,
                  float eps, const int32_t* __restrict__ cu, int64_t T_total, int H, int N,
                  uint8_t* __restrict__ ws, int64_t n_items) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  PrepSmem& P = *reinterpret_cast<PrepSmem*>(smem_raw);
  RawTiles R;
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    R.lo[x] = P.raw + x * 4096;
    R.hi[x] = P.raw + x * 4096 + 2048;
  }
  const int t = threadIdx.x;
  const int64_t row_stride = static_cast<int64_t>(H) * kDim;
  clear_inverse_workspace(P.chunk, t);
  for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int64_t slot = item / H;
    const int h = static_cast<int>(item - slot * H);
    int n;
    int64_t bos, eos, c;
    if (!locate_slot(cu, T_total, N, slot, n, bos, eos, c)) continue;
    const int64_t t0 = bos + c * kChunk;
    const int nc = static_cast<int>(((eos - t0) < kChunk ? (eos - t0) : kChunk));
    const int64_t base = t0 * row_stride + static_cast<int64_t>(h) * kDim;
    issue_raw_loads(R, q + base, k + base, v + base, g + base, row_stride, nc, t);
    const uint32_t bbits =
        (t < nc) ? __bfloat16_as_ushort(beta_raw[(t0 + t) * H + h]) : 0u;
    build_chunk_record(P.chunk, R, bbits, nc, scale, lb_log2e, eps,
                       ws + static_cast<int64_t>(item) * REC_BYTES, t,
                       [] { chunk_sync(); return true; }, [] {});
  }
}

cudaError_t launch_chunk_prep(const void* q, const void* k, const void* v, const void* g,
                              const void* beta_raw, float scale, float lower_bound, float eps,
                              const int32_t* cu, int64_t T_total, int H, int N, void* ws,
                              int sm_count, cudaStream_t stream) {
  const int64_t n_items = slot_count(T_total, N) * H;
  const int smem = static_cast<int>(sizeof(PrepSmem));
  static bool attr_done = false;  // per process; the attribute is per function
  if (!attr_done) {
    cudaError_t e =
        cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chunk_prep_kernel, 128, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t grid = (n_items < static_cast<int64_t>(sm_count) * per_sm ? n_items : static_cast<int64_t>(sm_count) * per_sm);
  if (grid <= 0) return cudaSuccess;
  chunk_prep_kernel<<<static_cast<unsigned>(grid), 128, smem, stream>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), static_cast<const __nv_bfloat16*>(g),
      static_cast<const __nv_bfloat16*>(beta_raw), scale, lower_bound * 1.4426950408889634f, eps,
      cu, T_total, H, N, static_cast<uint8_t*>(ws), n_items);
  return cudaGetLastError();
}

}  // namespace kda
