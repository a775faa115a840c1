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
  uint8_t raw[QKG_BYTES];  // q, k, g_raw tiles
  uint8_t vt[V_BYTES];     // v tile
};

__global__ void __launch_bounds__(128, 4)
chunk_prep_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                  const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ g,
                  const __nv_bfloat16* __restrict__ beta_raw, float scale, float lb_log2e,
                  float eps, const int32_t* __restrict__ cu, int64_t T_total, int H, int N,
                  uint8_t* __restrict__ ws, int64_t n_items, int gate_scalar) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  PrepSmem& P = *reinterpret_cast<PrepSmem*>(smem_raw);
  const int t = threadIdx.x;
  const int64_t row_stride = static_cast<int64_t>(H) * kDim;
  const TileLoader loader(t, row_stride);

  // the next used slot at or after `item` on this CTA's grid stride
  struct Item {
    int64_t item, base, t0;
    int h, nc;
  };
  auto find = [&](int64_t item, Item& it) -> bool {
    for (; item < n_items; item += gridDim.x) {
      const int64_t slot = item / H;
      const int h = static_cast<int>(item - slot * H);
      int n;
      int64_t bos, eos, c;
      if (locate_slot(cu, T_total, N, slot, n, bos, eos, c)) {
        it.item = item;
        it.h = h;
        it.t0 = bos + c * kChunk;
        it.nc = static_cast<int>(((eos - it.t0) < kChunk ? (eos - it.t0) : kChunk));
        it.base = it.t0 * row_stride + static_cast<int64_t>(h) * kDim;
        return true;
      }
    }
    return false;
  };
  auto start = [&](const Item& it) -> uint32_t {
    if (gate_scalar)
      issue_qkg_loads(loader, P.raw, q + it.base, k + it.base, g + it.t0 * H + it.h, it.nc, H);
    else
      issue_qkg_loads(loader, P.raw, q + it.base, k + it.base, g + it.base, it.nc);
    return (t < it.nc) ? __bfloat16_as_ushort(beta_raw[(it.t0 + t) * H + it.h]) : 0u;
  };

  Item cur, nxt;
  bool have = find(blockIdx.x, cur);
  uint32_t bbits = have ? start(cur) : 0u;
  while (have) {
    bool have_next = false;
    uint32_t next_bits = 0u;
    build_chunk_record<false>(
        P.chunk, P.raw, P.vt, false, bbits, cur.nc, scale, lb_log2e, eps,
        ws + static_cast<int64_t>(cur.item) * REC_BYTES, t,
        [] {
          chunk_sync();
          return true;
        },
        [&] { issue_v_loads(loader, P.vt, v + cur.base, cur.nc); },
        [&] {
          have_next = find(cur.item + gridDim.x, nxt);
          if (have_next) next_bits = start(nxt);
          return have_next;
        });
    cur = nxt;
    have = have_next;
    bbits = next_bits;
  }
}

cudaError_t launch_chunk_prep(const void* q, const void* k, const void* v, const void* g,
                              const void* beta_raw, float scale, float lower_bound, float eps,
                              const int32_t* cu, int64_t T_total, int H, int N, void* ws,
                              int gate_scalar, int sm_count, cudaStream_t stream) {
  const int64_t n_items = slot_count(T_total, N) * H;
  const int smem = static_cast<int>(sizeof(PrepSmem));
  static std::atomic<uint64_t> smem_set{0};
  cudaError_t e =
      ensure_smem_limit(reinterpret_cast<const void*>(chunk_prep_kernel), smem, smem_set);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chunk_prep_kernel, 128, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t grid = (n_items < static_cast<int64_t>(sm_count) * per_sm ? n_items : static_cast<int64_t>(sm_count) * per_sm);
  if (grid <= 0) return cudaSuccess;
  chunk_prep_kernel<<<static_cast<unsigned>(grid), 128, smem, stream>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), static_cast<const __nv_bfloat16*>(g),
      static_cast<const __nv_bfloat16*>(beta_raw), scale, lower_bound * 1.4426950408889634f, eps,
      cu, T_total, H, N, static_cast<uint8_t*>(ws), n_items, gate_scalar);
  return cudaGetLastError();
}

}  // namespace kda
