// kda_prep.cu -- K1, the token-parallel chunk kernel.  One 128-thread CTA
// walks (chunk slot, head) work items with a grid-stride loop and writes one
// record per item (kda_chunk.cuh).  FlashKDA's K1 ("FlashKDA: MoonshotAI's
// High-Performance Kimi Delta Attention Kernels", sec. 2.2) has the same
// parallel axes (N x H x chunks); this one adds the W/U factors and stores
// everything the recurrence kernel reads.
#include "kda_chunk.cuh"
#include "kda_tma.cuh"

namespace kda {

struct PrepSmem {
  ChunkSmem chunk;
  alignas(128) uint8_t raw[QKG_BYTES];  // q, k, g_raw tiles (TMA destinations)
  alignas(128) uint8_t vt[V_BYTES];     // v tile
  uint64_t qkg_bar, v_bar;
  int abort;
};

__global__ void __launch_bounds__(128, 4)
chunk_prep_kernel(const __grid_constant__ RawMaps maps, const __nv_bfloat16* __restrict__ g,
                  const __nv_bfloat16* __restrict__ beta_raw, float scale, float lb_log2e,
                  float eps, const int32_t* __restrict__ cu, int64_t T_total, int H, int N,
                  uint8_t* __restrict__ ws, int64_t n_items, int gate_scalar,
                  int* __restrict__ err) {
  grid_dep_launch();  // the recurrence kernel may be scheduled now; it waits for this one
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // 128-byte aligned base (the TMA destinations inside are 128-byte aligned)
  PrepSmem& P = *reinterpret_cast<PrepSmem*>(smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u));
  const int t = threadIdx.x;
  if (t == 0) {
    mbar_init(&P.qkg_bar, 1);
    mbar_init(&P.v_bar, 1);
    P.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // the next used slot at or after `item` on this CTA's grid stride
  struct Item {
    int64_t item, t0;
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
        return true;
      }
    }
    return false;
  };
  // q, k, g_raw of an item into P.raw (the previous item's factor pass is
  // done with it); returns this thread's beta_raw bits of the item
  auto start = [&](const Item& it) -> uint32_t {
    if (gate_scalar) broadcast_gate_tile(P.raw + RAW_G * RAW_TILE, g + it.t0 * H + it.h, H, it.nc, t);
    if (t == 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue_qkg_tma(maps, P.raw, it.h, it.t0, gate_scalar != 0, &P.qkg_bar);
    }
    return (t < it.nc) ? __bfloat16_as_ushort(beta_raw[(it.t0 + t) * H + it.h]) : 0u;
  };

  Item cur, nxt;
  bool have = find(blockIdx.x, cur);
  uint32_t bbits = have ? start(cur) : 0u;
  // copies issued so far on each barrier; item i waits for phase i of both
  uint32_t qkg_issued = have ? 1u : 0u, v_issued = 0u, item = 0u;
  while (have) {
    bool have_next = false;
    uint32_t next_bits = 0u;
    const RawSync rs{&P.qkg_bar, item & 1u, &P.v_bar, item & 1u, &P.abort, err};
    const bool ok = build_chunk_record<false>(
        P.chunk, P.raw, P.vt, rs, bbits, cur.nc, scale, lb_log2e, eps,
        ws + static_cast<int64_t>(cur.item) * REC_BYTES, t,
        [&](bool arrived) {
          return chunk_all(arrived && !*reinterpret_cast<volatile int*>(&P.abort));
        },
        [&] {
          if (t == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue_v_tma(maps, P.vt, cur.h, cur.t0, &P.v_bar);
          }
          ++v_issued;
        },
        [&] {
          have_next = find(cur.item + gridDim.x, nxt);
          if (have_next) {
            next_bits = start(nxt);
            ++qkg_issued;
          }
        });
    if (!ok) break;
    cur = nxt;
    have = have_next;
    bbits = next_bits;
    ++item;
  }
  // after a timeout, copies still in flight must land before the CTA exits:
  // each barrier has at most one phase pending, the last one issued
  if (t == 0 && *reinterpret_cast<volatile int*>(&P.abort)) {
    if (qkg_issued) mbar_wait(&P.qkg_bar, (qkg_issued - 1) & 1u);
    if (v_issued) mbar_wait(&P.v_bar, (v_issued - 1) & 1u);
  }
}

cudaError_t launch_chunk_prep(const void* q, const void* k, const void* v, const void* g,
                              const void* beta_raw, float scale, float lower_bound, float eps,
                              const int32_t* cu, int64_t T_total, int H, int N, void* ws,
                              int gate_scalar, int sm_count, int* err, cudaStream_t stream) {
  const int64_t n_items = slot_count(T_total, N) * H;
  const int smem = static_cast<int>(sizeof(PrepSmem)) + 128;
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
  RawMaps maps;
  e = make_raw_maps(&maps, q, k, v, g, T_total, H, gate_scalar != 0);
  if (e != cudaSuccess) return e;
  chunk_prep_kernel<<<static_cast<unsigned>(grid), 128, smem, stream>>>(
      maps, static_cast<const __nv_bfloat16*>(g), static_cast<const __nv_bfloat16*>(beta_raw),
      scale, lower_bound * 1.4426950408889634f, eps, cu, T_total, H, N,
      static_cast<uint8_t*>(ws), n_items, gate_scalar, err);
  return cudaGetLastError();
}

}  // namespace kda
