// kda_common.cuh -- device helpers and the chunk-record layout shared by the
// sm_103a kernels of libkda (chunk kernel K1, recurrence kernel K2).
//
// The record is what one 16-token chunk of one head contributes to the
// chunkwise KDA recurrence ("You Could Have Come Up with Kimi Delta
// Attention", sec. 6.2-6.5), written so that the recurrence kernel can feed it
// to tcgen05 MMAs with no reshuffling:
//
//   E^T  = U - W S_c^T                 (corrected errors, sec. 6.3, WY form)
//   O    = Qdec S_c^T + Aqk E^T        (chunk outputs, sec. 6.5)
//   S'   = S_c Diag(dlast) + E Kend    (state fast-forward, sec. 6.4)
//
// The key-side factors carry a per-token rescaling D = diag(rk), rk_j =
// 1 / |k_j|, that cancels in these products: the record holds W' = D W,
// U' = D U (so the recurrence forms E'^T = D E^T), Kend' = D^-1 Kend = the
// unnormalised k_j D_{j+1:last}, and Aqk' = Aqk D^-1.
//
// Byte layout of one record (REC_BYTES):
//   [OFF_B1, +8192)    [Qdec ; W'], 32 rows x 128 key channels, bf16, K-major
//                      with the 128-byte swizzle: 2 blocks of 64 channels, each
//                      32 rows x 128 B; row n of block kb at kb*4096 + n*128,
//                      its 16-byte piece c at (c ^ (n & 7))*16.
//                      Rows 0..15 are Qdec, rows 16..31 are W'.
//   [OFF_KA, +9216)    [Kend' ; Aqk'] fp32 (the tensor core reads its tf32
//                      part), 144 rows r x 16 tokens j as two K=8 tiles (j 0-7,
//                      j 8-15) of 4608 B, K-major with the 32-byte swizzle: row
//                      r at r*32, 16-byte piece p at (p ^ ((r >> 2) & 1))*16.
//                      Rows 0..127 are Kend'[j][d] (r = d), rows 128..143 are
//                      Aqk'[i][j] (r = 128 + i; zero above the diagonal).
//   [OFF_U,  +8192)    U'^T fp32 [128 value channels c][16 tokens i], 64 B per
//                      row c; its four 16-byte pieces (4 tokens each) in the
//                      order p ^ (2 ((c >> 1) & 1) + ((c >> 2) & 1)).
//   [OFF_DL, +512)     dlast fp32 [128] = diagonal of D_{0:C-1}.
//   [OFF_RQ, +64)      rq fp32 [16]: the query factors s / |q_i| that Qdec and
//                      Aqk' leave out; the recurrence scales each output row
//                      by them.
// Rows of tokens past a ragged sequence end are zero, which makes them no-ops.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kda_bounds.h"

namespace kda {

constexpr int kChunk = 16;
constexpr int kDim = 128;

constexpr int OFF_B1 = 0;
constexpr int OFF_KA = 8192;
constexpr int KA_TILE = 4608;  // one K=8 tile of [Kend ; Aqk]: 144 rows x 32 B
constexpr int OFF_U = OFF_KA + 2 * KA_TILE;
constexpr int OFF_DL = OFF_U + 8192;
constexpr int OFF_RQ = OFF_DL + 512;
constexpr int REC_BYTES = OFF_RQ + 64;  // 26176
constexpr int REC_STRIDE_SMEM = 26624;   // 1024-aligned stage stride in smem
static_assert(REC_BYTES == 26176 && REC_STRIDE_SMEM >= REC_BYTES, "record layout");

__host__ __device__ constexpr int b1_offset(int n, int d) {
  // byte offset of bf16 element (row n, channel d) of the [Qdec ; W] tile
  return OFF_B1 + (d >> 6) * 4096 + n * 128 + ((((d & 63) >> 3) ^ (n & 7)) << 4) + ((d & 7) << 1);
}

// Byte offset of fp32 element (row r, token j) of the [Kend ; Aqk] tiles.
__host__ __device__ constexpr int ka_offset(int r, int j) {
  return OFF_KA + (j >> 3) * KA_TILE + r * 32 + (((((j & 7) >> 2) ^ (r >> 2)) & 1) << 4) +
         ((j & 3) << 2);
}
__host__ __device__ constexpr int kend_offset(int d, int j) { return ka_offset(d, j); }
// Byte offset of U^T element (value channel c, token i).
// The piece order swizzle keeps both the chunk side's stores (rows c, c + 2 of
// an MMA tile at once) and the state side's row reads (8 consecutive rows)
// conflict-free.
__host__ __device__ constexpr int u_piece_swz(int c) { return (((c >> 1) & 1) << 1) | ((c >> 2) & 1); }
__host__ __device__ constexpr int u_offset(int c, int i) {
  return OFF_U + c * 64 + (((i >> 2) ^ u_piece_swz(c)) << 4) + ((i & 3) << 2);
}
__host__ __device__ constexpr int aqk_offset(int i, int j) { return ka_offset(128 + i, j); }

// A kernel's dynamic shared-memory limit, set once per device: the attribute
// belongs to the function in the current device's context, so a process that
// drives several GPUs sets it on each.  `done` is the launcher's mask of
// devices already set (devices >= 64 set it on every call).
inline cudaError_t ensure_smem_limit(const void* func, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Per-call options of the forward pass (uniform over the grid).
struct FwdOpts {
  int state_bf16;   // initial / final states are bf16 instead of fp32
  int gate_scalar;  // g_raw is one value per token and head [T_total, H]
};

// Segmented launch of the fused kernel (the affine-map split of each sequence
// into P pieces, kda_segmented.cu).  With P > 0 the kernel's N is the number
// of segments, N_seq * P, and its grid holds two CTAs per (segment, head):
//   blocks [0, N H)      X role: the segment from a zero state (the first
//                        segment of each sequence from that sequence's initial
//                        state, element ((n / P) H + h) of `init`), outputs to
//                        `out`, final state to `final_state` [N, H, V, K]
//                        (always fp32 here; FwdOpts.state_bf16 then concerns
//                        `init` only);
//   blocks [N H, 2 N H)  M role: the same segment with v = 0 from the identity,
//                        whose state is the product of the segment's
//                        transition matrices and whose outputs are those
//                        matrices applied to the scaled queries; outputs to `y`,
//                        final state to `m_final`.  Not run for first segments.
struct SegArgs {
  int P;                 // segments per sequence; 0 = a plain forward pass
  __nv_bfloat16* y;      // M-role outputs [T_total, H, 128]
  float* m_final;        // M-role final states [N, H, 128, 128] (fp32)
};

// Address of element `elem` of a state buffer of fp32 (or bf16) entries; null stays null.
__device__ __forceinline__ const void* state_at(const void* base, int64_t elem, bool bf16) {
  return base ? static_cast<const uint8_t*>(base) + elem * (bf16 ? 2 : 4) : nullptr;
}
__device__ __forceinline__ void* state_at(void* base, int64_t elem, bool bf16) {
  return base ? static_cast<uint8_t*>(base) + elem * (bf16 ? 2 : 4) : nullptr;
}

// ---------------------------------------------------------------------------
// small PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// First 1024-byte-aligned byte of a dynamic shared-memory buffer.  Pointer
// arithmetic on the __shared__ array itself (no round trip through an integer)
// keeps the shared address space visible to the compiler.
__device__ __forceinline__ uint8_t* align1024(uint8_t* base) {
  return base + ((1024u - (smem_u32(base) & 1023u)) & 1023u);
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// sigma(x) = 1 / (1 + 2^(-x log2 e)), from the exponential and reciprocal units
__device__ __forceinline__ float sigmoid_fast(float x) {
  return rcp_approx(1.0f + ex2_approx(-1.4426950408889634f * x));
}

// fp32 -> tf32 bits (round to nearest, ties away), in an fp32 container
__device__ __forceinline__ uint32_t tf32_bits(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the same condition: its result can be read some
// instructions later, so the test's latency overlaps other work.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Same test, but a thread whose phase is not complete sleeps in hardware until
// it completes or about `hint_ns` nanoseconds pass, instead of spinning on the
// issue slots that the other warps of its SM partition need.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Every wait in libkda is bounded: ~2^31 SM cycles (about a second) and then
// the caller records an error and unwinds instead of hanging the GPU.
constexpr long long kWaitLimitCycles = 1LL << 31;
constexpr uint32_t kSleepHintNs = 20000;

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity, kSleepHintNs)) {
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
  return true;
}

// ---------------------------------------------------------------------------
// bulk (TMA, untiled) copies
// ---------------------------------------------------------------------------
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor core, accumulators in tensor memory)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// D (tmem, fp32) (+)= A (tmem) * B (smem descriptor); A/B tf32, one K=8 step.
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (tmem, fp32) (+)= A (tmem) * B (smem descriptor); A/B bf16, one K=16 step.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor for dense tcgen05.mma with fp32 accumulation.
// fmt: 1 = bf16 operands (kind::f16), 2 = tf32 operands (kind::tf32).
// Both operands K-major.  Bits: [4,6) D format (1 = f32), [7,10) A format,
// [10,13) B format, [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t fmt, uint32_t M, uint32_t N) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (all >> 4), version 1 at bit 46, layout type at
// bits [61,64): 0 = no swizzle, 2 = 128-byte, 4 = 64-byte, 6 = 32-byte swizzle.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                               uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;
  d |= static_cast<uint64_t>(layout & 7u) << 61;
  return d;
}

// 32 lanes x 32 bits, 32 consecutive columns per thread
#define KDA_R32(r)                                                                              \
  "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),          \
      "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),  \
      "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),            \
      "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),            \
      "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
#define KDA_W32(r)                                                                              \
  "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),      \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),        \
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),      \
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),      \
      "r"(r[29]), "r"(r[30]), "r"(r[31])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : KDA_R32(r)
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      KDA_W32(r)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Named barrier over the first `nthreads` threads (multiple of 32).
// Programmatic dependent launch, for the chains of kernels on one stream
// (the segmented pass): a kernel launched with launch_pdl may be scheduled
// while the kernel before it still runs.  grid_dep_wait: wait until that
// kernel has completed and its memory writes are visible (a no-op for a
// kernel launched without the attribute).  grid_dep_launch: let the next
// kernel, if launched with launch_pdl, be scheduled now.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch with the programmatic-stream-serialization attribute (see above).
template <class... KArgs, class... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

__device__ __forceinline__ void named_bar(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// sequence geometry.  Chunk records of sequence n live at record slots
// slot0(n) .. slot0(n) + nchunks(n) - 1 with slot0(n) = floor(bos_n / 16) + n,
// which never overlap and stay below T_total / 16 + N + 1.  The bounds read
// from cu_seqlens are clamped (kda_bounds.h): a malformed cu_seqlens gives
// wrong results (and kda_validate_cu_seqlens reports it) but every access stays
// inside the tensors and the workspace, since the last slot of a sequence is
// below eos / 16 + n + 1 for any 0 <= bos <= eos <= T_total.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void seq_bounds(const int32_t* cu, int64_t T_total, int N, int n,
                                           int64_t& bos, int64_t& eos) {
  if (cu) {
    clamp_seq_bounds(__ldg(cu + n), __ldg(cu + n + 1), T_total, bos, eos);
  } else {
    const int64_t L = T_total / N;
    bos = static_cast<int64_t>(n) * L;
    eos = bos + L;
  }
}

// Longest-first order of packed sequences.  The chunkwise kernels run one CTA
// per (sequence, head) and CTAs start in blockIdx order, so a varlen batch
// whose longest sequences come last ends with a tail of a few long units.
// Starting the longest sequences first (list scheduling, longest processing
// time first) shortens it.  Returns the sequence of rank r (lengths
// descending, ties by index).  Every thread of the CTA must call it.  It uses
// `scratch` (kOrderMaxN + 1 ints of shared memory) and ends with a barrier,
// after which scratch is free again.  For N <= kOrderMaxN; the cost is
// N^2 / blockDim comparisons per thread.
constexpr int kOrderMaxN = 256;
static __device__ __noinline__ int seq_by_rank(const int32_t* __restrict__ cu, int N, int r,
                                           int* scratch) {
  int* len = scratch;
  int* pick = scratch + kOrderMaxN;
  for (int m = threadIdx.x; m < N; m += blockDim.x) len[m] = __ldg(cu + m + 1) - __ldg(cu + m);
  __syncthreads();
  for (int m = threadIdx.x; m < N; m += blockDim.x) {
    const int lm = len[m];
    int rank = 0;
    for (int j = 0; j < N; ++j) rank += (len[j] > lm) | ((len[j] == lm) & (j < m));
    if (rank == r) *pick = m;  // ranks are a permutation: exactly one writer
  }
  __syncthreads();
  const int n = *pick;
  __syncthreads();
  return n;
}

__host__ __device__ __forceinline__ int64_t slot_count(int64_t T_total, int N) {
  return T_total / kChunk + N + 1;
}

}  // namespace kda
