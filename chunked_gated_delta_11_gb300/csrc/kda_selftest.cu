// kda_selftest.cu -- one-CTA check of the tcgen05 operand conventions that the
// recurrence relies on, with values that are exact in bf16 / tf32 so the fp32
// results can be compared bit for bit on the host.  Shared memory is laid out
// as one chunk record (kda_common.cuh):
//
//   MMA1-like: D1[128 x 32]  = A1[128 x 128] (bf16 pairs in tensor memory)
//                             * B1^T (bf16 [32 x 128] in the record's [Qdec ; W]
//                               layout), 8 K=16 steps.
//   MMA2-like: D2[128 x 144] = D0 + A2[128 x 16] (tf32, tensor memory)
//                             * B2^T (fp32 [144 x 16] in the record's
//                               [Kend ; Aqk] layout), 2 K=8 steps, accumulating.
//
// Every smem address the descriptors can form stays inside the 17 KB record
// area, so a wrong convention gives wrong numbers only.
#include "kda_state.cuh"

namespace kda {

__host__ __device__ inline float st_a1(int m, int k) { return ((m * 3 + k * 5) % 11 - 5) * 0.25f; }
__host__ __device__ inline float st_b1(int n, int k) { return ((n * 7 + k * 3) % 13 - 6) * 0.125f; }
__host__ __device__ inline float st_a2(int m, int j) { return ((m + 2 * j) % 7 - 3) * 0.5f; }
__host__ __device__ inline float st_b2(int d, int j) { return ((d * 5 + j * 11) % 9 - 4) * 0.25f; }
__host__ __device__ inline float st_d0(int m, int d) { return (m - d) * 0.0625f; }

__global__ void __launch_bounds__(128, 1)
selftest_tcgen05_kernel(float* __restrict__ out1, float* __restrict__ out2,
                        int* __restrict__ status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* rec = align1024(smem_raw);       // one record: B1 then [Kend ; Aqk]
  uint64_t* bar = reinterpret_cast<uint64_t*>(rec + OFF_U);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rec + OFF_U + 8);
  const int t = threadIdx.x, w = t >> 5;

  for (int e = t; e < 32 * 64; e += 128) {
    const int n = e >> 6, d = (e & 63) * 2;
    *reinterpret_cast<uint32_t*>(rec + b1_offset(n, d)) = pack_bf16(st_b1(n, d), st_b1(n, d + 1));
  }
  for (int e = t; e < 144 * 16; e += 128) {
    const int r = e >> 4, j = e & 15;
    *reinterpret_cast<float*>(rec + ka_offset(r, j)) = st_b2(r, j);
  }
  if (t == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (w == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  // generic-proxy smem writes must be visible to the tensor core (async proxy)
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t A1 = tbase, D2 = tbase + 64, D1 = tbase + 256, A2 = tbase + 288;
  const uint32_t lane_off = static_cast<uint32_t>(w * 32) << 16;
  const int m = t;

  // A1 row m as bf16 pairs (low half = even k), D0 row m, A2 row m (fp32)
  for (int q = 0; q < 2; ++q) {
    uint32_t r[32];
    for (int i = 0; i < 32; ++i) {
      const int k = (q * 32 + i) * 2;
      r[i] = pack_bf16(st_a1(m, k), st_a1(m, k + 1));
    }
    tmem_st32(A1 + lane_off + q * 32, r);
  }
  for (int q = 0; q < 5; ++q) {
    uint32_t r[32];
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(st_d0(m, q * 32 + i));
    if (q < 4) {
      tmem_st32(D2 + lane_off + q * 32, r);
    } else {
      uint32_t r16[16];
      for (int i = 0; i < 16; ++i) r16[i] = r[i];
      tmem_st16(D2 + lane_off + 128, r16);
    }
  }
  {
    uint32_t r[16];
    for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(st_a2(m, j));
    tmem_st16(A2 + lane_off, r);
  }
  tmem_wait_st();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (t == 0) {
    const uint32_t sb = smem_u32(rec);
    const uint32_t id1 = make_idesc(1, 128, 32);
    for (int kk = 0; kk < 8; ++kk) {
      const uint64_t bd = make_sdesc(sb + OFF_B1 + (kk >> 2) * 4096 + (kk & 3) * 32, 16, 1024, 2);
      mma_bf16_ts(D1, A1 + kk * 8, bd, id1, kk > 0);
    }
    const uint32_t id2 = make_idesc(2, 128, 144);
    for (int kk = 0; kk < 2; ++kk)
      mma_tf32_ts(D2, A2 + kk * 8, make_sdesc(sb + OFF_KA + kk * KA_TILE, 16, 256, 6), id2, 1);
    tc_commit(bar);
  }
  __syncwarp();
  const bool ok = mbar_wait(bar, 0);
  if (!ok && t == 0) atomicExch(status, 5);
  tc_fence_after();
  if (ok) {
    uint32_t r[32];
    tmem_ld32(D1 + lane_off, r);
    tmem_wait_ld();
    for (int i = 0; i < 32; ++i) out1[m * 32 + i] = __uint_as_float(r[i]);
    for (int q = 0; q < 4; ++q) {
      tmem_ld32(D2 + lane_off + q * 32, r);
      tmem_wait_ld();
      for (int i = 0; i < 32; ++i) out2[m * 144 + q * 32 + i] = __uint_as_float(r[i]);
    }
    uint32_t r16[16];
    tmem_ld16(D2 + lane_off + 128, r16);
    tmem_wait_ld();
    for (int i = 0; i < 16; ++i) out2[m * 144 + 128 + i] = __uint_as_float(r16[i]);
  }
  tc_fence_before();
  __syncthreads();
  if (w == 0) tmem_dealloc(tbase, 512);
}

// The timeout path of the bounded waits, exercised on purpose: one CTA of 128
// threads holds tensor memory, as the state threads of the forward kernels do,
// and waits with wait_or_abort on an mbarrier that nothing arrives at.  Each
// wait gives up after `limit` cycles, sets the CTA's abort flag and the device
// error word; the CTA agrees to stop through the same barrier reduction the
// recurrence uses (state_all), frees its tensor memory and exits.
__global__ void __launch_bounds__(128, 1) selftest_timeout_kernel(long long limit, int* err) {
  __shared__ StateCtl<1> ctl;
  const int t = threadIdx.x;
  if (t == 0) {
    mbar_init(&ctl.full[0], 1);  // one arrival expected, none ever made
    ctl.abort = 0;
    fence_mbar_init();
  }
  if (t < 32) {
    tmem_alloc(&ctl.tmem, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool ok = wait_or_abort(&ctl.full[0], 0, &ctl, err, limit);
  const bool all_ok = state_all(ok);  // false: every thread leaves together
  (void)all_ok;
  tc_fence_before();
  __syncthreads();
  if (t < 32) tmem_dealloc(ctl.tmem, 32);
}

cudaError_t launch_selftest_timeout(long long limit, int* err, cudaStream_t stream) {
  selftest_timeout_kernel<<<1, 128, 0, stream>>>(limit, err);
  return cudaGetLastError();
}

}  // namespace kda

extern "C" int kda_selftest_tcgen05(float* out1, float* out2, int* status, void* stream) {
  if (!out1 || !out2 || !status) return 1;
  const int smem = kda::OFF_U + 64 + 1024;
  kda::selftest_tcgen05_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(
      out1, out2, status);
  return cudaGetLastError() == cudaSuccess ? 0 : 4;
}
