// kda_recurrence.cu -- K2, the head-parallel recurrence kernel.  One CTA per
// (sequence, head) keeps the 128 x 128 fp32 state S resident in tensor memory
// and walks the chunk records in order ("You Could Have Come Up with Kimi
// Delta Attention", sec. 6.3-6.5; "FlashKDA Delta Attention Algorithm", Kernel
// K2):
//
//   MMA1 (tcgen05, tf32):  D1[v][n] = sum_d S[v][d] B1[n][d],  B1 = [W ; Qdec]
//                          -> D1[:, 0:16] = (W S^T)^T,  D1[:, 16:32] = (Qdec S^T)^T
//   threads (row v each):  S[v][:] *= dlast  (forget, sec. 6.4)
//                          e[v][i] = U[i][v] - D1[v][i]                (sec. 6.3)
//   MMA2 (tcgen05, bf16):  S += E^T_hi Kend_hi + E^T_lo Kend_hi + E^T_hi Kend_lo
//   threads:               o[i][v] = D1[v][16+i] + sum_{j<=i} Aqk[i][j] e[v][j]  (sec. 6.5)
//
// MMA1 reads the fp32 state straight from tensor memory as its A operand (the
// tensor core uses its tf32 part), so no operand copy of S is ever built.
//
// Roles: warps 0-3 own tensor-memory lanes 0-127 (state row v = thread id);
// warp 4 lane 0 streams records into a 3-stage shared-memory ring with bulk
// copies and issues every MMA.  All waits are bounded (kda_common.cuh); on a
// timeout the CTA records KDA_ERR_TIMEOUT in the error word and unwinds.
#include "kda_common.cuh"

namespace kda {

constexpr int NST = 3;
constexpr int K2_THREADS = 160;
constexpr uint32_t TM_S = 0, TM_D1 = 128, TM_A2H = 160, TM_A2L = 168, TM_COLS = 256;

struct K2Ctl {
  uint64_t full[NST];
  uint64_t empty[NST];
  uint64_t mma1, mma2, eready;
  uint32_t tmem;
  int abort;
};

constexpr int K2_SMEM = NST * REC_STRIDE_SMEM + 1024 + static_cast<int>(sizeof(K2Ctl)) + 64;

__device__ __forceinline__ uint64_t kend_desc(uint32_t saddr) {
#if KDA_KEND_LAYOUT == 0
  return make_sdesc(saddr, 16, 256, 6);
#else
  return make_sdesc(saddr, 128, 256, 0);
#endif
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, K2Ctl* ctl,
                                              int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*reinterpret_cast<volatile int*>(&ctl->abort)) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      *reinterpret_cast<volatile int*>(&ctl->abort) = 1;
      atomicExch(err, 5);
      return false;
    }
  }
  return true;
}

__global__ void __launch_bounds__(K2_THREADS, 2)
recurrence_kernel(const uint8_t* __restrict__ ws, const float* __restrict__ init,
                  const int32_t* __restrict__ cu, int64_t T_total, int H, int N,
                  __nv_bfloat16* __restrict__ out, float* __restrict__ final_state,
                  int* __restrict__ err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  K2Ctl* ctl = reinterpret_cast<K2Ctl*>(smem + NST * REC_STRIDE_SMEM);
  const int t = threadIdx.x, w = t >> 5, l = t & 31;
  const int unit = blockIdx.x;
  const int n = unit / H, h = unit - (unit / H) * H;
  int64_t bos, eos;
  seq_bounds(cu, T_total, N, n, bos, eos);
  const int nchunks = static_cast<int>((eos - bos + kChunk - 1) / kChunk);
  const int64_t slot0 = bos / kChunk + n;
  const uint8_t* rec0 = ws + (slot0 * H + h) * static_cast<int64_t>(REC_BYTES);
  const int64_t rec_step = static_cast<int64_t>(H) * REC_BYTES;

  if (t == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 129);
    }
    mbar_init(&ctl->mma1, 1);
    mbar_init(&ctl->mma2, 1);
    mbar_init(&ctl->eready, 128);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (w == 0) {
    tmem_alloc(&ctl->tmem, TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = ctl->tmem;
  const uint32_t lane_off = static_cast<uint32_t>((w & 3) * 32) << 16;
  const int64_t state_base = (static_cast<int64_t>(n) * H + h) * kDim * kDim;

  // initial state -> tensor memory (row v of S in lane v)
  if (w < 4) {
    const float* src = init ? init + state_base + static_cast<int64_t>(t) * kDim : nullptr;
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
      uint32_t r[32];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        float4 x = src ? __ldg(reinterpret_cast<const float4*>(src + qd * 32 + i))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        r[i] = __float_as_uint(x.x);
        r[i + 1] = __float_as_uint(x.y);
        r[i + 2] = __float_as_uint(x.z);
        r[i + 3] = __float_as_uint(x.w);
      }
      tmem_st32(tb + TM_S + lane_off + qd * 32, r);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (w == 4) {
    if (l == 0) {
      // ---------------- producer + MMA issuer ----------------
      const uint32_t id1 = make_idesc(2, 128, 32), id2 = make_idesc(1, 128, 128);
      int issued = 0, mma1_issued = 0, mma2_issued = 0;
      const int pre = nchunks < NST ? nchunks : NST;
      for (int p = 0; p < pre; ++p) {
        mbar_arrive_expect_tx(&ctl->full[p], REC_BYTES);
        bulk_g2s(smem + p * REC_STRIDE_SMEM, rec0 + p * rec_step, REC_BYTES, &ctl->full[p]);
        ++issued;
      }
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % NST;
        const uint32_t ph = (c / NST) & 1;
        if (!wait_or_abort(&ctl->full[s], ph, ctl, err)) break;
        if (c > 0 && !wait_or_abort(&ctl->mma2, (c - 1) & 1, ctl, err)) break;
        tc_fence_after();
        const uint32_t sb = smem_u32(smem + s * REC_STRIDE_SMEM);
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const uint64_t bd =
              make_sdesc(sb + OFF_B1 + (kk >> 2) * 4096 + (kk & 3) * 32, 16, 1024, 2);
          mma_tf32_ts(tb + TM_D1, tb + TM_S + kk * 8, bd, id1, kk > 0 ? 1u : 0u);
        }
        tc_commit(&ctl->mma1);
        ++mma1_issued;
        if (!wait_or_abort(&ctl->eready, c & 1, ctl, err)) break;
        tc_fence_after();
        const uint64_t kh = kend_desc(sb + OFF_KH), kl = kend_desc(sb + OFF_KL);
        mma_bf16_ts(tb + TM_S, tb + TM_A2H, kh, id2, 1u);
        mma_bf16_ts(tb + TM_S, tb + TM_A2L, kh, id2, 1u);
        mma_bf16_ts(tb + TM_S, tb + TM_A2H, kl, id2, 1u);
        tc_commit(&ctl->mma2);
        tc_commit(&ctl->empty[s]);
        ++mma2_issued;
        if (c >= 1 && c - 1 + NST < nchunks) {
          const int ps = (c - 1) % NST;
          if (!wait_or_abort(&ctl->empty[ps], ((c - 1) / NST) & 1, ctl, err)) break;
          const int p = c - 1 + NST;
          mbar_arrive_expect_tx(&ctl->full[ps], REC_BYTES);
          bulk_g2s(smem + ps * REC_STRIDE_SMEM, rec0 + p * rec_step, REC_BYTES, &ctl->full[ps]);
          ++issued;
        }
      }
      if (*reinterpret_cast<volatile int*>(&ctl->abort)) {
        // let copies and MMAs in flight land before the CTA releases its memory
        // (only the last copy issued into each stage can still be in flight)
        for (int p = issued > NST ? issued - NST : 0; p < issued; ++p)
          mbar_wait(&ctl->full[p % NST], (p / NST) & 1);
        if (mma1_issued) mbar_wait(&ctl->mma1, (mma1_issued - 1) & 1);
        if (mma2_issued) mbar_wait(&ctl->mma2, (mma2_issued - 1) & 1);
      }
    }
  } else {
    // ---------------- state rows: warps 0-3, thread t = value channel v ----------------
    const int v = t;
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % NST;
      const uint8_t* st = smem + s * REC_STRIDE_SMEM;
      if (!wait_or_abort(&ctl->full[s], (c / NST) & 1, ctl, err)) { ok = false; break; }
      if (!wait_or_abort(&ctl->mma1, c & 1, ctl, err)) { ok = false; break; }
      tc_fence_after();
      uint32_t d1[32];
      tmem_ld32(tb + TM_D1 + lane_off, d1);
      // forget: S[v][:] *= dlast
      const float* dl = reinterpret_cast<const float*>(st + OFF_DL);
#pragma unroll
      for (int qd = 0; qd < 4; ++qd) {
        uint32_t r[32];
        tmem_ld32(tb + TM_S + lane_off + qd * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i)
          r[i] = __float_as_uint(__uint_as_float(r[i]) * dl[qd * 32 + i]);
        tmem_st32(tb + TM_S + lane_off + qd * 32, r);
      }
      // corrected errors e[v][i] = U[i][v] - (W S^T)[i][v]
      const float4* U4 = reinterpret_cast<const float4*>(st + OFF_U + v * 64);
      float e[16];
#pragma unroll
      for (int i4 = 0; i4 < 4; ++i4) {
        const float4 u = U4[i4];
        e[i4 * 4 + 0] = u.x - __uint_as_float(d1[i4 * 4 + 0]);
        e[i4 * 4 + 1] = u.y - __uint_as_float(d1[i4 * 4 + 1]);
        e[i4 * 4 + 2] = u.z - __uint_as_float(d1[i4 * 4 + 2]);
        e[i4 * 4 + 3] = u.w - __uint_as_float(d1[i4 * 4 + 3]);
      }
      uint32_t pk[16];
#pragma unroll
      for (int c2 = 0; c2 < 8; ++c2) {
        const __nv_bfloat16 h0 = __float2bfloat16_rn(e[2 * c2]);
        const __nv_bfloat16 h1 = __float2bfloat16_rn(e[2 * c2 + 1]);
        pk[c2] = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) |
                 (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
        pk[8 + c2] = pack_bf16(e[2 * c2] - __bfloat162float(h0), e[2 * c2 + 1] - __bfloat162float(h1));
      }
      tmem_st16(tb + TM_A2H + lane_off, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&ctl->eready);
      // outputs o[i][v] = (Qdec S^T)[i][v] + sum_{j <= i} Aqk[i][j] e[v][j]
      const float* Aq = reinterpret_cast<const float*>(st + OFF_AQK);
      const int64_t t0 = bos + static_cast<int64_t>(c) * kChunk;
      const int nc = static_cast<int>(((eos - t0) < kChunk ? (eos - t0) : kChunk));
      __nv_bfloat16* orow = out + (t0 * H + h) * kDim + v;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float o = __uint_as_float(d1[16 + i]);
#pragma unroll
        for (int j = 0; j <= i; ++j) o = fmaf(Aq[i * 16 + j], e[j], o);
        if (i < nc) orow[static_cast<int64_t>(i) * H * kDim] = __float2bfloat16_rn(o);
      }
      mbar_arrive(&ctl->empty[s]);
    }
    if (ok && nchunks > 0 && !wait_or_abort(&ctl->mma2, (nchunks - 1) & 1, ctl, err)) ok = false;
    tc_fence_after();
    if (ok && final_state) {
      float* dst = final_state + state_base + static_cast<int64_t>(v) * kDim;
#pragma unroll
      for (int qd = 0; qd < 4; ++qd) {
        uint32_t r[32];
        tmem_ld32(tb + TM_S + lane_off + qd * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(dst + qd * 32 + i) =
              make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]),
                          __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (w == 0) tmem_dealloc(tb, TM_COLS);
}

cudaError_t launch_recurrence(const void* ws, const float* init, const int32_t* cu,
                              int64_t T_total, int H, int N, void* out, float* final_state,
                              int* err, cudaStream_t stream) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(recurrence_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, K2_SMEM);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int64_t units = static_cast<int64_t>(N) * H;
  if (units == 0) return cudaSuccess;
  recurrence_kernel<<<static_cast<unsigned>(units), K2_THREADS, K2_SMEM, stream>>>(
      static_cast<const uint8_t*>(ws), init, cu, T_total, H, N,
      static_cast<__nv_bfloat16*>(out), final_state, err);
  return cudaGetLastError();
}

}  // namespace kda
