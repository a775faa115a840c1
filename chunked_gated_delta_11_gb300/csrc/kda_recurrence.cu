// kda_recurrence.cu -- K2, the head-parallel recurrence kernel of the
// two-kernel path.  One CTA per (sequence, head) walks that unit's chunk
// records in order ("FlashKDA Delta Attention Algorithm", Kernel K2; the
// per-chunk arithmetic is in kda_state.cuh).
//
// 128 threads, the state threads (tensor-memory lanes 0-127, state row v =
// thread id).  Thread 0 also streams the records written by the chunk kernel
// from HBM into a 4-stage shared-memory ring (one cp.async.bulk per record,
// refilled as soon as a record's MMAs have finished) and issues every MMA.
#include "kda_state.cuh"

namespace kda {

constexpr int K2_NST = 4;
constexpr int K2_THREADS = 128;
constexpr int K2_OST_OFF = K2_NST * REC_STRIDE_SMEM;
constexpr int K2_CTL_OFF = K2_OST_OFF + 4096 + 256;  // output staging, then rq slots
constexpr int K2_SMEM = K2_CTL_OFF + static_cast<int>(sizeof(StateCtl<K2_NST>)) + 1024 + 64;
static_assert(2 * (K2_SMEM + 1024) <= 228 * 1024, "recurrence kernel must fit two CTAs per SM");

template <bool kTimed>
__global__ void __launch_bounds__(K2_THREADS, 2)
recurrence_kernel(const uint8_t* __restrict__ ws, const void* init,
                  const int32_t* __restrict__ cu, int64_t T_total, int H, int N,
                  __nv_bfloat16* __restrict__ out, void* final_state, FwdOpts opts,
                  int* __restrict__ err, long long* stamps, int max_chunks) {
  // this launch may start while the chunk kernel runs: wait for its records
  grid_dep_wait();
  constexpr int NST = K2_NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  auto* ctl = reinterpret_cast<StateCtl<NST>*>(smem + K2_CTL_OFF);
  const int t = threadIdx.x, w = t >> 5, l = t & 31;
  const int unit = blockIdx.x;
  const int h = unit - (unit / H) * H;
  // packed sequences start longest first (seq_by_rank); the record ring is
  // free until the first copy is issued
  const int n = (cu && N > 1 && N <= kOrderMaxN)
                    ? seq_by_rank(cu, N, unit / H, reinterpret_cast<int*>(smem))
                    : unit / H;
  int64_t bos, eos;
  seq_bounds(cu, T_total, N, n, bos, eos);
  const int nchunks = static_cast<int>((eos - bos + kChunk - 1) / kChunk);
  const int64_t slot0 = bos / kChunk + n;
  const uint8_t* rec0 = ws + (slot0 * H + h) * static_cast<int64_t>(REC_BYTES);
  const int64_t rec_step = static_cast<int64_t>(H) * REC_BYTES;

  if (t == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    mbar_init(&ctl->mma1, 1);
    mbar_init(&ctl->mma2, 1);
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
  load_state(tb, lane_off, state_at(init, state_base + static_cast<int64_t>(t) * kDim, opts.state_bf16),
             opts.state_bf16);
  int issued = 0;
  if (t == 0) {
    const int pre = nchunks < NST ? nchunks : NST;
    for (int p = 0; p < pre; ++p) {
      mbar_arrive_expect_tx(&ctl->full[p], REC_BYTES);
      bulk_g2s(smem + p * REC_STRIDE_SMEM, rec0 + p * rec_step, REC_BYTES, &ctl->full[p]);
      ++issued;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // a record's stage is refilled with the record NST chunks later once its
  // MMAs are done (the state threads finished reading it before MMA2 started)
  auto refill = [&](int c, int s) {
    const int p = c + NST;
    if (p < nchunks) {
      mbar_arrive_expect_tx(&ctl->full[s], REC_BYTES);
      bulk_g2s(smem + s * REC_STRIDE_SMEM, rec0 + p * rec_step, REC_BYTES, &ctl->full[s]);
      ++issued;
    }
  };
  state_rows<NST, 32, kTimed>(ctl, smem, nchunks, tb, lane_off, t, bos, eos, H, h, out,
                          state_at(final_state, state_base + static_cast<int64_t>(t) * kDim,
                                   opts.state_bf16),
                          opts.state_bf16, err, smem + K2_OST_OFF, refill, [](int, int) {}, false,
                          blockIdx.x == 0 ? stamps : nullptr, max_chunks);
  if (t == 0 && *reinterpret_cast<volatile int*>(&ctl->abort)) {
    // copies still in flight must land before the CTA releases its memory
    for (int p = issued > NST ? issued - NST : 0; p < issued; ++p)
      mbar_wait(&ctl->full[p % NST], (p / NST) & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (w == 0) tmem_dealloc(tb, TM_COLS);
}

template <bool kTimed>
cudaError_t launch_recurrence_t(const void* ws, const void* init, const int32_t* cu,
                                int64_t T_total, int H, int N, void* out, void* final_state,
                                FwdOpts opts, int* err, long long* stamps, int max_chunks,
                                cudaStream_t stream) {
  static std::atomic<uint64_t> smem_set{0};
  if (const cudaError_t e = ensure_smem_limit(
          reinterpret_cast<const void*>(recurrence_kernel<kTimed>), K2_SMEM, smem_set);
      e != cudaSuccess)
    return e;
  const int64_t units = static_cast<int64_t>(N) * H;
  if (units == 0) return cudaSuccess;
  return launch_pdl(recurrence_kernel<kTimed>, dim3(static_cast<unsigned>(units)), dim3(K2_THREADS),
                    K2_SMEM, stream, static_cast<const uint8_t*>(ws), init, cu, T_total, H, N,
                    static_cast<__nv_bfloat16*>(out), final_state, opts, err, stamps, max_chunks);
}

cudaError_t launch_recurrence(const void* ws, const void* init, const int32_t* cu,
                              int64_t T_total, int H, int N, void* out, void* final_state,
                              FwdOpts opts, int* err, cudaStream_t stream) {
  return launch_recurrence_t<false>(ws, init, cu, T_total, H, N, out, final_state, opts, err,
                                    nullptr, 0, stream);
}

// The diagnostic instantiation: thread 0 of CTA 0 records the phase stamps
// of state_rows (kda_state.cuh) for its first max_chunks chunks.
cudaError_t launch_recurrence_timed(const void* ws, const void* init, const int32_t* cu,
                                    int64_t T_total, int H, int N, void* out, void* final_state,
                                    FwdOpts opts, int* err, long long* stamps, int max_chunks,
                                    cudaStream_t stream) {
  return launch_recurrence_t<true>(ws, init, cu, T_total, H, N, out, final_state, opts, err,
                                   stamps, max_chunks, stream);
}

}  // namespace kda
