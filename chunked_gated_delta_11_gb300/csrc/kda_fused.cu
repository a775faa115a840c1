// kda_fused.cu -- the single-kernel forward path.  One CTA per (sequence,
// head) builds each chunk record in shared memory and runs the recurrence on
// it, so the records never travel through HBM: HBM traffic is the algorithmic
// q, k, v, g_raw and beta_raw in, `out` out (plus the states).  Packed
// sequences start longest first (seq_by_rank in kda_common.cuh).  A segmented
// launch (SegArgs, kda_common.cuh) runs two CTA roles per (segment, head).
//
// Roles (256 threads, two CTAs per SM):
//   warps 0-3  state threads (tensor-memory lanes 0-127); thread 0 also
//              issues the tcgen05 MMAs                        kda_state.cuh
//   warps 4-7  chunk threads: build record c+1 into the other stage of a
//              2-stage ring while the state threads work on record c
//                                                             kda_chunk.cuh
// The chunk threads write the records with ordinary shared-memory stores; each
// of them fences those stores against the tensor core's (async-proxy) reads,
// and each chunk warp then arrives once on full[s].
//
// FlashKDA measured its fused prototype as slower than the two-kernel split
// ("FlashKDA v1: A Deep Dive", sec. 2) because the token-parallel work waited
// on the serial recurrence; here the chunk math of chunk c+1 overlaps the
// recurrence of chunk c inside every CTA instead.
#include "kda_chunk.cuh"
#include "kda_state.cuh"
#include "kda_tma.cuh"

namespace kda {

constexpr int F_NST = 2;
constexpr int F_THREADS = 256;
// Registers per thread: the kernel is compiled for 128 (two CTAs of 256
// threads per SM); after the prologue the state warpgroup takes 136 and the
// chunk warpgroup 120 (setmaxnreg), 128 x 136 + 128 x 120 = 256 x 128, so the
// increase is always covered by the decrease.  launch_fused checks the
// compiled count before the first launch.
constexpr int F_REGS = 128, F_STATE_REGS = 136, F_CHUNK_REGS = 120;
static_assert(128 * F_STATE_REGS + 128 * F_CHUNK_REGS == F_THREADS * F_REGS,
              "register split must add up to the launch allocation");
constexpr int F_CHUNK_OFF = F_NST * REC_STRIDE_SMEM;
constexpr int F_RAW_OFF = F_CHUNK_OFF + ((static_cast<int>(sizeof(ChunkSmem)) + 127) & ~127);
constexpr int F_V_OFF = F_RAW_OFF + 2 * QKG_BYTES;  // q, k, g_raw double-buffered
constexpr int F_OST_OFF = F_V_OFF + V_BYTES;
constexpr int F_CTL_OFF = F_OST_OFF + 4096 + 256;  // output staging, then rq slots
// the raw tiles' barriers (q/k/g_raw buffers 0 and 1, v) and how many copy
// groups each has had (read after an abort, to let the last ones land)
struct RawBars {
  uint64_t qkg[2];
  uint64_t v;
  int qkg_n, v_n;
};
constexpr int F_RB_OFF = (F_CTL_OFF + static_cast<int>(sizeof(StateCtl<F_NST>)) + 7) & ~7;
constexpr int F_SMEM = F_RB_OFF + static_cast<int>(sizeof(RawBars)) + 1024 + 64;
static_assert(F_RAW_OFF % 128 == 0 && F_V_OFF % 128 == 0, "TMA destinations are 128-byte aligned");
// two CTAs per SM: 228 KB of shared memory per SM, 1 KB of it reserved per CTA
static_assert(2 * (F_SMEM + 1024) <= 228 * 1024, "fused kernel must fit two CTAs per SM");

// kTimed: the diagnostic instantiation of kda_profile_phases, in which thread
// 0 of CTA 0 records the state side's phase stamps (state_rows).
template <bool kGateScalar, bool kTimed>
__global__ void __launch_bounds__(F_THREADS, 2)
fused_kernel(const __grid_constant__ RawMaps maps, const __nv_bfloat16* __restrict__ g,
             const __nv_bfloat16* __restrict__ beta_raw, float scale, float lb_log2e, float eps,
             const void* init, const int32_t* __restrict__ cu, int64_t T_total, int H, int N,
             __nv_bfloat16* __restrict__ out, void* final_state, FwdOpts opts, SegArgs seg,
             int* __restrict__ err, long long* stamps, int max_chunks) {
  // this launch may start while the previous kernel on the stream runs (in
  // a segmented pass, the plan kernel whose cu_seqlens are read below)
  grid_dep_wait();
  grid_dep_launch();
  constexpr int NST = F_NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  ChunkSmem& CS = *reinterpret_cast<ChunkSmem*>(smem + F_CHUNK_OFF);
  auto* ctl = reinterpret_cast<StateCtl<NST>*>(smem + F_CTL_OFF);
  auto* rb = reinterpret_cast<RawBars*>(smem + F_RB_OFF);
  const int t = threadIdx.x, w = t >> 5, l = t & 31;
  int unit = blockIdx.x;
  const bool mrole = seg.P > 0 && unit >= N * H;  // segmented launch, M role (SegArgs)
  if (mrole) unit -= N * H;
  const int h = unit - (unit / H) * H;
  // packed sequences start longest first (seq_by_rank); the chunk scratch is
  // free until the build starts
  const int n = (seg.P == 0 && cu && N > 1 && N <= kOrderMaxN)
                    ? seq_by_rank(cu, N, unit / H, reinterpret_cast<int*>(smem + F_CHUNK_OFF))
                    : unit / H;
  // a first segment starts from the sequence's own state: it needs no M role
  if (mrole && n % seg.P == 0) return;
  // initial state: the M role starts from the identity, a later segment from
  // zero, a first segment from its sequence's state
  const void* init_u = (mrole || (seg.P > 0 && n % seg.P != 0)) ? nullptr : init;
  const int64_t init_unit = seg.P > 0 ? n / seg.P : n;
  int64_t bos, eos;
  seq_bounds(cu, T_total, N, n, bos, eos);
  const int nchunks = static_cast<int>((eos - bos + kChunk - 1) / kChunk);

  if (t == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&ctl->full[s], 4);  // one arrival per chunk warp
      mbar_init(&ctl->empty[s], 1);
    }
    mbar_init(&ctl->mma1, 1);
    mbar_init(&ctl->mma2, 1);
    mbar_init(&rb->qkg[0], 1);  // one arrive.expect_tx per copy group
    mbar_init(&rb->qkg[1], 1);
    mbar_init(&rb->v, 1);
    rb->qkg_n = 0;
    rb->v_n = 0;
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
  // Raw input tiles: q, k, g_raw double-buffered, v single.  One state
  // thread issues each copy group (kda_tma.cuh): those of chunks 0 and 1 (v:
  // chunk 0) as soon as the barriers exist, so that they arrive while the
  // state loads, then each as soon as record j is there
  // (on_record): chunk j is done with its q, k, g_raw buffer, which takes
  // chunk j + 2, and with the v buffer, which takes chunk j + 1.  So the
  // copies cost the chunk threads nothing, and q, k, g_raw have a whole
  // build to arrive, v the first part of one.
  auto rawbuf = [&](int c) { return smem + F_RAW_OFF + (c & 1) * QKG_BYTES; };
  uint8_t* vt = smem + F_V_OFF;
  auto chunk_t0 = [&](int c) { return bos + static_cast<int64_t>(c) * kChunk; };
  auto issue_qkg = [&](int c) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    issue_qkg_tma(maps, rawbuf(c), h, chunk_t0(c), kGateScalar, &rb->qkg[c & 1]);
    ++rb->qkg_n;
  };
  // M role: v = 0, nothing to load (the record's U' is taken as zero)
  auto issue_v = [&](int c) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    issue_v_tma(maps, vt, h, chunk_t0(c), &rb->v);
    ++rb->v_n;
  };

  if (t == 32) {
    if (nchunks > 0) issue_qkg(0);
    if (nchunks > 1) issue_qkg(1);
  }
  if (t == 64 && !mrole && nchunks > 0) issue_v(0);

  const uint32_t tb = ctl->tmem;
  const uint32_t lane_off = static_cast<uint32_t>((w & 3) * 32) << 16;
  const int64_t state_base = (static_cast<int64_t>(n) * H + h) * kDim * kDim;
  const int64_t init_base = (init_unit * H + h) * kDim * kDim;
  if (w < 4)
    load_state(tb, lane_off, state_at(init_u, init_base + static_cast<int64_t>(t) * kDim, opts.state_bf16),
               opts.state_bf16, mrole ? t : -1);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (w >= 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(F_CHUNK_REGS));
    // ---------------- chunk threads ----------------
    const int tc = t - 128;
    // g_raw of head h as one value per token (the scalar gate, [T, H])
    const __nv_bfloat16* g0 = g + h;
    auto chunk_nc = [&](int c) {
      const int64_t left = eos - chunk_t0(c);
      return static_cast<int>(left < kChunk ? left : kChunk);
    };
    // beta_raw of chunk c (and, for the scalar gate, its g_raw tile, written
    // once the buffer's previous chunk is done with it)
    auto prepare = [&](int c) -> uint32_t {
      const int64_t t0 = chunk_t0(c);
      const int nc = chunk_nc(c);
      if (kGateScalar) broadcast_gate_tile(rawbuf(c) + RAW_G * RAW_TILE, g0 + t0 * H, H, nc, tc);
      return (tc < nc) ? __bfloat16_as_ushort(beta_raw[(t0 + tc) * H + h]) : 0u;
    };
    uint32_t bbits[2] = {0u, 0u};  // beta_raw bits of chunks c and c+1
    // whether an earlier test found the next chunk's q, k, g_raw there
    bool qkg_ready = false;
    if (nchunks > 0) bbits[0] = prepare(0);
    if (nchunks > 1) bbits[1] = prepare(1);
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % NST;
      const int nc = chunk_nc(c);
      uint32_t next_bits = 0u;
      // before writing record c into stage s: its raw tiles are there, and
      // record c - NST in that stage is fully consumed (its MMAs read
      // [Qdec ; W] and [Kend ; Aqk]).  The first chunk warp polls the empty
      // barrier; all of them agree through the barrier reduction.
      auto may_write = [&](bool arrived) -> bool {
        bool ok = arrived && (c < NST || tc >= 32 ||
                              wait_or_abort(&ctl->empty[s], ((c / NST) - 1) & 1, ctl, err));
        ok = ok && !*reinterpret_cast<volatile int*>(&ctl->abort);
        return chunk_all(ok);
      };
      auto next_qkg = [&] {
        if (c + 2 < nchunks) next_bits = prepare(c + 2);
      };
      uint8_t* rec = smem + s * REC_STRIDE_SMEM;
      // chunk c is the (c >> 1)-th use of its q, k, g_raw buffer and the
      // c-th v copy
      const bool has_next = c + 1 < nchunks;
      const RawSync rs{&rb->qkg[c & 1], static_cast<uint32_t>((c >> 1) & 1), &rb->v,
                       static_cast<uint32_t>(c & 1), &ctl->abort, err, qkg_ready,
                       has_next ? &rb->qkg[(c + 1) & 1] : nullptr,
                       static_cast<uint32_t>(((c + 1) >> 1) & 1), &qkg_ready};
      if (!build_chunk_record<true>(CS, rawbuf(c), vt, rs, bbits[0], nc, scale, lb_log2e, eps,
                                    rec, tc, may_write, [] {}, next_qkg, mrole))
        break;
      // every thread's record stores -> async proxy, then one arrival per warp
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if ((tc & 31) == 0) mbar_arrive(&ctl->full[s]);
      bbits[0] = bbits[1];
      bbits[1] = next_bits;
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(F_STATE_REGS));
    // ---------------- state threads (thread 0 issues the MMAs) ----------------
    auto release = [&](int, int s) { mbar_arrive(&ctl->empty[s]); };
    // once record j is there: q, k, g_raw of chunk j + 2 (state warp 1), v
    // of chunk j + 1 (state warp 2)
    auto on_record = [&](int j, int sw) {
      if (sw == 1 && j + 2 < nchunks) issue_qkg(j + 2);
      if (sw == 2 && !mrole && j + 1 < nchunks) issue_v(j + 1);
    };
    // a segmented launch writes every piece's final state to its fp32 workspace
    const bool final_bf16 = opts.state_bf16 && seg.P == 0;
    // 16-column snapshot pieces: the state warps run under the 136-register cap
    state_rows<NST, 16, kTimed>(ctl, smem, nchunks, tb, lane_off, t, bos, eos, H, h,
                            mrole ? seg.y : out,
                            state_at(mrole ? static_cast<void*>(seg.m_final) : final_state,
                                     state_base + static_cast<int64_t>(t) * kDim, final_bf16),
                            final_bf16, err, smem + F_OST_OFF, release, on_record, mrole,
                            blockIdx.x == 0 ? stamps : nullptr, max_chunks);
  }
  tc_fence_before();
  __syncthreads();
  // after an abort, copies still in flight must land before the CTA exits:
  // each barrier has at most one phase pending, the last one issued
  if (t == 0 && *reinterpret_cast<volatile int*>(&ctl->abort)) {
    const int nq = rb->qkg_n, nv = rb->v_n;
    for (int b = 0; b < 2; ++b) {
      const int last = nq - 1 - ((nq - 1 - b) & 1);  // last chunk in buffer b
      if (last >= 0) mbar_wait(&rb->qkg[b], (last >> 1) & 1);
    }
    if (nv > 0) mbar_wait(&rb->v, (nv - 1) & 1);
  }
  if (w == 0) tmem_dealloc(tb, TM_COLS);
}

template <bool kGateScalar, bool kTimed = false>
cudaError_t launch_fused_t(const void* q, const void* k, const void* v, const void* g,
                           const void* beta_raw, float scale, float lower_bound, float eps,
                           const void* init, const int32_t* cu, int64_t T_total, int H, int N,
                           void* out, void* final_state, FwdOpts opts, SegArgs seg, int* err,
                           cudaStream_t stream, long long* stamps = nullptr, int max_chunks = 0) {
  // the register split above is only safe if every thread starts with F_REGS
  static std::atomic<uint64_t> checked{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  if (dev >= 64 || !(checked.load(std::memory_order_acquire) & (uint64_t{1} << dev))) {
    cudaFuncAttributes fa;
    const cudaError_t e = cudaFuncGetAttributes(&fa, fused_kernel<kGateScalar, kTimed>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != F_REGS) return cudaErrorInvalidConfiguration;
    if (dev < 64) checked.fetch_or(uint64_t{1} << dev, std::memory_order_release);
  }
  static std::atomic<uint64_t> smem_set{0};
  if (const cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(fused_kernel<kGateScalar, kTimed>),
                                              F_SMEM, smem_set);
      e != cudaSuccess)
    return e;
  const int64_t units = static_cast<int64_t>(N) * H * (seg.P > 0 ? 2 : 1);
  if (units == 0) return cudaSuccess;
  if (units > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  RawMaps maps;
  if (const cudaError_t e = make_raw_maps(&maps, q, k, v, g, T_total, H, kGateScalar);
      e != cudaSuccess)
    return e;
  // programmatic dependent launch: the kernel's first action is to wait for
  // the previous kernel on the stream, so its launch may overlap that
  // kernel's tail (the segmented pass chains its plan, this kernel, the scan
  // and the fix-up this way)
  return launch_pdl(fused_kernel<kGateScalar, kTimed>, dim3(static_cast<unsigned>(units)),
                    dim3(F_THREADS), F_SMEM, stream, maps, static_cast<const __nv_bfloat16*>(g),
                    static_cast<const __nv_bfloat16*>(beta_raw), scale,
                    lower_bound * 1.4426950408889634f, eps, init, cu, T_total, H, N,
                    static_cast<__nv_bfloat16*>(out), final_state, opts, seg, err, stamps,
                    max_chunks);
}

cudaError_t launch_fused(const void* q, const void* k, const void* v, const void* g,
                         const void* beta_raw, float scale, float lower_bound, float eps,
                         const void* init, const int32_t* cu, int64_t T_total, int H, int N,
                         void* out, void* final_state, FwdOpts opts, SegArgs seg, int* err,
                         cudaStream_t stream) {
  return opts.gate_scalar
             ? launch_fused_t<true>(q, k, v, g, beta_raw, scale, lower_bound, eps, init, cu,
                                    T_total, H, N, out, final_state, opts, seg, err, stream)
             : launch_fused_t<false>(q, k, v, g, beta_raw, scale, lower_bound, eps, init, cu,
                                     T_total, H, N, out, final_state, opts, seg, err, stream);
}

// The diagnostic instantiation (per-channel gate, fp32 states, no segments).
cudaError_t launch_fused_timed(const void* q, const void* k, const void* v, const void* g,
                               const void* beta_raw, float scale, float lower_bound, float eps,
                               const int32_t* cu, int64_t T_total, int H, int N, void* out,
                               void* final_state, int* err, long long* stamps, int max_chunks,
                               cudaStream_t stream) {
  return launch_fused_t<false, true>(q, k, v, g, beta_raw, scale, lower_bound, eps, nullptr, cu,
                                     T_total, H, N, out, final_state, FwdOpts{0, 0},
                                     SegArgs{0, nullptr, nullptr}, err, stream, stamps,
                                     max_chunks);
}

}  // namespace kda
