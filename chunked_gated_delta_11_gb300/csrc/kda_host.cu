// kda_host.cu -- kda_fwd_host: the forward pass on host buffers, with the
// host <-> device copies and the kernels pipelined inside libkda.
//
// The tokens are cut into G pieces, each copied in, run and copied out on
// streams of its own, so that piece g computes while piece g + 1 is copied in
// and piece g - 1 is copied out (the link carries both directions at once):
//   - group mode: G contiguous groups of whole sequences, each one call of
//     kda_forward over its own rebased cu_seqlens;
//   - slice mode (N equal sequences, no cu_seqlens, fewer sequences than
//     pieces, fp32 states): every sequence cut in time into G chunk-aligned
//     slices; slice p of all N sequences is one kda_forward call that starts
//     from the state slice p - 1 left (kept in device memory, fp32, updated in
//     place), which is exact: the recurrence is a left-to-right scan of the
//     state ("You Could Have Come Up with Kimi Delta Attention", sec. 4).
// Every copy is one cudaMemcpyAsync, or one cudaMemcpy2DAsync for the rows of
// all N sequences of a slice.  Streams and events are created once per device
// and reused; a mutex serialises the enqueueing of concurrent calls.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "kda.h"
#include "kda_common.cuh"

namespace kda {
namespace {

constexpr int kHostMaxGroups = 16;
constexpr int kHostDefaultGroups = 8;
constexpr int kMaxDevicesHost = 64;

int64_t r256(int64_t x) { return (x + 255) & ~static_cast<int64_t>(255); }

// One piece of the pipeline: device token range [t0, t1) (slice mode: the
// slice-major device rows), host token rows (group mode: the same range;
// slice mode: [a, b) inside each sequence), sequences [n0, n1).
struct Piece {
  int64_t t0, t1, a, b;
  int32_t n0, n1;
  int64_t ws_off, ws_bytes;  // this piece's kda_forward workspace
};

struct Plan {
  bool slices = false;
  int32_t G = 0;
  size_t gate_row = 0;  // bytes of g_raw per token: H * 256 (per channel) or H * 2
  size_t state_bytes = 0;
  int64_t off_q, off_k, off_v, off_g, off_beta, off_out, off_init, off_fs, off_cu, total;
  std::vector<Piece> pieces;
  std::vector<int32_t> cu_dev;  // group mode: the groups' rebased cu_seqlens, concatenated
};

// Workspace bytes one kda_forward call needs for this shape and schedule.
int64_t call_workspace(int32_t schedule, int64_t T, int32_t H, int32_t N) {
  if (T <= 0) return 0;
  if (schedule == KDA_SCHEDULE_SPLIT) return static_cast<int64_t>(kda_workspace_size(T, H, N, kDim));
  const bool maybe_seg = schedule == KDA_SCHEDULE_SEGMENTED ||
                         (schedule == KDA_SCHEDULE_AUTO && T > 8 * static_cast<int64_t>(N));
  if (maybe_seg && T < (static_cast<int64_t>(1) << 31))
    return static_cast<int64_t>(kda_segmented_workspace_size(T, H, N, kDim, 0));
  return 0;
}

kda_status make_plan(const kda_options* opts, int64_t T_total, int32_t H, int32_t N, int32_t D,
                     const int32_t* cu, int32_t groups, Plan& P) {
  if (!opts) return KDA_ERR_INVALID_ARG;
  const int32_t sc = opts->schedule, sd = opts->state_dtype, gt = opts->gate;
  if (sc < KDA_SCHEDULE_SPLIT || sc > KDA_SCHEDULE_AUTO) return KDA_ERR_INVALID_ARG;
  if ((sd != KDA_STATE_F32 && sd != KDA_STATE_BF16) ||
      (gt != KDA_GATE_PER_CHANNEL && gt != KDA_GATE_PER_HEAD))
    return KDA_ERR_INVALID_ARG;
  if (D != kDim) return KDA_ERR_UNSUPPORTED;
  if (T_total < 0 || H <= 0 || N <= 0 || groups < 0 || groups > kHostMaxGroups)
    return KDA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(N) * H > 0x7fffffffLL ||
      T_total > (static_cast<int64_t>(1) << 40) / (static_cast<int64_t>(H) * kDim))
    return KDA_ERR_INVALID_ARG;
  std::vector<int64_t> bounds(static_cast<size_t>(N) + 1);
  if (cu) {
    // the host array is checked here, on the host
    if (cu[0] != 0 || cu[N] != T_total) return KDA_ERR_INVALID_ARG;
    for (int32_t n = 0; n < N; ++n) {
      if (cu[n + 1] < cu[n]) return KDA_ERR_INVALID_ARG;
    }
    for (int32_t n = 0; n <= N; ++n) bounds[n] = cu[n];
  } else {
    if (T_total % N) return KDA_ERR_INVALID_ARG;
    for (int32_t n = 0; n <= N; ++n) bounds[n] = (T_total / N) * n;
  }
  const int32_t want = groups == 0 ? kHostDefaultGroups : groups;
  const int64_t L = cu ? 0 : T_total / N;
  const int64_t chunks = (L + kChunk - 1) / kChunk;
  P.slices = !cu && N < want && sd == KDA_STATE_F32 && chunks > 1;
  P.gate_row = static_cast<size_t>(H) * (gt == KDA_GATE_PER_HEAD ? 2 : kDim * 2);
  P.state_bytes = static_cast<size_t>(N) * H * kDim * kDim * (sd == KDA_STATE_BF16 ? 2 : 4);
  P.pieces.clear();
  P.cu_dev.clear();
  if (P.slices) {
    const int64_t G = std::min<int64_t>(want, chunks);
    int64_t prev = 0;
    for (int64_t p = 1; p <= G; ++p) {
      const int64_t cut = p == G ? L : std::min<int64_t>(L, kChunk * ((chunks * p) / G));
      if (cut > prev) P.pieces.push_back(Piece{N * prev, N * cut, prev, cut, 0, N, 0, 0});
      prev = cut;
    }
  } else {
    const int32_t G = std::max<int32_t>(1, std::min<int32_t>(want, N));
    for (int32_t g = 0; g < G; ++g) {
      const int32_t n0 = static_cast<int32_t>((static_cast<int64_t>(N) * g) / G);
      const int32_t n1 = static_cast<int32_t>((static_cast<int64_t>(N) * (g + 1)) / G);
      if (n1 == n0) continue;
      P.pieces.push_back(Piece{bounds[n0], bounds[n1], bounds[n0], bounds[n1], n0, n1, 0, 0});
      for (int32_t n = n0; n <= n1; ++n)
        P.cu_dev.push_back(static_cast<int32_t>(bounds[n] - bounds[n0]));
    }
  }
  P.G = static_cast<int32_t>(P.pieces.size());
  // device layout, every part 256-byte aligned
  const int64_t rows = T_total * H;
  int64_t off = 0;
  auto take = [&](int64_t bytes) {
    const int64_t o = off;
    off += r256(bytes);
    return o;
  };
  P.off_q = take(rows * kDim * 2);
  P.off_k = take(rows * kDim * 2);
  P.off_v = take(rows * kDim * 2);
  P.off_g = take(T_total * static_cast<int64_t>(P.gate_row));
  P.off_beta = take(rows * 2);
  P.off_out = take(rows * kDim * 2);
  P.off_init = take(static_cast<int64_t>(P.state_bytes));
  P.off_fs = take(static_cast<int64_t>(P.state_bytes));
  P.off_cu = take(static_cast<int64_t>(P.cu_dev.size()) * 4 + 4);
  // slices run one after another on one stream and share one workspace
  int64_t shared_ws = 0;
  for (Piece& pc : P.pieces) {
    const int32_t n = pc.n1 - pc.n0;
    const int64_t need = call_workspace(sc, pc.t1 - pc.t0, H, n);
    if (P.slices) {
      shared_ws = std::max(shared_ws, need);
    } else {
      pc.ws_off = take(need);
      pc.ws_bytes = need;
    }
  }
  if (P.slices) {
    const int64_t o = take(shared_ws);
    for (Piece& pc : P.pieces) {
      pc.ws_off = o;
      pc.ws_bytes = shared_ws;
    }
  }
  P.total = off;
  return KDA_OK;
}

// Streams and events of one device, created on first use and kept.
struct HostPipe {
  bool ready = false;
  cudaStream_t copy_in = nullptr, copy_out = nullptr;
  cudaStream_t work[kHostMaxGroups] = {};
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t in[kHostMaxGroups] = {}, done[kHostMaxGroups] = {};
};
std::mutex g_host_mu;
HostPipe g_pipe[kMaxDevicesHost];

kda_status pipe_for_device(HostPipe*& out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesHost)
    return KDA_ERR_LAUNCH;
  HostPipe& p = g_pipe[dev];
  if (!p.ready) {
    // handles that exist are kept, so a call after a failed creation only
    // creates the missing ones
    const unsigned sf = cudaStreamNonBlocking, ef = cudaEventDisableTiming;
    auto stream = [&](cudaStream_t& x) { return x || cudaStreamCreateWithFlags(&x, sf) == cudaSuccess; };
    auto event = [&](cudaEvent_t& x) { return x || cudaEventCreateWithFlags(&x, ef) == cudaSuccess; };
    bool ok = stream(p.copy_in) && stream(p.copy_out) && event(p.start) && event(p.end);
    for (int g = 0; ok && g < kHostMaxGroups; ++g)
      ok = stream(p.work[g]) && event(p.in[g]) && event(p.done[g]);
    if (!ok) {
      cudaGetLastError();
      return KDA_ERR_LAUNCH;
    }
    p.ready = true;
  }
  out = &p;
  return KDA_OK;
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" size_t kda_fwd_host_workspace_size(const kda_options* opts, int64_t T_total,
                                              int32_t H, int32_t N, int32_t D,
                                              const int32_t* cu_seqlens, int32_t groups) {
  Plan P;
  if (make_plan(opts, T_total, H, N, D, cu_seqlens, groups, P) != KDA_OK) return 0;
  return static_cast<size_t>(P.total);
}

extern "C" kda_status kda_fwd_host(const kda_options* opts, const void* q, const void* k,
                                   const void* v, const void* g_raw, const void* beta_raw,
                                   float scale, float lower_bound, const void* initial_state,
                                   const int32_t* cu_seqlens, int64_t T_total, int32_t H,
                                   int32_t N, int32_t D, void* out, void* final_state,
                                   int32_t groups, void* workspace, size_t workspace_bytes,
                                   void* stream) {
  Plan P;
  kda_status s = make_plan(opts, T_total, H, N, D, cu_seqlens, groups, P);
  if (s != KDA_OK) return s;
  if (!(lower_bound >= -5.0f && lower_bound <= 0.0f)) return KDA_ERR_UNSUPPORTED;
  if (T_total > 0 && (!q || !k || !v || !g_raw || !beta_raw || !out)) return KDA_ERR_INVALID_ARG;
  if (workspace && ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
                    workspace_bytes < static_cast<size_t>(P.total)))
    return KDA_ERR_WORKSPACE;
  std::lock_guard<std::mutex> lock(g_host_mu);
  HostPipe* pipe = nullptr;
  if ((s = pipe_for_device(pipe)) != KDA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* ws = workspace;
  if (!ws) {
    if (cudaMallocAsync(&ws, static_cast<size_t>(P.total), st) != cudaSuccess) {
      cudaGetLastError();
      return KDA_ERR_WORKSPACE;
    }
  }
  uint8_t* base = static_cast<uint8_t*>(ws);
  auto dptr = [&](int64_t off) { return static_cast<void*>(base + off); };
  const auto* hq = static_cast<const uint8_t*>(q);
  const auto* hk = static_cast<const uint8_t*>(k);
  const auto* hv = static_cast<const uint8_t*>(v);
  const auto* hg = static_cast<const uint8_t*>(g_raw);
  const auto* hb = static_cast<const uint8_t*>(beta_raw);
  auto* ho = static_cast<uint8_t*>(out);
  const size_t row = static_cast<size_t>(H) * kDim * 2;  // bytes of one token of q, k, v, out
  const size_t brow = static_cast<size_t>(H) * 2;        // of beta_raw
  const size_t state_one = P.state_bytes / static_cast<size_t>(N);
  cudaError_t e = cudaSuccess;
  auto ok = [&](cudaError_t r) {
    if (e == cudaSuccess && r != cudaSuccess) e = r;
    return e == cudaSuccess;
  };
  // one copy; empty ranges (empty groups, no tokens) are skipped
  auto copy = [&](void* dst, const void* src, size_t bytes, cudaMemcpyKind kind, cudaStream_t cs) {
    if (bytes) ok(cudaMemcpyAsync(dst, src, bytes, kind, cs));
  };
  // everything below is ordered after the work already queued on `stream`
  ok(cudaEventRecord(pipe->start, st));
  ok(cudaStreamWaitEvent(pipe->copy_in, pipe->start, 0));
  ok(cudaStreamWaitEvent(pipe->copy_out, pipe->start, 0));
  kda_status fs = KDA_OK;  // status of the kernel calls
  // the groups' rebased cu_seqlens (a pageable copy of this local vector:
  // cudaMemcpyAsync has staged it when it returns)
  if (cu_seqlens && !P.cu_dev.empty())
    copy(dptr(P.off_cu), P.cu_dev.data(), P.cu_dev.size() * 4, cudaMemcpyHostToDevice,
         pipe->copy_in);
  // the initial states all at once (slice mode: into the running state buffer)
  const bool have_init = initial_state != nullptr;
  if (have_init)
    copy(dptr(P.slices ? P.off_fs : P.off_init), initial_state, P.state_bytes,
         cudaMemcpyHostToDevice, pipe->copy_in);
  const kda_options fo = *opts;
  size_t cu_pos = 0;
  for (int32_t i = 0; i < P.G && e == cudaSuccess && fs == KDA_OK; ++i) {
    const Piece& pc = P.pieces[i];
    const int32_t n = pc.n1 - pc.n0;
    const int64_t rows_p = pc.t1 - pc.t0;
    cudaStream_t work = pipe->work[P.slices ? 0 : i];
    if (P.slices) {
      // rows [a, b) of each of the N sequences -> rows [t0 + s n_p, ...) of the slice
      const int64_t L = T_total / N, np = pc.b - pc.a;
      struct {
        int64_t off;
        const uint8_t* h;
        size_t rb;
      } ins[] = {{P.off_q, hq, row}, {P.off_k, hk, row}, {P.off_v, hv, row},
                 {P.off_g, hg, P.gate_row}, {P.off_beta, hb, brow}};
      for (auto& x : ins)
        ok(cudaMemcpy2DAsync(base + x.off + pc.t0 * x.rb, np * x.rb, x.h + pc.a * x.rb, L * x.rb,
                             np * x.rb, static_cast<size_t>(N), cudaMemcpyHostToDevice,
                             pipe->copy_in));
    } else {
      const size_t t0 = static_cast<size_t>(pc.t0), nr = static_cast<size_t>(rows_p);
      const auto h2d = cudaMemcpyHostToDevice;
      if (nr) {
        copy(base + P.off_q + t0 * row, hq + t0 * row, nr * row, h2d, pipe->copy_in);
        copy(base + P.off_k + t0 * row, hk + t0 * row, nr * row, h2d, pipe->copy_in);
        copy(base + P.off_v + t0 * row, hv + t0 * row, nr * row, h2d, pipe->copy_in);
        copy(base + P.off_g + t0 * P.gate_row, hg + t0 * P.gate_row, nr * P.gate_row, h2d,
             pipe->copy_in);
        copy(base + P.off_beta + t0 * brow, hb + t0 * brow, nr * brow, h2d, pipe->copy_in);
      }
    }
    ok(cudaEventRecord(pipe->in[i], pipe->copy_in));
    ok(cudaStreamWaitEvent(work, pipe->in[i], 0));
    if (e != cudaSuccess) break;
    // the piece's pass
    const size_t t0 = static_cast<size_t>(pc.t0);
    const void* init_d = nullptr;
    void* fs_d = nullptr;
    const int32_t* cu_d = nullptr;
    if (P.slices) {
      init_d = (i > 0 || have_init) ? dptr(P.off_fs) : nullptr;
      fs_d = dptr(P.off_fs);
    } else {
      init_d = have_init ? static_cast<const void*>(base + P.off_init + pc.n0 * state_one)
                         : nullptr;
      fs_d = base + P.off_fs + pc.n0 * state_one;
      if (cu_seqlens) cu_d = reinterpret_cast<const int32_t*>(base + P.off_cu) + cu_pos;
      cu_pos += static_cast<size_t>(n) + 1;
    }
    fs = kda_forward(&fo, base + P.off_q + t0 * row, base + P.off_k + t0 * row,
                     base + P.off_v + t0 * row, base + P.off_g + t0 * P.gate_row,
                     base + P.off_beta + t0 * brow, scale, lower_bound, init_d, cu_d, rows_p, H,
                     n, D, base + P.off_out + t0 * row, fs_d,
                     pc.ws_bytes ? dptr(pc.ws_off) : nullptr, static_cast<size_t>(pc.ws_bytes),
                     work);
    if (fs != KDA_OK) break;
    ok(cudaEventRecord(pipe->done[i], work));
    ok(cudaStreamWaitEvent(pipe->copy_out, pipe->done[i], 0));
    if (P.slices) {
      const int64_t L = T_total / N, np = pc.b - pc.a;
      ok(cudaMemcpy2DAsync(ho + pc.a * row, L * row, base + P.off_out + t0 * row, np * row,
                           np * row, static_cast<size_t>(N), cudaMemcpyDeviceToHost,
                           pipe->copy_out));
    } else {
      if (rows_p)
        copy(ho + t0 * row, base + P.off_out + t0 * row, static_cast<size_t>(rows_p) * row,
             cudaMemcpyDeviceToHost, pipe->copy_out);
      if (final_state)
        copy(static_cast<uint8_t*>(final_state) + pc.n0 * state_one, fs_d,
             static_cast<size_t>(n) * state_one, cudaMemcpyDeviceToHost, pipe->copy_out);
    }
  }
  if (final_state && e == cudaSuccess && fs == KDA_OK) {
    if (P.slices) {
      if (P.G > 0) {
        ok(cudaMemcpyAsync(final_state, dptr(P.off_fs), P.state_bytes, cudaMemcpyDeviceToHost,
                           pipe->copy_out));
      } else if (have_init) {
        std::memcpy(final_state, initial_state, P.state_bytes);
      } else {
        std::memset(final_state, 0, P.state_bytes);
      }
    } else if (P.G == 0) {
      // no tokens and no groups: the final state is the initial one
      if (have_init)
        std::memcpy(final_state, initial_state, P.state_bytes);
      else
        std::memset(final_state, 0, P.state_bytes);
    }
  }
  // join every stream back into the caller's stream, also after an error
  for (int32_t i = 0; i < (P.slices ? 1 : P.G); ++i) {
    cudaEventRecord(pipe->done[i], pipe->work[i]);
    cudaStreamWaitEvent(pipe->copy_out, pipe->done[i], 0);
  }
  cudaEventRecord(pipe->in[0], pipe->copy_in);
  cudaStreamWaitEvent(pipe->copy_out, pipe->in[0], 0);
  cudaEventRecord(pipe->end, pipe->copy_out);
  cudaStreamWaitEvent(st, pipe->end, 0);
  if (!workspace) cudaFreeAsync(ws, st);
  if (fs != KDA_OK) return fs;
  return e == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}
