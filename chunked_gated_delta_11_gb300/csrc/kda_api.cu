// kda_api.cu -- host side of the libkda C ABI (include/kda.h): argument
// validation, workspace sizing, kernel launches and the device error word.
#include <cstdint>
#include <cstring>
#include <mutex>

#include "kda.h"
#include "kda_common.cuh"

namespace kda {

cudaError_t launch_chunk_prep(const void* q, const void* k, const void* v, const void* g,
                              const void* beta_raw, float scale, float lower_bound, float eps,
                              const int32_t* cu, int64_t T_total, int H, int N, void* ws,
                              int gate_scalar, int sm_count, int* err, cudaStream_t stream);
cudaError_t launch_recurrence(const void* ws, const void* init, const int32_t* cu,
                              int64_t T_total, int H, int N, void* out, void* final_state,
                              FwdOpts opts, int* err, cudaStream_t stream);
cudaError_t launch_fused(const void* q, const void* k, const void* v, const void* g,
                         const void* beta_raw, float scale, float lower_bound, float eps,
                         const void* init, const int32_t* cu, int64_t T_total, int H, int N,
                         void* out, void* final_state, FwdOpts opts, SegArgs seg, int* err,
                         cudaStream_t stream);
cudaError_t launch_seg_plan(const int32_t* cu, int64_t T_total, int N, int P, int32_t* cu_seg,
                            int32_t* blk, cudaStream_t stream);
// s0_bf16 / sstart16 (optional): a bf16 copy of every later segment's S_0,
// written by the scan and read by the fix-up instead of converting S_0
cudaError_t launch_affine_scan(float* xs, const float* ms, int N, int P, int H,
                               void* final_state, bool final_bf16, int sm_count,
                               cudaStream_t stream, void* s0_bf16);
cudaError_t launch_seg_fixup(const int32_t* cu_seg, const int32_t* blk, int Nseg, int H,
                             const float* sstart, const void* y, void* out, int sm_count,
                             cudaStream_t stream, const void* sstart16);
cudaError_t launch_selftest_timeout(long long limit, int* err, cudaStream_t stream);
cudaError_t launch_recurrence_timed(const void* ws, const void* init, const int32_t* cu,
                                    int64_t T_total, int H, int N, void* out, void* final_state,
                                    FwdOpts opts, int* err, long long* stamps, int max_chunks,
                                    cudaStream_t stream);
cudaError_t launch_fused_timed(const void* q, const void* k, const void* v, const void* g,
                               const void* beta_raw, float scale, float lower_bound, float eps,
                               const int32_t* cu, int64_t T_total, int H, int N, void* out,
                               void* final_state, int* err, long long* stamps, int max_chunks,
                               cudaStream_t stream);
cudaError_t launch_decode(const void* q, const void* k, const void* v, const void* g,
                          const void* beta_raw, float scale, float lower_bound, float eps,
                          const void* init, const int32_t* cu, int64_t T_total, int H, int N,
                          void* out, void* final_state, FwdOpts opts, cudaStream_t stream);

// Error word written by kernels: KDA_ERR_TIMEOUT when a bounded wait runs out,
// KDA_ERR_INVALID_ARG when validate_cu_kernel finds a bad cu_seqlens.  Kernels
// get its address as an argument; cudaGetSymbolAddress is resolved once per
// device.
__device__ int g_kda_error = 0;

// cu_seqlens must start at 0, be non-decreasing and end at T_total.  One
// thread per entry; the first violation found latches KDA_ERR_INVALID_ARG
// (later ones leave it).  No trap: the host reads the word back.
__global__ void validate_cu_kernel(const int32_t* __restrict__ cu, int N, int64_t T_total,
                                   int* __restrict__ err) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i <= N; i += gridDim.x * blockDim.x) {
    const int64_t c = __ldg(cu + i);
    bool bad = (i == 0 && c != 0) || (i == N && c != T_total);
    if (i < N) bad = bad || __ldg(cu + i + 1) < c;
    if (bad) atomicCAS(err, 0, static_cast<int>(KDA_ERR_INVALID_ARG));
  }
}

namespace {

constexpr float kNormEps = 1e-6f;
constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int sm_count = 0;
  int* err = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

kda_status device_info(DeviceInfo& out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.err == nullptr) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return KDA_ERR_LAUNCH;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_kda_error) != cudaSuccess || p == nullptr)
      return KDA_ERR_LAUNCH;
    d.sm_count = sms;
    d.err = static_cast<int*>(p);
  }
  out = d;
  return KDA_OK;
}

}  // namespace

// The device error word of the current device, for the entry points in the
// other translation units.
kda_status error_word(int** out) {
  DeviceInfo info;
  const kda_status s = device_info(info);
  if (s == KDA_OK) *out = info.err;
  return s;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kda_status check_sizes(int64_t T_total, int32_t H, int32_t N, int32_t D,
                       const int32_t* cu_seqlens) {
  if (D != KDA_HEAD_DIM) return KDA_ERR_UNSUPPORTED;
  if (T_total < 0 || H <= 0 || N <= 0) return KDA_ERR_INVALID_ARG;
  if (!cu_seqlens && (T_total % N) != 0) return KDA_ERR_INVALID_ARG;
  // grid and index limits: one CTA per (sequence, head); element offsets in int64
  if (static_cast<int64_t>(N) * H > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
  if (T_total > (static_cast<int64_t>(1) << 40) / (static_cast<int64_t>(H) * KDA_HEAD_DIM))
    return KDA_ERR_INVALID_ARG;
  // token coordinates of the tensor-map copies are int32
  if (T_total >= (static_cast<int64_t>(1) << 31)) return KDA_ERR_INVALID_ARG;
  return KDA_OK;
}

bool aligned2(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1u) == 0; }

kda_status check_inputs(const void* q, const void* k, const void* v, const void* g,
                        const void* beta_raw, float scale, float lower_bound, int64_t T_total,
                        bool gate_scalar = false) {
  if (!(lower_bound >= -5.0f && lower_bound <= 0.0f)) return KDA_ERR_UNSUPPORTED;
  if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f) return KDA_ERR_INVALID_ARG;
  if (T_total > 0) {
    if (!q || !k || !v || !g || !beta_raw) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return KDA_ERR_INVALID_ARG;
    if (gate_scalar ? !aligned2(g) : !aligned16(g)) return KDA_ERR_INVALID_ARG;
    if (!aligned2(beta_raw)) return KDA_ERR_INVALID_ARG;
  }
  return KDA_OK;
}

kda_status check_outputs(const void* out, const void* initial_state, const void* final_state,
                         int64_t T_total) {
  if (T_total > 0 && (!out || !aligned16(out))) return KDA_ERR_INVALID_ARG;
  if (initial_state && !aligned16(initial_state)) return KDA_ERR_INVALID_ARG;
  if (final_state && !aligned16(final_state)) return KDA_ERR_INVALID_ARG;
  return KDA_OK;
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" size_t kda_workspace_size(int64_t T_total, int32_t H, int32_t N, int32_t D) {
  if (check_sizes(T_total, H, N, D, reinterpret_cast<const int32_t*>(1)) != KDA_OK) return 0;
  const int64_t bytes = slot_count(T_total, N) * H * static_cast<int64_t>(REC_BYTES);
  return static_cast<size_t>((bytes + 255) & ~static_cast<int64_t>(255));
}

namespace {

// The forward pass behind every entry point.  schedule: 0 split (K1 then K2
// through `workspace`, or one allocated on the stream), 1 fused, 2 decode.
kda_status forward(int schedule, FwdOpts opts, const void* q, const void* k, const void* v,
                   const void* g_raw, const void* beta_raw, float scale, float lower_bound,
                   const void* initial_state, const int32_t* cu_seqlens, int64_t T_total,
                   int32_t H, int32_t N, int32_t D, void* out, void* final_state,
                   void* workspace, size_t workspace_bytes, void* stream) {
  kda_status s = check_sizes(T_total, H, N, D, cu_seqlens);
  if (s != KDA_OK) return s;
  if ((s = check_inputs(q, k, v, g_raw, beta_raw, scale, lower_bound, T_total,
                        opts.gate_scalar != 0)) != KDA_OK)
    return s;
  if ((s = check_outputs(out, initial_state, final_state, T_total)) != KDA_OK) return s;
  const size_t need = schedule == 0 ? kda_workspace_size(T_total, H, N, D) : 0;
  if (schedule == 0 && workspace && (!aligned16(workspace) || workspace_bytes < need))
    return KDA_ERR_WORKSPACE;
  DeviceInfo info;
  if ((s = device_info(info)) != KDA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (schedule == 1) {
    e = launch_fused(q, k, v, g_raw, beta_raw, scale, lower_bound, kNormEps, initial_state,
                     cu_seqlens, T_total, H, N, out, final_state, opts, SegArgs{0, nullptr, nullptr},
                     info.err, st);
  } else if (schedule == 2) {
    e = launch_decode(q, k, v, g_raw, beta_raw, scale, lower_bound, kNormEps, initial_state,
                      cu_seqlens, T_total, H, N, out, final_state, opts, st);
  } else {
    void* ws = workspace;
    if (!ws) {
      if (cudaMallocAsync(&ws, need, st) != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_WORKSPACE;
      }
    }
    if (T_total > 0)
      e = launch_chunk_prep(q, k, v, g_raw, beta_raw, scale, lower_bound, kNormEps, cu_seqlens,
                            T_total, H, N, ws, opts.gate_scalar, info.sm_count, info.err, st);
    if (e == cudaSuccess)
      e = launch_recurrence(ws, initial_state, cu_seqlens, T_total, H, N, out, final_state, opts,
                            info.err, st);
    if (!workspace) cudaFreeAsync(ws, st);
  }
  return e == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

}  // namespace

extern "C" kda_status kda_chunk_prep(const void* q, const void* k, const void* v,
                                     const void* g_raw, const void* beta_raw, float scale,
                                     float lower_bound, const int32_t* cu_seqlens,
                                     int64_t T_total, int32_t H, int32_t N, int32_t D,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  kda_status s = check_sizes(T_total, H, N, D, cu_seqlens);
  if (s != KDA_OK) return s;
  s = check_inputs(q, k, v, g_raw, beta_raw, scale, lower_bound, T_total);
  if (s != KDA_OK) return s;
  if (!workspace || !aligned16(workspace)) return KDA_ERR_INVALID_ARG;
  if (workspace_bytes < kda_workspace_size(T_total, H, N, D)) return KDA_ERR_WORKSPACE;
  DeviceInfo info;
  if ((s = device_info(info)) != KDA_OK) return s;
  if (T_total == 0) return KDA_OK;
  cudaError_t e = launch_chunk_prep(q, k, v, g_raw, beta_raw, scale, lower_bound, kNormEps,
                                    cu_seqlens, T_total, H, N, workspace, 0, info.sm_count,
                                    info.err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

extern "C" kda_status kda_chunk_recurrence(const void* workspace, size_t workspace_bytes,
                                           const float* initial_state,
                                           const int32_t* cu_seqlens, int64_t T_total,
                                           int32_t H, int32_t N, int32_t D, void* out,
                                           float* final_state, void* stream) {
  kda_status s = check_sizes(T_total, H, N, D, cu_seqlens);
  if (s != KDA_OK) return s;
  if ((s = check_outputs(out, initial_state, final_state, T_total)) != KDA_OK) return s;
  if (!workspace || !aligned16(workspace)) return KDA_ERR_INVALID_ARG;
  if (workspace_bytes < kda_workspace_size(T_total, H, N, D)) return KDA_ERR_WORKSPACE;
  DeviceInfo info;
  if ((s = device_info(info)) != KDA_OK) return s;
  cudaError_t e = launch_recurrence(workspace, initial_state, cu_seqlens, T_total, H, N, out,
                                    final_state, FwdOpts{0, 0}, info.err,
                                    static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

extern "C" kda_status kda_fwd(const void* q, const void* k, const void* v, const void* g_raw,
                              const void* beta_raw, float scale, float lower_bound,
                              const float* initial_state, const int32_t* cu_seqlens,
                              int64_t T_total, int32_t H, int32_t N, int32_t D, void* out,
                              float* final_state, void* workspace, size_t workspace_bytes,
                              void* stream) {
  return forward(0, FwdOpts{0, 0}, q, k, v, g_raw, beta_raw, scale, lower_bound, initial_state,
                 cu_seqlens, T_total, H, N, D, out, final_state, workspace, workspace_bytes,
                 stream);
}

extern "C" kda_status kda_fwd_fused(const void* q, const void* k, const void* v,
                                    const void* g_raw, const void* beta_raw, float scale,
                                    float lower_bound, const float* initial_state,
                                    const int32_t* cu_seqlens, int64_t T_total, int32_t H,
                                    int32_t N, int32_t D, void* out, float* final_state,
                                    void* stream) {
  return forward(1, FwdOpts{0, 0}, q, k, v, g_raw, beta_raw, scale, lower_bound, initial_state,
                 cu_seqlens, T_total, H, N, D, out, final_state, nullptr, 0, stream);
}

extern "C" kda_status kda_decode(const void* q, const void* k, const void* v, const void* g_raw,
                                 const void* beta_raw, float scale, float lower_bound,
                                 const float* initial_state, const int32_t* cu_seqlens,
                                 int64_t T_total, int32_t H, int32_t N, int32_t D, void* out,
                                 float* final_state, void* stream) {
  return forward(2, FwdOpts{0, 0}, q, k, v, g_raw, beta_raw, scale, lower_bound, initial_state,
                 cu_seqlens, T_total, H, N, D, out, final_state, nullptr, 0, stream);
}

namespace {
int32_t auto_segments(int64_t T_total, int32_t H, int32_t N, int sms);
kda_status segmented_forward(FwdOpts opts, const void* q, const void* k, const void* v,
                             const void* g_raw, const void* beta_raw, float scale,
                             float lower_bound, const void* initial_state,
                             const int32_t* cu_seqlens, int64_t T_total, int32_t H, int32_t N,
                             int32_t D, void* out, void* final_state, int32_t segments,
                             void* workspace, size_t workspace_bytes, void* stream);
}  // namespace

extern "C" kda_status kda_forward(const kda_options* opts, const void* q, const void* k,
                                  const void* v, const void* g_raw, const void* beta_raw,
                                  float scale, float lower_bound, const void* initial_state,
                                  const int32_t* cu_seqlens, int64_t T_total, int32_t H,
                                  int32_t N, int32_t D, void* out, void* final_state,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  if (!opts) return KDA_ERR_INVALID_ARG;
  const int32_t sc = opts->schedule, sd = opts->state_dtype, gt = opts->gate;
  if (sc != KDA_SCHEDULE_SPLIT && sc != KDA_SCHEDULE_FUSED && sc != KDA_SCHEDULE_DECODE &&
      sc != KDA_SCHEDULE_SEGMENTED && sc != KDA_SCHEDULE_AUTO)
    return KDA_ERR_INVALID_ARG;
  if ((sd != KDA_STATE_F32 && sd != KDA_STATE_BF16) ||
      (gt != KDA_GATE_PER_CHANNEL && gt != KDA_GATE_PER_HEAD))
    return KDA_ERR_INVALID_ARG;
  int32_t sched = sc;
  if (sc == KDA_SCHEDULE_AUTO) {
    kda_status s = check_sizes(T_total, H, N, D, cu_seqlens);
    if (s != KDA_OK) return s;
    DeviceInfo info;
    if ((s = device_info(info)) != KDA_OK) return s;
    if (T_total <= 8 * static_cast<int64_t>(N))
      sched = KDA_SCHEDULE_DECODE;  // serving steps: the state traffic dominates
    else if (T_total < (static_cast<int64_t>(1) << 31) &&
             auto_segments(T_total, H, N, info.sm_count) > 1)
      sched = KDA_SCHEDULE_SEGMENTED;  // too few units for the SMs
    else
      sched = KDA_SCHEDULE_FUSED;
  }
  if (sched == KDA_SCHEDULE_SEGMENTED)
    return segmented_forward(FwdOpts{sd == KDA_STATE_BF16, gt == KDA_GATE_PER_HEAD}, q, k, v,
                             g_raw, beta_raw, scale, lower_bound, initial_state, cu_seqlens,
                             T_total, H, N, D, out, final_state, 0, workspace, workspace_bytes,
                             stream);
  const int schedule = sched == KDA_SCHEDULE_SPLIT ? 0 : sched == KDA_SCHEDULE_FUSED ? 1 : 2;
  return forward(schedule, FwdOpts{sd == KDA_STATE_BF16, gt == KDA_GATE_PER_HEAD}, q, k, v,
                 g_raw, beta_raw, scale, lower_bound, initial_state, cu_seqlens, T_total, H, N,
                 D, out, final_state, workspace, workspace_bytes, stream);
}

namespace {

constexpr int kMaxSegments = 64;

int64_t round256(int64_t x) { return (x + 255) & ~static_cast<int64_t>(255); }

// Byte offsets of the segmented pass's workspace parts (each 256-byte aligned):
// cu_seg and blk [N P + 1] int32, the X and M final states [N P, H, 128, 128]
// fp32, the segments' starting states as bf16 [N P, H, 128, 128] (written by
// the scan for the fix-up), the M outputs y [T_total, H, 128] bf16.
struct SegLayout {
  int64_t cu, blk, xs, ms, sb, y, total;
};
SegLayout seg_layout(int64_t T_total, int32_t H, int32_t N, int32_t P) {
  SegLayout L;
  const int64_t ns = static_cast<int64_t>(N) * P;
  const int64_t states = ns * H * KDA_HEAD_DIM * KDA_HEAD_DIM * 4;
  L.cu = 0;
  L.blk = L.cu + round256((ns + 1) * 4);
  L.xs = L.blk + round256((ns + 1) * 4);
  L.ms = L.xs + round256(states);
  L.sb = L.ms + round256(states);
  L.y = L.sb + round256(states / 2);
  L.total = L.y + round256(T_total * H * KDA_HEAD_DIM * 2);
  return L;
}

// Segments per sequence for a device with `sms` SMs: the fused kernel runs
// two CTAs per SM, and P segments take N H (2 P - 1) CTAs (X roles for all,
// M roles for all but the first); each segment keeps at least 24 chunks
// (fewer cost more in the scan and fix-up than they save in the chain).
int32_t auto_segments(int64_t T_total, int32_t H, int32_t N, int sms) {
  const int64_t units = static_cast<int64_t>(N) * H;
  if (units <= 0 || sms <= 0) return 1;
  int64_t P = (2 * static_cast<int64_t>(sms) / units + 1) / 2;
  const int64_t chunks = (T_total / N + 15) / 16;
  if (P > chunks / 24) P = chunks / 24;
  if (P > kMaxSegments) P = kMaxSegments;
  return static_cast<int32_t>(P < 1 ? 1 : P);
}

kda_status seg_checks(int64_t T_total, int32_t H, int32_t N, int32_t D, int32_t segments,
                      const int32_t* cu_seqlens) {
  kda_status s = check_sizes(T_total, H, N, D, cu_seqlens);
  if (s != KDA_OK) return s;
  if (segments < 0 || segments > kMaxSegments) return KDA_ERR_INVALID_ARG;
  if (T_total >= (static_cast<int64_t>(1) << 31)) return KDA_ERR_INVALID_ARG;  // int32 boundaries
  if (static_cast<int64_t>(N) * kMaxSegments * H * 2 > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
  return KDA_OK;
}

}  // namespace

extern "C" int32_t kda_segments_auto(int64_t T_total, int32_t H, int32_t N) {
  if (check_sizes(T_total, H, N, KDA_HEAD_DIM, reinterpret_cast<const int32_t*>(1)) != KDA_OK)
    return 1;
  DeviceInfo info;
  if (device_info(info) != KDA_OK) return 1;
  return auto_segments(T_total, H, N, info.sm_count);
}

extern "C" size_t kda_segmented_workspace_size(int64_t T_total, int32_t H, int32_t N, int32_t D,
                                               int32_t segments) {
  if (seg_checks(T_total, H, N, D, segments, reinterpret_cast<const int32_t*>(1)) != KDA_OK)
    return 0;
  const int32_t P = segments == 0 ? kda_segments_auto(T_total, H, N) : segments;
  if (P <= 1) return 0;
  return static_cast<size_t>(seg_layout(T_total, H, N, P).total);
}

namespace {

// The segmented pass behind kda_fwd_segmented and KDA_SCHEDULE_SEGMENTED.
kda_status segmented_forward(FwdOpts opts, const void* q, const void* k, const void* v,
                             const void* g_raw, const void* beta_raw, float scale,
                             float lower_bound, const void* initial_state,
                             const int32_t* cu_seqlens, int64_t T_total, int32_t H, int32_t N,
                             int32_t D, void* out, void* final_state, int32_t segments,
                             void* workspace, size_t workspace_bytes, void* stream) {
  kda_status s = seg_checks(T_total, H, N, D, segments, cu_seqlens);
  if (s != KDA_OK) return s;
  if ((s = check_inputs(q, k, v, g_raw, beta_raw, scale, lower_bound, T_total,
                        opts.gate_scalar != 0)) != KDA_OK)
    return s;
  if ((s = check_outputs(out, initial_state, final_state, T_total)) != KDA_OK) return s;
  DeviceInfo info;
  if ((s = device_info(info)) != KDA_OK) return s;
  const int32_t P = segments == 0 ? auto_segments(T_total, H, N, info.sm_count) : segments;
  if (P <= 1 || T_total == 0)
    return forward(1, opts, q, k, v, g_raw, beta_raw, scale, lower_bound, initial_state,
                   cu_seqlens, T_total, H, N, D, out, final_state, nullptr, 0, stream);
  const SegLayout L = seg_layout(T_total, H, N, P);
  if (workspace && (!aligned16(workspace) || workspace_bytes < static_cast<size_t>(L.total)))
    return KDA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* ws = workspace;
  if (!ws) {
    if (cudaMallocAsync(&ws, static_cast<size_t>(L.total), st) != cudaSuccess) {
      cudaGetLastError();
      return KDA_ERR_WORKSPACE;
    }
  }
  uint8_t* wb = static_cast<uint8_t*>(ws);
  int32_t* cu_seg = reinterpret_cast<int32_t*>(wb + L.cu);
  int32_t* blk = reinterpret_cast<int32_t*>(wb + L.blk);
  float* xs = reinterpret_cast<float*>(wb + L.xs);
  float* ms = reinterpret_cast<float*>(wb + L.ms);
  __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(wb + L.y);
  void* sb = wb + L.sb;
  const int Nseg = N * P;
  cudaError_t e = launch_seg_plan(cu_seqlens, T_total, N, P, cu_seg, blk, st);
  if (e == cudaSuccess)
    e = launch_fused(q, k, v, g_raw, beta_raw, scale, lower_bound, kNormEps, initial_state,
                     cu_seg, T_total, H, Nseg, out, xs, opts, SegArgs{P, y, ms}, info.err, st);
  if (e == cudaSuccess)
    e = launch_affine_scan(xs, ms, N, P, H, final_state, opts.state_bf16 != 0, info.sm_count, st,
                           sb);
  if (e == cudaSuccess)
    e = launch_seg_fixup(cu_seg, blk, Nseg, H, xs, y, out, info.sm_count, st, sb);
  if (!workspace) cudaFreeAsync(ws, st);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

}  // namespace

extern "C" kda_status kda_fwd_segmented(const void* q, const void* k, const void* v,
                                        const void* g_raw, const void* beta_raw, float scale,
                                        float lower_bound, const float* initial_state,
                                        const int32_t* cu_seqlens, int64_t T_total, int32_t H,
                                        int32_t N, int32_t D, void* out, float* final_state,
                                        int32_t segments, int32_t gate, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  if (gate != KDA_GATE_PER_CHANNEL && gate != KDA_GATE_PER_HEAD) return KDA_ERR_INVALID_ARG;
  return segmented_forward(FwdOpts{0, gate == KDA_GATE_PER_HEAD}, q, k, v, g_raw, beta_raw,
                           scale, lower_bound, initial_state, cu_seqlens, T_total, H, N, D, out,
                           final_state, segments, workspace, workspace_bytes, stream);
}

extern "C" kda_status kda_device_status(void* stream) {
  DeviceInfo info;
  kda_status s = device_info(info);
  if (s != KDA_OK) return s;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return KDA_ERR_LAUNCH;
  int word = 0;
  if (cudaMemcpy(&word, info.err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return KDA_ERR_LAUNCH;
  if (word != 0) {
    const int zero = 0;
    if (cudaMemcpy(info.err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return KDA_ERR_LAUNCH;
    return word == KDA_ERR_INVALID_ARG ? KDA_ERR_INVALID_ARG : KDA_ERR_TIMEOUT;
  }
  return KDA_OK;
}

extern "C" kda_status kda_validate_cu_seqlens(const int32_t* cu_seqlens, int32_t N,
                                              int64_t T_total, void* stream) {
  if (!cu_seqlens || N <= 0 || T_total < 0 || T_total >= (static_cast<int64_t>(1) << 31) ||
      (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0)
    return KDA_ERR_INVALID_ARG;
  DeviceInfo info;
  const kda_status s = device_info(info);
  if (s != KDA_OK) return s;
  const int threads = 256;
  const int64_t blocks = (static_cast<int64_t>(N) + threads) / threads;
  validate_cu_kernel<<<static_cast<unsigned>(blocks < 1024 ? blocks : 1024), threads, 0,
                       static_cast<cudaStream_t>(stream)>>>(cu_seqlens, N, T_total, info.err);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

extern "C" kda_status kda_selftest_timeout(int64_t limit_cycles, void* stream) {
  if (limit_cycles < 1 || limit_cycles > kWaitLimitCycles) return KDA_ERR_INVALID_ARG;
  DeviceInfo info;
  const kda_status s = device_info(info);
  if (s != KDA_OK) return s;
  return launch_selftest_timeout(limit_cycles, info.err, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? KDA_OK
             : KDA_ERR_LAUNCH;
}

extern "C" kda_status kda_profile_phases(int32_t kernel, const void* q, const void* k,
                                         const void* v, const void* g_raw, const void* beta_raw,
                                         float scale, float lower_bound, int64_t T_total,
                                         int32_t H, int32_t N, int32_t D, void* out,
                                         float* final_state, void* workspace,
                                         size_t workspace_bytes, long long* stamps,
                                         int32_t max_chunks, void* stream) {
  if (kernel != 0 && kernel != 1) return KDA_ERR_INVALID_ARG;
  kda_status s = check_sizes(T_total, H, N, D, nullptr);
  if (s != KDA_OK) return s;
  if ((s = check_inputs(q, k, v, g_raw, beta_raw, scale, lower_bound, T_total)) != KDA_OK) return s;
  if ((s = check_outputs(out, nullptr, final_state, T_total)) != KDA_OK) return s;
  if (!stamps || max_chunks < 0 || (reinterpret_cast<uintptr_t>(stamps) & 7u) != 0)
    return KDA_ERR_INVALID_ARG;
  DeviceInfo info;
  if ((s = device_info(info)) != KDA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (kernel == 1) {
    e = launch_fused_timed(q, k, v, g_raw, beta_raw, scale, lower_bound, kNormEps, nullptr,
                           T_total, H, N, out, final_state, info.err, stamps, max_chunks, st);
  } else {
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < kda_workspace_size(T_total, H, N, D))
      return KDA_ERR_WORKSPACE;
    e = T_total > 0 ? launch_chunk_prep(q, k, v, g_raw, beta_raw, scale, lower_bound, kNormEps,
                                        nullptr, T_total, H, N, workspace, 0, info.sm_count,
                                        info.err, st)
                    : cudaSuccess;
    if (e == cudaSuccess)
      e = launch_recurrence_timed(workspace, nullptr, nullptr, T_total, H, N, out, final_state,
                                  FwdOpts{0, 0}, info.err, stamps, max_chunks, st);
  }
  return e == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

extern "C" const char* kda_status_string(kda_status status) {
  switch (status) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported size or parameter (D must be 128, lower_bound in [-5, 0])";
    case KDA_ERR_WORKSPACE: return "workspace too small or not allocatable";
    case KDA_ERR_LAUNCH: return "CUDA launch or runtime error";
    case KDA_ERR_TIMEOUT: return "a device-side wait ran out; outputs are invalid";
  }
  return "unknown status";
}
