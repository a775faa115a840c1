// kda_cp.cu -- the per-rank steps of a context-parallel split of one long
// sequence: each rank holds one contiguous piece of the tokens.
//
// Each token step is an affine map of the state, S -> S A_t + beta_t v_t k_t^T
// with A_t = Diag(alpha_t) (I - beta_t k_t k_t^T) ("You Could Have Come Up with
// Kimi Delta Attention", sec. 4.1), so piece r maps its starting state S_0 to
// S_0 M_r + X_r, and inside it o_t = o^X_t + S_0 y_t with y_t = M_t (s q^_t).
// The steps of one rank:
//   kda_piece_forward  X_r and o^X (from zero; the first piece from the
//                      sequence's initial state), and M_r and y (the same
//                      piece with v = 0 from the identity): one launch of the
//                      fused kernel's segment mode over a two-segment plan
//                      [0, 0, T] whose second segment is the piece;
//   (exchange)         the (M_r, X_r) pairs of all ranks, 2 x H x 64 KiB each,
//                      gathered in rank order by the caller (NCCL or gloo);
//   kda_pieces_scan    S_0 of every piece and the final state, S <- S M + X in
//                      fp32 (the segmented pass's scan kernel);
//   kda_piece_fixup    o_t += S_0 y_t over the piece (its fix-up kernel).
// The same kernels as kda_fwd_segmented, which runs all pieces on one GPU.
#include <cstdint>

#include "kda.h"
#include "kda_common.cuh"

namespace kda {

cudaError_t launch_fused(const void* q, const void* k, const void* v, const void* g,
                         const void* beta_raw, float scale, float lower_bound, float eps,
                         const void* init, const int32_t* cu, int64_t T_total, int H, int N,
                         void* out, void* final_state, FwdOpts opts, SegArgs seg, int* err,
                         cudaStream_t stream);
// s0_bf16 / sstart16 (optional): a bf16 copy of every later segment's S_0,
// written by the scan and read by the fix-up instead of converting S_0
cudaError_t launch_affine_scan(float* xs, const float* ms, int N, int P, int H,
                               void* final_state, bool final_bf16, int sm_count,
                               cudaStream_t stream, void* s0_bf16);
cudaError_t launch_seg_fixup(const int32_t* cu_seg, const int32_t* blk, int Nseg, int H,
                             const float* sstart, const void* y, void* out, int sm_count,
                             cudaStream_t stream, const void* sstart16);

namespace {

constexpr float kEps = 1e-6f;
constexpr int kFixupBlock = 64;  // tokens per fix-up work item (the kernel's SG_BLOCK)

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Dev {
  int sm_count = 0;
  int* err = nullptr;
};

// SM count and the device error word (kda_device_status reads the same word;
// the symbol lives in kda_api.cu).
kda_status dev_info(Dev& d) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_LAUNCH;
  if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return KDA_ERR_LAUNCH;
  return KDA_OK;
}

int64_t r256(int64_t x) { return (x + 255) & ~static_cast<int64_t>(255); }

// workspace: the plan ints (256 B), then two [2, H, 128, 128] fp32 state pairs
int64_t states_bytes(int32_t H) { return 2 * static_cast<int64_t>(H) * kDim * kDim * 4; }

}  // namespace

extern kda_status error_word(int** out);

}  // namespace kda

using namespace kda;

extern "C" size_t kda_piece_workspace_size(int64_t T_local, int32_t H) {
  if (T_local < 0 || H <= 0 || T_local >= (static_cast<int64_t>(1) << 31)) return 0;
  return static_cast<size_t>(256 + 2 * r256(states_bytes(H)));
}

extern "C" kda_status kda_piece_forward(const void* q, const void* k, const void* v,
                                        const void* g_raw, const void* beta_raw, float scale,
                                        float lower_bound, const float* initial_state,
                                        int64_t T_local, int32_t H, int32_t D, void* out,
                                        float* x_state, float* m_state, void* y, int32_t gate,
                                        void* workspace, size_t workspace_bytes, void* stream) {
  if (gate != KDA_GATE_PER_CHANNEL && gate != KDA_GATE_PER_HEAD) return KDA_ERR_INVALID_ARG;
  if (!x_state || !a16(x_state)) return KDA_ERR_INVALID_ARG;
  if (!m_state) {
    // the first piece: the plain pass from the sequence's initial state
    const kda_options o{KDA_SCHEDULE_FUSED, KDA_STATE_F32, gate};
    return kda_forward(&o, q, k, v, g_raw, beta_raw, scale, lower_bound, initial_state, nullptr,
                       T_local, H, 1, D, out, x_state, nullptr, 0, stream);
  }
  // an empty piece (T_local = 0) has X = 0 and M = I and needs no y
  if (initial_state || !a16(m_state) || (T_local > 0 && (!y || !a16(y)))) return KDA_ERR_INVALID_ARG;
  if (D != KDA_HEAD_DIM) return KDA_ERR_UNSUPPORTED;
  if (!(lower_bound >= -5.0f && lower_bound <= 0.0f)) return KDA_ERR_UNSUPPORTED;
  if (T_local < 0 || H <= 0 || T_local >= (static_cast<int64_t>(1) << 31)) return KDA_ERR_INVALID_ARG;
  if (T_local > 0 && (!q || !k || !v || !g_raw || !beta_raw || !out || !a16(q) || !a16(k) ||
                      !a16(v) || !a16(out) || (gate == KDA_GATE_PER_CHANNEL && !a16(g_raw))))
    return KDA_ERR_INVALID_ARG;
  const size_t need = kda_piece_workspace_size(T_local, H);
  if (!workspace || !a16(workspace) || workspace_bytes < need) return KDA_ERR_WORKSPACE;
  Dev d;
  kda_status s = dev_info(d);
  if (s != KDA_OK) return s;
  if ((s = error_word(&d.err)) != KDA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* wb = static_cast<uint8_t*>(workspace);
  int32_t* plan = reinterpret_cast<int32_t*>(wb);
  float* xs2 = reinterpret_cast<float*>(wb + 256);
  float* ms2 = reinterpret_cast<float*>(wb + 256 + r256(states_bytes(H)));
  // two segments of one sequence: [0, 0) and [0, T_local); the second is the
  // piece, run from zero (X role) and from the identity with v = 0 (M role)
  const int32_t cu_seg[3] = {0, 0, static_cast<int32_t>(T_local)};
  cudaError_t e = cudaMemcpyAsync(plan, cu_seg, sizeof(cu_seg), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = launch_fused(q, k, v, g_raw, beta_raw, scale, lower_bound, kEps, nullptr, plan, T_local,
                     H, 2, out, xs2, FwdOpts{0, gate == KDA_GATE_PER_HEAD},
                     SegArgs{2, static_cast<__nv_bfloat16*>(y), ms2}, d.err, st);
  const size_t one = static_cast<size_t>(states_bytes(H)) / 2;  // H states: segment 1's
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(x_state, reinterpret_cast<uint8_t*>(xs2) + one, one,
                        cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(m_state, reinterpret_cast<uint8_t*>(ms2) + one, one,
                        cudaMemcpyDeviceToDevice, st);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

extern "C" kda_status kda_pieces_scan(float* xs, const float* ms, int32_t P, int32_t H,
                                      int32_t D, float* final_state, void* stream) {
  if (D != KDA_HEAD_DIM) return KDA_ERR_UNSUPPORTED;
  if (P <= 0 || H <= 0 || !xs || !ms || !a16(xs) || !a16(ms) ||
      (final_state && !a16(final_state)) || static_cast<int64_t>(P) * H > 0x7fffffffLL)
    return KDA_ERR_INVALID_ARG;
  Dev d;
  kda_status s = dev_info(d);
  if (s != KDA_OK) return s;
  return launch_affine_scan(xs, ms, 1, P, H, final_state, false, d.sm_count,
                            static_cast<cudaStream_t>(stream), nullptr) == cudaSuccess
             ? KDA_OK
             : KDA_ERR_LAUNCH;
}

extern "C" kda_status kda_piece_fixup(void* out, const void* y, const float* s0, int64_t T_local,
                                      int32_t H, int32_t D, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  if (D != KDA_HEAD_DIM) return KDA_ERR_UNSUPPORTED;
  if (T_local < 0 || H <= 0 || T_local >= (static_cast<int64_t>(1) << 31)) return KDA_ERR_INVALID_ARG;
  if (T_local == 0) return KDA_OK;
  if (!out || !y || !s0 || !a16(out) || !a16(y) || !a16(s0)) return KDA_ERR_INVALID_ARG;
  if (!workspace || !a16(workspace) || workspace_bytes < 256) return KDA_ERR_WORKSPACE;
  Dev d;
  kda_status s = dev_info(d);
  if (s != KDA_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // one segment covering the piece: cu [0, T], work items [0, blocks)
  const int32_t plan[4] = {0, static_cast<int32_t>(T_local), 0,
                           static_cast<int32_t>((T_local + kFixupBlock - 1) / kFixupBlock)};
  int32_t* dp = static_cast<int32_t*>(workspace);
  cudaError_t e = cudaMemcpyAsync(dp, plan, sizeof(plan), cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess)
    e = launch_seg_fixup(dp, dp + 2, 1, H, s0, y, out, d.sm_count, st, nullptr);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}
