// kda_noalloc.cu -- kda_fwd_noalloc: the forward pass with its chunk-record
// workspace in a fixed device array that belongs to the library, so the call
// itself allocates nothing.
//
// Who needs it: callers that cannot call cudaMalloc (or any allocator) at
// all, for example a plugin inside a host engine that owns every byte of
// device memory and gives its plugins no allocator, or code on a path where
// an allocation that may fail or wait is not acceptable.  kda_fwd needs a
// workspace either from the caller or from cudaMallocAsync; this entry point
// takes it from g_noalloc_ws instead.
//
// Cost of the array: KDA_NOALLOC_WORKSPACE_BYTES (64 MiB) of device memory on
// each GPU that uses it, from the first kda_fwd_noalloc call on that device
// (or from library load, under eager module loading) until the process
// exits.  Under CUDA's default lazy module loading the module that holds the
// array is loaded, and the memory taken, when the first call looks up its
// address.
#include <mutex>

#include "kda.h"
#include "kda_common.cuh"

namespace kda {
namespace {

// The shared scratch: one chunk record per (chunk slot, head), written by the
// chunk kernel and read by the recurrence kernel of the same call.  Nothing in
// it has to start at zero: the chunk kernel writes every byte of every record
// that the recurrence kernel then reads.
static __device__ __align__(256) uint8_t g_noalloc_ws[KDA_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ws_ptr[kMaxDevices] = {};

// Device address of g_noalloc_ws on the current device.  In host code the name
// g_noalloc_ws is only a host-side stand-in for the symbol, so the address is
// looked up once per device, with that device current, and cached.
kda_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_LAUNCH;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_ws_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_ws) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return KDA_ERR_LAUNCH;
    }
    g_ws_ptr[dev] = p;
  }
  *out = g_ws_ptr[dev];
  return KDA_OK;
}

}  // namespace
}  // namespace kda

extern "C" kda_status kda_fwd_noalloc(const void* q, const void* k, const void* v,
                                      const void* g_raw, const void* beta_raw, float scale,
                                      float lower_bound, const float* initial_state,
                                      const int32_t* cu_seqlens, int64_t T_total, int32_t H,
                                      int32_t N, int32_t D, void* out, float* final_state,
                                      void* stream) {
  const size_t need = kda_workspace_size(T_total, H, N, D);
  if (need > static_cast<size_t>(KDA_NOALLOC_WORKSPACE_BYTES)) return KDA_ERR_WORKSPACE;
  void* ws = nullptr;
  const kda_status s = kda::scratch_address(&ws);
  if (s != KDA_OK) return s;
  // kda_fwd validates every argument and, given a workspace, allocates nothing
  return kda_fwd(q, k, v, g_raw, beta_raw, scale, lower_bound, initial_state, cu_seqlens,
                 T_total, H, N, D, out, final_state, ws, KDA_NOALLOC_WORKSPACE_BYTES, stream);
}
