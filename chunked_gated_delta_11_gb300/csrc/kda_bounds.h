// kda_bounds.h -- sequence bounds from a cu_seqlens pair, clamped so that a
// malformed cu_seqlens (not starting at 0, decreasing, or ending past T_total)
// can only give wrong results, never a read or write outside the tensors.
// Plain C++ so that the host tests compile it too; the kernels include it
// through kda_common.cuh.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define KDA_HD __host__ __device__ __forceinline__
#else
#define KDA_HD inline
#endif

namespace kda {

// Tokens [bos, eos) of a sequence whose cu_seqlens entries are lo and hi:
// 0 <= bos <= eos <= T_total always holds.  For a well-formed cu_seqlens
// (0 <= lo <= hi <= T_total) these are lo and hi themselves.
KDA_HD void clamp_seq_bounds(int64_t lo, int64_t hi, int64_t T_total, int64_t& bos,
                             int64_t& eos) {
  bos = lo < 0 ? 0 : (lo > T_total ? T_total : lo);
  eos = hi < bos ? bos : (hi > T_total ? T_total : hi);
}

}  // namespace kda
