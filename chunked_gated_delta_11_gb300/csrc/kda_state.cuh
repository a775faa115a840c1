// kda_state.cuh -- the recurrence side of the chunkwise KDA forward pass
// ("You Could Have Come Up with Kimi Delta Attention", sec. 6.3-6.5), shared by
// the head-parallel recurrence kernel (records streamed from HBM) and the fused
// kernel (records built in shared memory by the same CTA).
//
// One CTA owns one (sequence, head) unit.  Its 128 x 128 fp32 state S lives in
// tensor memory, row v in lane v.  For each chunk record c (kda_common.cuh):
//
//   MMA1 (tcgen05 kind::tf32, M=128 N=32 K=128, issued by one thread):
//        D1[v][n] = sum_d S[v][d] B1[n][d],  B1 = [W ; Qdec]
//        -> D1[v][i] = (W S^T)[i][v],  D1[v][16+i] = (Qdec S^T)[i][v]
//   state threads (thread v = row v):
//        S[v][:] *= dlast                                  (forget, sec. 6.4)
//        e[v][i] = U[i][v] - D1[v][i]                       (corrected errors)
//        E^T -> tensor memory (fp32 rounded to tf32)
//   MMA2 (tcgen05 kind::tf32, M=128 N=128 K=16, two instructions):
//        S += E^T Kend                                      (write, sec. 6.4)
//   MMA3 (kind::tf32, M=128 N=16 K=16, two instructions):
//        D1[v][16+i] += sum_j E^T[v][j] Aqk[i][j]  -> o[i][v]     (read, sec. 6.5)
//   state threads: o -> bf16 -> out.
//
// MMA1 takes the fp32 state as its A operand directly (the tensor core reads its
// tf32 part), so no operand copy of S is kept.  D1 alternates between two
// tensor-memory buffers so that chunk c's outputs can be read while MMA1 of
// chunk c+1 writes the other one.  Barriers per CTA (mbarriers): full[s]
// (record s ready), empty[s] (record s consumed: 128 state threads + one MMA
// commit), mma1/mma2 (MMA completion), eready (128 state threads wrote E^T).
// Every wait is bounded; a timeout sets the CTA's abort flag and the error word.
#pragma once

#include "kda_common.cuh"

namespace kda {

constexpr uint32_t TM_S = 0, TM_D1 = 128, TM_E = 192, TM_COLS = 256;
// D1 of chunk c: columns TM_D1 + 32 * (c & 1) .. + 31
__device__ __forceinline__ uint32_t d1_col(int c) { return TM_D1 + 32u * static_cast<uint32_t>(c & 1); }

template <int NST>
struct StateCtl {
  uint64_t full[NST];
  uint64_t empty[NST];  // record fully consumed (its MMAs are done)
  uint64_t mma1, mma1b, mma2;  // MMA1 k-steps over channels 0-63, then 64-127; MMA2/3
  uint32_t tmem;
  int abort;
};

template <class Ctl>
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Ctl* ctl, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity, kSleepHintNs)) {
    if (*reinterpret_cast<volatile int*>(&ctl->abort)) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      *reinterpret_cast<volatile int*>(&ctl->abort) = 1;
      atomicExch(err, 5);
      return false;
    }
  }
  return true;
}

// AND of `pred` over the 128 state threads (named barrier 2).  Every decision
// to stop goes through it, so no state thread is ever left at a barrier.
__device__ __forceinline__ bool state_all(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, 2, 128, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred))
      : "memory");
  return r != 0;
}

// descriptor of a K=8 tf32 tile with the 32-byte swizzle (rows of 32 bytes)
__device__ __forceinline__ uint64_t sw32_desc(uint32_t saddr) { return make_sdesc(saddr, 16, 256, 6); }

// Initial state (or zeros) -> tensor memory.  State threads only (t < 128).
__device__ __forceinline__ void load_state(uint32_t tb, uint32_t lane_off,
                                           const float* __restrict__ src) {
#pragma unroll
  for (int qd = 0; qd < 4; ++qd) {
    uint32_t r[32];
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      const float4 x = src ? __ldg(reinterpret_cast<const float4*>(src + qd * 32 + i))
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

// MMA1 of chunk c (16 tf32 steps into D1 of that chunk) on the record at
// shared address sb, committed in two halves: `bar_a` completes once the steps
// over key channels 0-63 are done (those state columns may then be rewritten),
// `bar_b` once all are.  Issuing thread only.
__device__ __forceinline__ void issue_mma1(int c, uint32_t sb, uint32_t tb, uint64_t* bar_a,
                                           uint64_t* bar_b) {
  const uint32_t id1 = make_idesc(2, 128, 32);
  const uint32_t d1 = tb + d1_col(c);
#pragma unroll
  for (int kk = 0; kk < 16; ++kk) {
    const uint64_t bd = make_sdesc(sb + OFF_B1 + (kk >> 2) * 4096 + (kk & 3) * 32, 16, 1024, 2);
    mma_tf32_ts(d1, tb + TM_S + kk * 8, bd, id1, kk > 0 ? 1u : 0u);
    if (kk == 7) tc_commit(bar_a);
  }
  tc_commit(bar_b);
}

// MMA2 (state update) and MMA3 (output correction) of chunk c, two K=8 tf32
// steps each.  Issuing thread only.
__device__ __forceinline__ void issue_mma23(int c, uint32_t sb, uint32_t tb, uint64_t* bar) {
  const uint32_t id2 = make_idesc(2, 128, 128), id3 = make_idesc(2, 128, 16);
  const uint32_t d1 = tb + d1_col(c);
#pragma unroll
  for (int kk = 0; kk < 2; ++kk)
    mma_tf32_ts(tb + TM_S, tb + TM_E + kk * 8, sw32_desc(sb + OFF_KEND + kk * 4096), id2, 1u);
#pragma unroll
  for (int kk = 0; kk < 2; ++kk)
    mma_tf32_ts(d1 + 16, tb + TM_E + kk * 8, sw32_desc(sb + OFF_AQK + kk * 512), id3, 1u);
  tc_commit(bar);
}

// The state threads' work for all chunks, then the final state.  Thread v = 0
// also issues every MMA.  `ring` is the 1024-aligned record ring (stage stride
// REC_STRIDE_SMEM).  On thread 0, `stage_free(c, s)` runs once all MMAs of
// record c are done and every state thread has finished reading it.
// `ostage` is 4 KB of shared memory (1 KB per state warp) that turns each
// warp's 16 x 32 output tile into 16-byte stores.
template <int NST, class StageFree>
__device__ __forceinline__ void state_rows(StateCtl<NST>* ctl, uint8_t* ring, int nchunks,
                                           uint32_t tb, uint32_t lane_off, int v, int64_t bos,
                                           int64_t eos, int H, int h,
                                           __nv_bfloat16* __restrict__ out,
                                           float* __restrict__ final_dst, int* err,
                                           uint8_t* ostage, StageFree&& stage_free) {
  bool ok = true;
  int n1 = 0, n2 = 0;  // MMA1 / MMA2 commits issued (thread 0)
  if (v == 0 && nchunks > 0) {
    ok = wait_or_abort(&ctl->full[0], 0, ctl, err);
    if (ok) {
      tc_fence_after();
      issue_mma1(0, smem_u32(ring), tb, &ctl->mma1, &ctl->mma1b);
      ++n1;
    }
  }
  for (int c = 0; c < nchunks; ++c) {
    const int s = c % NST;
    const uint8_t* st = ring + s * REC_STRIDE_SMEM;
    if (ok) ok = wait_or_abort(&ctl->full[s], (c / NST) & 1, ctl, err);
    if (ok) ok = wait_or_abort(&ctl->mma1, c & 1, ctl, err);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      // forget: S[v][:] *= dlast, 32 columns at a time; columns 0-63 while MMA1
      // still reads columns 64-127, the rest once MMA1 is done
      const float4* dl4 = reinterpret_cast<const float4*>(st + OFF_DL);
#pragma unroll
      for (int qd = 0; qd < 4; ++qd) {
        if (qd == 2) {
          ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->mma1b, c & 1, ctl, err));
          if (!ok) break;
          tc_fence_after();
        }
        uint32_t r[32];
        tmem_ld32(tb + TM_S + lane_off + qd * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int i4 = 0; i4 < 8; ++i4) {
          const float4 dv = dl4[qd * 8 + i4];
          r[4 * i4 + 0] = __float_as_uint(__uint_as_float(r[4 * i4 + 0]) * dv.x);
          r[4 * i4 + 1] = __float_as_uint(__uint_as_float(r[4 * i4 + 1]) * dv.y);
          r[4 * i4 + 2] = __float_as_uint(__uint_as_float(r[4 * i4 + 2]) * dv.z);
          r[4 * i4 + 3] = __float_as_uint(__uint_as_float(r[4 * i4 + 3]) * dv.w);
        }
        tmem_st32(tb + TM_S + lane_off + qd * 32, r);
      }
      if (ok) {
        uint32_t d1[16];
        tmem_ld16(tb + d1_col(c) + lane_off, d1);
        tmem_wait_ld();
        // corrected errors e[v][i] = U[i][v] - (W S^T)[i][v] -> tensor memory
        const float4* U4 = reinterpret_cast<const float4*>(st + OFF_U + v * 64);
        uint32_t pk[16];
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) {
          const float4 u = U4[i4];
          pk[i4 * 4 + 0] = tf32_bits(u.x - __uint_as_float(d1[i4 * 4 + 0]));
          pk[i4 * 4 + 1] = tf32_bits(u.y - __uint_as_float(d1[i4 * 4 + 1]));
          pk[i4 * 4 + 2] = tf32_bits(u.z - __uint_as_float(d1[i4 * 4 + 2]));
          pk[i4 * 4 + 3] = tf32_bits(u.w - __uint_as_float(d1[i4 * 4 + 3]));
        }
        tmem_st16(tb + TM_E + lane_off, pk);
        tmem_wait_st();
        tc_fence_before();
      }
    }
    // every state thread has written E^T and finished reading U and dlast
    if (!state_all(ok)) { ok = false; break; }
    if (v == 0) {
      tc_fence_after();
      issue_mma23(c, smem_u32(st), tb, &ctl->mma2);
      ++n2;
    }
    ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->mma2, c & 1, ctl, err));
    // outputs: D1[v][16 + i] = o[i][v], read while the tensor pipe is idle
    // (MMA1 of chunk c+1 writes the other D1 buffer)
    uint32_t o[16];
    if (ok) {
      tc_fence_after();
      tmem_ld16(tb + d1_col(c) + 16 + lane_off, o);
      tmem_wait_ld();
    }
    if (v == 0 && ok) {
      stage_free(c, s);
      if (c + 1 < nchunks) {
        const int s1 = (c + 1) % NST;
        ok = wait_or_abort(&ctl->full[s1], ((c + 1) / NST) & 1, ctl, err);
        if (ok) {
          tc_fence_after();
          issue_mma1(c + 1, smem_u32(ring + s1 * REC_STRIDE_SMEM), tb, &ctl->mma1, &ctl->mma1b);
          ++n1;
        }
      }
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      // warp tile [16 tokens][32 channels] bf16 through shared memory, then
      // 16-byte stores (each row of the tile is 64 contiguous bytes of `out`)
      const int64_t t0 = bos + static_cast<int64_t>(c) * kChunk;
      const int nc = static_cast<int>((eos - t0) < kChunk ? (eos - t0) : kChunk);
      const int w = v >> 5, l = v & 31;
      uint8_t* ost = ostage + w * 1024;
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        // tokens i, i+1 of channel v: two bf16 in one 4-byte store would
        // stride rows, so keep one bf16 per store (conflict-free, 64 B rows)
        *reinterpret_cast<__nv_bfloat16*>(ost + i * 64 + l * 2) =
            __float2bfloat16_rn(__uint_as_float(o[i]));
        *reinterpret_cast<__nv_bfloat16*>(ost + (i + 1) * 64 + l * 2) =
            __float2bfloat16_rn(__uint_as_float(o[i + 1]));
      }
      __syncwarp();
#pragma unroll
      for (int rep = 0; rep < 2; ++rep) {
        const int p = l + 32 * rep, i = p >> 2, sub = p & 3;
        if (i < nc)
          *reinterpret_cast<uint4*>(out + ((t0 + i) * H + h) * kDim + w * 32 + sub * 8) =
              *reinterpret_cast<const uint4*>(ost + i * 64 + sub * 16);
      }
      __syncwarp();
    }
  }
  ok = __all_sync(0xffffffffu, ok && !*reinterpret_cast<volatile int*>(&ctl->abort));
  if (!ok && v == 0) {
    // let MMAs still in flight finish before the CTA frees its tensor memory
    if (n1 > 0) mbar_wait(&ctl->mma1b, (n1 - 1) & 1);
    if (n2 > 0) mbar_wait(&ctl->mma2, (n2 - 1) & 1);
  }
  tc_fence_after();
  if (ok && final_dst) {
#pragma unroll
    for (int qd = 0; qd < 4; ++qd) {
      uint32_t r[32];
      tmem_ld32(tb + TM_S + lane_off + qd * 32, r);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(final_dst + qd * 32 + i) =
            make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]),
                        __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
    }
  }
}

}  // namespace kda
