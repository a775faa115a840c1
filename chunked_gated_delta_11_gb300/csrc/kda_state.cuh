// kda_state.cuh -- the recurrence side of the chunkwise KDA forward pass
// ("You Could Have Come Up with Kimi Delta Attention", sec. 6.3-6.5), shared by
// the head-parallel recurrence kernel (records streamed from HBM) and the fused
// kernel (records built in shared memory by the same CTA).
//
// One CTA owns one (sequence, head) unit.  Its 128 x 128 fp32 state S lives in
// tensor memory, row v in lane v, next to a bf16 snapshot Sb of it.  For each
// chunk record c (layout in kda_common.cuh: W', U', Kend', Aqk' carry the
// per-token key-norm rescaling D that cancels in the products below), with
// S = S_c Diag(dlast_c) already applied and Sb = bf16(S_c):
//
//   MMA1 (tcgen05 kind::f16, bf16, M=128 N=32 K=128, 8 instructions):
//        D1[v][n] = sum_d Sb[v][d] B1[n][d],  B1 = [Qdec ; W']
//        -> D1[v][i] = (Qdec S_c^T)[i][v],  D1[v][16+i] = (W' S_c^T)[i][v]
//   state threads (thread v = row v):
//        e'[v][i] = U'[i][v] - D1[v][16+i]    (corrected errors D E^T, sec. 6.3)
//        E'^T -> tensor memory (fp32; the MMA reads its tf32 part)
//   MMA2 (kind::tf32, M=128 N=144 K=16, 2 instructions), D = [S | D1 cols 0-15]:
//        S[v][d]    += sum_j E'^T[v][j] Kend'[j][d]        (write, sec. 6.4)
//        D1[v][i]   += sum_j E'^T[v][j] Aqk'[i][j]  -> o[i][v] / rq_i (read, sec. 6.5)
//   state threads: o read out and scaled by the record's rq; then, once record c+1 is there,
//        Sb = bf16(S) (= bf16(S_{c+1})),  S *= dlast_{c+1}   (forget, sec. 6.4)
//   while MMA1 of chunk c+1 runs: o -> bf16 -> out.
//
// The tensor core spends tens of cycles per MMA instruction whatever its size
// at these shapes, so the chain uses few, wide instructions: bf16 for MMA1
// (K=16 per instruction, half the count of tf32) and one N=144 tf32 MMA for
// the state update and the output correction together.  Barriers per CTA
// (mbarriers): full[s] (record s ready), empty[s] (record s consumed), mma1 and
// mma2 (MMA completion).  Every wait is bounded; a timeout sets the CTA's abort
// flag and the error word.
#pragma once

#include "kda_common.cuh"

namespace kda {

// tensor-memory columns: S (fp32), D1 = [O | W S^T] (fp32), E^T (tf32), Sb (bf16 pairs)
constexpr uint32_t TM_S = 0, TM_D1 = 128, TM_E = 160, TM_SB = 176, TM_COLS = 256;
static_assert(TM_SB + 64 <= TM_COLS, "tensor-memory map");

template <int NST>
struct StateCtl {
  uint64_t full[NST];
  uint64_t empty[NST];  // record fully consumed (its MMAs are done)
  uint64_t mma1, mma2;
  uint32_t tmem;
  int abort;
};

// Wait for phase `parity` of `bar`; false if the CTA's abort flag is set or if
// `limit` cycles pass first, in which case this thread sets the abort flag and
// the error word (KDA_ERR_TIMEOUT).  The kernels use the default limit
// (about a second); kda_selftest_timeout passes a short one.
template <class Ctl>
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Ctl* ctl, int* err,
                                              long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity, kSleepHintNs)) {
    if (*reinterpret_cast<volatile int*>(&ctl->abort)) return false;
    if (clock64() - t0 > limit) {
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

// Initial state row (fp32, or bf16 if `bf16`; null = zeros) -> tensor memory.
// identity_row >= 0 loads row identity_row of the identity matrix instead.
// State threads only (t < 128).
__device__ __forceinline__ void load_state(uint32_t tb, uint32_t lane_off, const void* src,
                                           bool bf16, int identity_row = -1) {
#pragma unroll
  for (int qd = 0; qd < 4; ++qd) {
    uint32_t r[32];
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (identity_row >= 0) {
        const int d = identity_row - (qd * 32 + i);
        x = make_float4(d == 0 ? 1.f : 0.f, d == 1 ? 1.f : 0.f, d == 2 ? 1.f : 0.f,
                        d == 3 ? 1.f : 0.f);
      } else if (src && bf16) {
        const uint2 b = __ldg(reinterpret_cast<const uint2*>(
            static_cast<const __nv_bfloat16*>(src) + qd * 32 + i));
        const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b.x));
        const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b.y));
        x = make_float4(lo.x, lo.y, hi.x, hi.y);
      } else if (src) {
        x = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(src) + qd * 32 + i));
      }
      r[i] = __float_as_uint(x.x);
      r[i + 1] = __float_as_uint(x.y);
      r[i + 2] = __float_as_uint(x.z);
      r[i + 3] = __float_as_uint(x.w);
    }
    tmem_st32(tb + TM_S + lane_off + qd * 32, r);
  }
  tmem_wait_st();
}

// Snapshot and forget: Sb = bf16(S), then S *= dlast (dlast of the next
// chunk, fp32 [128] in shared memory).  Thread v's row, kCols (32 or 16)
// columns at a time: 16 keeps fewer values live (r, the bf16 pairs and the
// dlast vectors of one piece), for state threads that run under a register
// cap (the fused kernel's setmaxnreg split); 32 needs half the tensor-memory
// round trips, for the recurrence kernel, which has registers to spare.
template <int kCols>
__device__ __forceinline__ void snapshot_and_decay(uint32_t tb, uint32_t lane_off,
                                                   const float* dlast) {
  static_assert(kCols == 16 || kCols == 32, "piece width");
  const float4* dl4 = reinterpret_cast<const float4*>(dlast);
#pragma unroll
  for (int qd = 0; qd < 128 / kCols; ++qd) {
    uint32_t r[kCols], b[kCols / 2];
    if constexpr (kCols == 32)
      tmem_ld32(tb + TM_S + lane_off + qd * 32, r);
    else
      tmem_ld16(tb + TM_S + lane_off + qd * 16, r);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < kCols / 2; ++i)
      b[i] = pack_bf16(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
    if constexpr (kCols == 32)
      tmem_st16(tb + TM_SB + lane_off + qd * 16, b);
    else
      tmem_st8(tb + TM_SB + lane_off + qd * 8, b);
#pragma unroll
    for (int i4 = 0; i4 < kCols / 4; ++i4) {
      const float4 dv = dl4[qd * (kCols / 4) + i4];
      const float2 a = __fmul2_rn(make_float2(__uint_as_float(r[4 * i4]), __uint_as_float(r[4 * i4 + 1])),
                                  make_float2(dv.x, dv.y));
      const float2 c = __fmul2_rn(make_float2(__uint_as_float(r[4 * i4 + 2]), __uint_as_float(r[4 * i4 + 3])),
                                  make_float2(dv.z, dv.w));
      r[4 * i4 + 0] = __float_as_uint(a.x);
      r[4 * i4 + 1] = __float_as_uint(a.y);
      r[4 * i4 + 2] = __float_as_uint(c.x);
      r[4 * i4 + 3] = __float_as_uint(c.y);
    }
    if constexpr (kCols == 32)
      tmem_st32(tb + TM_S + lane_off + qd * 32, r);
    else
      tmem_st16(tb + TM_S + lane_off + qd * 16, r);
  }
  tmem_wait_st();
}

// MMA1 on the record at shared address sb: 8 bf16 K=16 steps into D1.
// Issuing thread only.  The K steps of one 64-channel block are 32 bytes
// apart and the two blocks 4096 bytes, which moves only the descriptor's
// start-address field (bits 0-13, in 16-byte units).
__device__ __forceinline__ void issue_mma1(uint32_t sb, uint32_t tb, uint64_t* bar) {
  const uint32_t id1 = make_idesc(1, 128, 32);
  const uint64_t bd0 = make_sdesc(sb + OFF_B1, 16, 1024, 2);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_bf16_ts(tb + TM_D1, tb + TM_SB + kk * 8, bd0 + static_cast<uint64_t>((kk >> 2) * 256 + (kk & 3) * 2),
                id1, kk > 0 ? 1u : 0u);
  tc_commit(bar);
}

// MMA2: [S | O] += E^T [Kend ; Aqk]^T, two tf32 K=8 steps with N = 144.
// Issuing thread only.
__device__ __forceinline__ void issue_mma2(uint32_t sb, uint32_t tb, uint64_t* bar) {
  const uint32_t id2 = make_idesc(2, 128, 144);
#pragma unroll
  for (int kk = 0; kk < 2; ++kk)
    mma_tf32_ts(tb + TM_S, tb + TM_E + kk * 8, make_sdesc(sb + OFF_KA + kk * KA_TILE, 16, 256, 6),
                id2, 1u);
  tc_commit(bar);
}

// The state threads' work for all chunks, then the final state.  Thread v = 0
// also issues every MMA.  `ring` is the 1024-aligned record ring (stage stride
// REC_STRIDE_SMEM).  On thread 0, `stage_free(c, s)` runs once all MMAs of
// record c are done and every state thread has finished reading it.
// `final_dst` is thread v's row of the final state (fp32, or bf16 if
// `state_bf16`; null = not written).
// `ostage` is 4 KB of shared memory (1 KB per state warp) that turns each
// warp's 16 x 32 output tile into 16-byte stores, followed by 256 B (64 B per
// state warp) that hold the chunk's rq between the U' read and the output.  u_zero: the records carry
// no U' (v is zero), which is taken as zero.
//
// kTimed (a diagnostic instantiation, kda_profile_phases): thread 0 writes
// clock64() at the phase boundaries of chunk c to stamps[8 c + k] for
// c < max_chunks (stamps null = not recorded):
//   k = 0 MMA1 issued, 1 MMA1 complete, 2 E'^T written (MMA2 issued),
//   3 MMA2 complete, 4 next record there, 5 snapshot and decay done (MMA1 of
//   chunk c + 1 issued), 6 outputs stored.
// kSnapCols: the column width of the snapshot pass (snapshot_and_decay).
// on_record(j, w) runs on lane 0 of state warps w = 1, 2, 3 once record j is
// there (after full[j % NST] passed; for j > 0 at the end of chunk j - 1):
// the record's producer is done with every input of chunk j, so a caller may
// reuse that chunk's input buffers.
template <int NST, int kSnapCols, bool kTimed = false, class StageFree, class OnRecord>
__device__ __forceinline__ void state_rows(StateCtl<NST>* ctl, uint8_t* ring, int nchunks,
                                           uint32_t tb, uint32_t lane_off, int v, int64_t bos,
                                           int64_t eos, int H, int h,
                                           __nv_bfloat16* __restrict__ out, void* final_dst,
                                           bool state_bf16, int* err, uint8_t* ostage,
                                           StageFree&& stage_free, OnRecord&& on_record,
                                           bool u_zero = false, long long* stamps = nullptr,
                                           int max_chunks = 0) {
  auto stamp = [&](int c, int k) {
    if constexpr (kTimed) {
      if (v == 0 && stamps && c < max_chunks) stamps[8 * c + k] = clock64();
    }
  };
  float* rqstage = reinterpret_cast<float*>(ostage + 4096) + (v >> 5) * 16;
  bool ok = true;
  int n1 = 0, n2 = 0;  // MMA1 / MMA2 commits issued (thread 0)
  // chunk 0: snapshot the initial state and apply chunk 0's decay
  if (nchunks > 0) {
    ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->full[0], 0, ctl, err));
    if (ok && v >= 32 && (v & 31) == 0) on_record(0, v >> 5);
    if (ok) {
      snapshot_and_decay<kSnapCols>(tb, lane_off, reinterpret_cast<const float*>(ring + OFF_DL));
      tc_fence_before();
    }
    ok = state_all(ok);
    if (ok && v == 0) {
      tc_fence_after();
      issue_mma1(smem_u32(ring), tb, &ctl->mma1);
      ++n1;
    }
    stamp(0, 0);
  }
  for (int c = 0; c < nchunks && ok; ++c) {
    const int s = c % NST;
    const uint8_t* st = ring + s * REC_STRIDE_SMEM;
    ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->mma1, c & 1, ctl, err));
    stamp(c, 1);
    if (ok) {
      // corrected errors e[v][i] = U[i][v] - (W S^T)[i][v] -> tensor memory
      tc_fence_after();
      uint32_t d1[16];
      tmem_ld16(tb + TM_D1 + 16 + lane_off, d1);
      tmem_wait_ld();
      const float4* U4 = reinterpret_cast<const float4*>(st + OFF_U + v * 64);
      const int usw = u_piece_swz(v);  // piece order of row v (u_offset)
      uint32_t pk[16];
      // (the tensor core reads the tf32 part of these fp32 values)
      const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
      for (int i4 = 0; i4 < 4; ++i4) {
        const float4 u = u_zero ? make_float4(0.f, 0.f, 0.f, 0.f) : U4[i4 ^ usw];
        const float2 e0 = __ffma2_rn(make_float2(__uint_as_float(d1[i4 * 4]), __uint_as_float(d1[i4 * 4 + 1])),
                                     m1, make_float2(u.x, u.y));
        const float2 e1 = __ffma2_rn(make_float2(__uint_as_float(d1[i4 * 4 + 2]), __uint_as_float(d1[i4 * 4 + 3])),
                                     m1, make_float2(u.z, u.w));
        pk[i4 * 4 + 0] = __float_as_uint(e0.x);
        pk[i4 * 4 + 1] = __float_as_uint(e0.y);
        pk[i4 * 4 + 2] = __float_as_uint(e1.x);
        pk[i4 * 4 + 3] = __float_as_uint(e1.y);
      }
      tmem_st16(tb + TM_E + lane_off, pk);
      // the query factors the record's Qdec and Aqk' leave out: copied with U'
      // to this warp's slot, since the stage may be released once MMA2 is done
      if ((v & 31) < 4)
        reinterpret_cast<float4*>(rqstage)[v & 3] = reinterpret_cast<const float4*>(st + OFF_RQ)[v & 3];
      tmem_wait_st();
      tc_fence_before();
    }
    // every state thread has written E^T and finished reading U' and rq
    if (!state_all(ok)) { ok = false; break; }
    if (v == 0) {
      tc_fence_after();
      issue_mma2(smem_u32(st), tb, &ctl->mma2);
      ++n2;
    }
    stamp(c, 2);
    ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->mma2, c & 1, ctl, err));
    stamp(c, 3);
    uint32_t o[16];
    if (ok) {
      tc_fence_after();
      tmem_ld16(tb + TM_D1 + lane_off, o);
      tmem_wait_ld();
      const float4* rq4 = reinterpret_cast<const float4*>(rqstage);
#pragma unroll
      for (int i4 = 0; i4 < 4; ++i4) {
        const float4 r = rq4[i4];
        o[4 * i4 + 0] = __float_as_uint(__uint_as_float(o[4 * i4 + 0]) * r.x);
        o[4 * i4 + 1] = __float_as_uint(__uint_as_float(o[4 * i4 + 1]) * r.y);
        o[4 * i4 + 2] = __float_as_uint(__uint_as_float(o[4 * i4 + 2]) * r.z);
        o[4 * i4 + 3] = __float_as_uint(__uint_as_float(o[4 * i4 + 3]) * r.w);
      }
    }
    if (ok && v == 0) stage_free(c, s);
    if (c + 1 < nchunks) {
      // snapshot S_{c+1} for MMA1 of chunk c+1 and apply that chunk's decay
      const int s1 = (c + 1) % NST;
      if (ok) ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->full[s1], ((c + 1) / NST) & 1, ctl, err));
      stamp(c, 4);
      if (ok) {
        snapshot_and_decay<kSnapCols>(
            tb, lane_off, reinterpret_cast<const float*>(ring + s1 * REC_STRIDE_SMEM + OFF_DL));
        tc_fence_before();
      }
      // also: every thread has read this chunk's outputs out of D1
      ok = state_all(ok);
      if (ok && v == 0) {
        tc_fence_after();
        issue_mma1(smem_u32(ring + s1 * REC_STRIDE_SMEM), tb, &ctl->mma1);
        ++n1;
      }
      stamp(c, 5);
      stamp(c + 1, 0);
    }
    if (ok) {
      // warp tile [16 tokens][32 channels] bf16 through shared memory, then
      // 16-byte stores (each row of the tile is 64 contiguous bytes of `out`)
      const int64_t t0 = bos + static_cast<int64_t>(c) * kChunk;
      const int nc = static_cast<int>((eos - t0) < kChunk ? (eos - t0) : kChunk);
      const int w = v >> 5, l = v & 31;
      uint8_t* ost = ostage + w * 1024;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        *reinterpret_cast<__nv_bfloat16*>(ost + i * 64 + l * 2) =
            __float2bfloat16_rn(__uint_as_float(o[i]));
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
    stamp(c, 6);
    // record c + 1 was there before the snapshot above (called here, where
    // the outputs no longer hold registers)
    if (ok && c + 1 < nchunks && v >= 32 && (v & 31) == 0) on_record(c + 1, v >> 5);
  }
  ok = state_all(ok && !*reinterpret_cast<volatile int*>(&ctl->abort));
  if (!ok && v == 0) {
    // let MMAs still in flight finish before the CTA frees its tensor memory
    if (n1 > 0) mbar_wait(&ctl->mma1, (n1 - 1) & 1);
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
      for (int i = 0; i < 32; i += 4) {
        if (state_bf16)
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(final_dst) + qd * 32 + i) =
              make_uint2(pack_bf16(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                         pack_bf16(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3])));
        else
          *reinterpret_cast<float4*>(static_cast<float*>(final_dst) + qd * 32 + i) =
              make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]),
                          __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
      }
    }
  }
}

}  // namespace kda
