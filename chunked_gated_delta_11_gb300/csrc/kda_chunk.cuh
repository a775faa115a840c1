// kda_chunk.cuh -- the per-chunk work of the chunkwise KDA forward pass
// ("You Could Have Come Up with Kimi Delta Attention", sec. 6.1-6.6; gates and
// norms as in "FlashKDA Delta Attention Algorithm", Core Architecture), done
// by one group of 128 threads for one (chunk, head) and written as one record
// (layout in kda_common.cuh).  Used by the chunk kernel (K1) and by the chunk
// warps of the fused kernel.
//
// Steps, for the n_c <= 16 tokens i of the chunk and key channel d:
//   beta_i = sigma(beta_raw_i)
//   a_i[d] = 2^(lower_bound * log2(e) * sigma(g_raw_i[d]))      (= alpha_i[d])
//   P_i = prod_{m<=i} a_m = D_{0:i},   Q_i = prod_{i<m<16} a_m = D_{i+1:last}
//   rq_i = s / |q_i|, rk_i = 1 / |k_i|  (tensor-core Gram diagonals of the raw rows)
//   the decayed factors of the unnormalised rows, taken relative to the
//   middle of the chunk, m = P_7 (the product over tokens 0-7):
//     qM_i = q_i P_i / m,  kM_i = k_i P_i / m,  kI_i = k_i m / P_i = k_i Q_i / Q_7,
//     and kQ_i = k_i Q_i (Kend')
//   Mkk = kM kI^T, Mqk = qM kI^T                         (16 x 16, K = 128)
// (m cancels in both products.)  With the midpoint, P_i / m and m / P_i stay
// within 2^(+-7.3 * 8) at lower_bound = -5, where P_i and 1 / P_i alone reach
// 2^(+-115.4): a key row k / P_i would overflow fp32 and bf16 for raw
// |k_d| above about 2^12.6, and k P_i would lose small rows below the normal
// range, while the midpoint form keeps raw rows up to about 2^60 finite.
// The normalisation is applied to the 16 x 16 matrices and the 16 per-token
// rows instead of the 128-channel factors, so the factor pass needs no norm:
// with D = diag(rk), the record holds
//   Qdec = qP,  Kend' = kQ (= D^-1 Kend),  Aqk' = lower(Mqk) (= diag(rq)^-1 Aqk D^-1),
//   W' = D W,  U' = D U,  and rq,
// and the recurrence computes E'^T = U' - W' S^T = D E^T, S += E' Kend' and
// O = diag(rq) (Qdec S^T + Aqk' E'^T), which equal the unscaled products (rho
// and chi of sec. 6.3/6.5 and the state update of sec. 6.4).  W' and U' come from
//   R' = D R D^-1 = strictly-lower(diag(beta rk^2) Mkk),  A' = (I + R')^-1 = D A D^-1
//   W' = A' diag(beta rk^2) kP = (A' diag(beta rk^2) kM) Diag(m),   U' = A' diag(beta rk) V.
// Decay factors are prefix/suffix products of per-token retention factors, so
// their range is that of D_{0:i} itself: with lower_bound >= -5 and 16 tokens
// every factor and its inverse stays a normal fp32 number.
//
// Precision.  The norms are exact fp32 sums: the raw rows are bf16, so their
// products are exact in the bf16 tensor-core MMA with fp32 accumulation.  The
// intra-chunk products Mkk, Mqk and W take bf16 operands with fp32
// accumulation, as FlashKDA's chunk kernel does ("FlashKDA v1: A Deep Dive",
// sec. 3).  A' comes from fp32 forward substitution.  U keeps A' diag(beta rk)
// as a bf16 high part plus remainder (two products) because its rounding would
// go straight into the state.  The record holds Qdec and W' as bf16 (the
// recurrence's first MMA reads a bf16 snapshot of the state, as FlashKDA's
// bf16 state does) and Kend', Aqk', U', dlast as fp32 (the tf32 MMAs read
// their tf32 part).
//
// Raw input tiles (16 rows of 128 bf16) live in shared buffers of the caller:
// q, k, g_raw of a chunk in one buffer (in that order), v in another.  They
// arrive by tensor-map (TMA) copies, two boxes per tile (layout in
// kda_tma.cuh), issued by one thread onto an mbarrier: q, k, g_raw during an
// earlier build, once that build's factor pass is done with its buffer, and
// v at the start of the chunk's own build.  In a partial chunk the rows past
// its end (whatever follows in the tensor) are overwritten once the tiles
// are there: zeros for q, k, v and -inf for g_raw, so those tokens are no-ops
// and their record rows are zero.
#pragma once

#include "kda_common.cuh"
#include "kda_tma.cuh"

namespace kda {

constexpr int RS = 20;  // float row stride of -R'^T (conflict-free accumulator stores)
constexpr int AS = 24;  // float row stride of the A' tiles (conflict-free fragment loads)

enum { RAW_Q = 0, RAW_K = 1, RAW_G = 2 };
constexpr int QKG_BYTES = 3 * RAW_TILE;  // one chunk's q, k, g_raw tiles
constexpr int V_BYTES = RAW_TILE;        // one chunk's v tile

// Per-group scratch.  Derived operand tiles are bf16, stored transposed,
// [128 channels][16 tokens] (32 B per channel, tokens 0-7 and 8-15 in two
// 16-byte halves); drv_off's swizzle keeps the ldmatrix reads and the factor
// pass's stores conflict-free.
struct ChunkSmem {
  uint8_t kd[4096];  // kM = k P / m
  uint8_t ki[4096];  // kI = k m / P
  uint8_t qd[4096];  // qM = q P / m
  float Rt[16][RS];  // Rt[m][i] = -R'[i][m] for m < i, 0 otherwise
  float Aw[16][AS];  // A' diag(beta rk^2)
  float Au[16][AS];  // A' diag(beta rk)
  float pm[128];     // m = P_7 per key channel (the W' columns are scaled by it)
  float rq[16], rk[16], beta[16];
  float g2[4][16];  // partial squared norms (warp w: q for w < 2, k otherwise)
  float2 hx[4][32];  // the half-chunk products of each thread's channel pair
};

// byte offset of (channel d, token half h) in a derived tile: the eight
// 16-byte slots of each 128-byte group of four channels are XOR-permuted by 3
// in every other group
__device__ __forceinline__ int drv_off(int d, int h) {
  return ((d >> 2) << 7) + ((((d & 3) << 1 | h) ^ (((d >> 2) & 1) * 3)) << 4);
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
// the same loads from a 32-bit shared-memory address (constant offsets fold
// into the instruction)
__device__ __forceinline__ void ldsm_x4_t_at(uint32_t (&r)[4], uint32_t a) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void ldsm_x2_t_at(uint32_t (&r)[2], uint32_t a) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(a));
}
// four 8 x 8 b16 tiles from mma fragments (lane l: row l / 4, elements
// 2 (l % 4), + 1 of each) to 16-byte rows of shared memory; lane l gives the
// address of row (l & 7) of tile l >> 3
__device__ __forceinline__ void stsm_x4(void* p, const uint32_t (&r)[4]) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(smem_u32(p)),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
               : "memory");
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}


__device__ __forceinline__ float2 bf2_at(const uint8_t* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}

// bf16 pair of an fp32 pair, and the bf16 pair of its remainder
__device__ __forceinline__ void split2(float2 x, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x.x, x.y);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 r = __floats2bfloat162_rn(x.x - hf.x, x.y - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&r);
}

// Barrier over the 128 threads that build records (named barrier 1, so that a
// larger CTA can run other warps beside them).
__device__ __forceinline__ void chunk_sync() { named_bar(1, 128); }

// AND of `pred` over the 128 chunk threads (named barrier 1).
__device__ __forceinline__ bool chunk_all(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, 1, 128, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred))
      : "memory");
  return r != 0;
}

// q, k and g_raw of one chunk (first token t0, head h) into the buffer `raw`,
// completing on `bar` (initialised for one arrival): one thread issues them.
// With the scalar gate only q and k are copied; broadcast_gate_tile writes g.
__device__ __forceinline__ void issue_qkg_tma(const RawMaps& maps, uint8_t* raw, int h,
                                              int64_t t0, bool gate_scalar, uint64_t* bar) {
  mbar_arrive_expect_tx(bar, (gate_scalar ? 2 : 3) * RAW_TILE);
  const int t = static_cast<int>(t0);
  tma_tile(raw + RAW_Q * RAW_TILE, &maps.q, h, t, bar);
  tma_tile(raw + RAW_K * RAW_TILE, &maps.k, h, t, bar);
  if (!gate_scalar) tma_tile(raw + RAW_G * RAW_TILE, &maps.g, h, t, bar);
}
// v of one chunk into the v buffer, completing on `bar`: one thread.
__device__ __forceinline__ void issue_v_tma(const RawMaps& maps, uint8_t* vt, int h, int64_t t0,
                                            uint64_t* bar) {
  mbar_arrive_expect_tx(bar, RAW_TILE);
  tma_tile(vt, &maps.v, h, static_cast<int>(t0), bar);
}
// Scalar gate (one g_raw per token and head, broadcast over the key channels):
// the g tile written with plain stores by the 128 threads, thread t the
// 16-byte pieces (t & 7) of row t >> 3 in both boxes.  gs points at the
// chunk's first token, head h, with token stride `gstride`; rows past the end
// hold -inf (sigma(-inf) = 0, so a = 2^0 = 1).
__device__ __forceinline__ void broadcast_gate_tile(uint8_t* tile, const __nv_bfloat16* gs,
                                                    int64_t gstride, int nc, int t) {
  const int r = t >> 3, pc = t & 7;
  uint32_t w = 0xFF80FF80u;
  if (r < nc) {
    const uint32_t b = __bfloat16_as_ushort(gs[r * gstride]);
    w = b | (b << 16);
  }
  const uint4 x = make_uint4(w, w, w, w);
  *reinterpret_cast<uint4*>(tile + r * RAW_ROW + pc * 16) = x;
  *reinterpret_cast<uint4*>(tile + RAW_BOX + r * RAW_ROW + pc * 16) = x;
}

// Rows nc .. 15 of a raw tile that arrived by TMA hold whatever follows the
// chunk in the tensor: in a partial chunk the 128 threads overwrite them with
// `fill` (two bf16 per word), thread t the 16-byte pieces (t & 7) of row
// t >> 3 in both boxes.  Zero rows of q, k and v, and -inf rows of g_raw
// (retention 2^0 = 1), make those tokens no-ops, as the record format states.
__device__ __forceinline__ void fill_rows_past_end(uint8_t* tile, int nc, uint32_t fill, int t) {
  const int r = t >> 3, pc = t & 7;
  if (r < nc) return;
  const uint4 x = make_uint4(fill, fill, fill, fill);
  *reinterpret_cast<uint4*>(tile + r * RAW_ROW + pc * 16) = x;
  *reinterpret_cast<uint4*>(tile + RAW_BOX + r * RAW_ROW + pc * 16) = x;
}

// Bounded wait of the chunk threads on a raw-tile barrier: false once
// *abort is set or the wait runs out (then *abort is set and the error word
// latches KDA_ERR_TIMEOUT), as every wait of libkda.
__device__ __forceinline__ bool raw_wait(uint64_t* bar, uint32_t parity, int* abort, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity, kSleepHintNs)) {
    if (*reinterpret_cast<volatile int*>(abort)) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      *reinterpret_cast<volatile int*>(abort) = 1;
      atomicExch(err, 5);
      return false;
    }
  }
  return true;
}

// Where the raw tiles of the chunk being built arrive: the q/k/g_raw barrier
// and phase, and (unless the record's U' is known to be zero) the v barrier
// and phase; `abort` and `err` as in raw_wait.  Optionally the q/k/g_raw
// barrier and phase of the next chunk the thread builds, which the build
// tests without waiting (at its v wait) and reports in *next_ready; a later
// build given qkg_ready = that result skips its own wait.  A parity test is
// only exact once the barrier's previous phase is known complete: true for
// the next chunk of a double buffer whose previous use this thread waited on.
struct RawSync {
  uint64_t* qkg_bar;
  uint32_t qkg_parity;
  uint64_t* v_bar;
  uint32_t v_parity;
  int* abort;
  int* err;
  bool qkg_ready = false;
  uint64_t* next_qkg_bar = nullptr;
  uint32_t next_qkg_parity = 0;
  bool* next_ready = nullptr;
};

// Build the record of one chunk whose q, k, g_raw tiles were issued into `raw`
// with issue_qkg_tma (this call waits for them on rs.qkg_bar).  Its v tile
// goes to `vt` (waited on rs.v_bar; issued by load_v, or by the caller before
// the call).  All 128 threads of the
// group must call it.  beta_raw_bits: thread t < 16 holds the bf16 bits of token t's
// beta_raw (any value for t >= nc).  `rec` is the record base (global or
// shared memory).  Hooks, each run by
// all 128 threads:
//   may_write(ok)  before the first write to the record, with ok = whether
//                the raw tiles arrived; returns, uniformly, whether to go on
//                (the fused kernel also waits there until the previous record
//                of this stage is consumed).  Includes a barrier of the group.
//                On false nothing is written.
//   load_v()     right after may_write: issue this chunk's v tile (issue_v_tma),
//                unless the caller issued it earlier.
//   next_qkg()   once the factor pass is done with `raw`: issue a later chunk's
//                q, k, g_raw tiles (into `raw` or another buffer).
// Returns may_write().  With u_zero (v known to be zero) U' is zero and is
// neither formed nor written; the reader must take it as zero.
// kRecShared: `rec` is in shared memory (the fused kernel's ring), so W' goes
// out through stmatrix, which addresses shared memory only; a global record
// (K1) takes plain 4-byte stores.
template <bool kRecShared, class MayWrite, class LoadV, class NextQKG>
__device__ __forceinline__ bool build_chunk_record(ChunkSmem& S, uint8_t* raw, uint8_t* vt,
                                                   const RawSync& rs, uint32_t beta_raw_bits,
                                                   int nc, float scale,
                                                   float lb_log2e, float eps, uint8_t* rec, int t,
                                                   MayWrite&& may_write, LoadV&& load_v,
                                                   NextQKG&& next_qkg, bool u_zero = false) {
  const int w = t >> 5, l = t & 31;
  const bool arrived = rs.qkg_ready || raw_wait(rs.qkg_bar, rs.qkg_parity, rs.abort, rs.err);
  if (nc < kChunk) {
    fill_rows_past_end(raw + RAW_Q * RAW_TILE, nc, 0u, t);
    fill_rows_past_end(raw + RAW_K * RAW_TILE, nc, 0u, t);
    fill_rows_past_end(raw + RAW_G * RAW_TILE, nc, 0xFF80FF80u, t);
  }
  if (t < 16) {
    const float br = __bfloat162float(__ushort_as_bfloat16(static_cast<unsigned short>(beta_raw_bits)));
    S.beta[t] = (t < nc) ? sigmoid_fast(br) : 0.f;
  }
  if (!may_write(arrived)) return false;  // includes a barrier of the 128 threads
  load_v();

  // ---- factor pass: norms (tensor cores), retention factors, decayed factors ----
  // Thread (w, l): token half hf = l & 1 (tokens 8 hf .. 8 hf + 7) and key
  // channels d0, d0 + 1 of the 32-channel group (w & 1) ^ hf of box w >> 1.
  // The two half-warps of one load thus read rows ii and 8 + ii in opposite
  // 64-byte halves of the banks (conflict-free); the thread with the same
  // channels and the other token half is lane l ^ 1 of warp w ^ 1.
  const int hf = l & 1;
  const int d0 = 64 * (w >> 1) + 32 * ((w & 1) ^ hf) + 2 * (l >> 1);
  // byte offset of the thread's bf16 pair in raw row 8 hf + ii
  const int rbase = raw_off(8 * hf, d0);
  auto roff = [&](int ii) { return rbase + ii * RAW_ROW; };

  // Warp w: the 16 x 16 Gram matrix G = X X^T of X = q (w < 2) or k over the
  // channels of k-steps 4 (w & 1) .. +3, of which only the diagonal is kept.
  // In X X^T the B fragments of each k-step are registers of the A fragment
  // (rows 0-7: a0, a2; rows 8-15: a1, a3), so one ldmatrix per k-step feeds
  // both column tiles.  The gate math below fills the MMA latency.
  const int nx = (w >> 1) ? RAW_K : RAW_Q;
  float gacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};  // column tiles 0, 1
  {
    const int mi = l >> 3;
    const uint8_t* pa = raw + nx * RAW_TILE + raw_off((l & 7) + (mi & 1) * 8, 64 * (w & 1)) +
                        (mi >> 1) * 16;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t a[4];
      ldsm_x4(a, pa + kk * 32);
      mma16816(gacc[0], a, a[0], a[2]);
      mma16816(gacc[1], a, a[1], a[3]);
    }
  }
  // retention factors of this thread's 8 tokens, two channels each, and their
  // running products inside the half
  float2 a[8], Pl[8];
  {
    const float hl = 0.5f * lb_log2e;  // a = 2^(lb log2e sigma(x)), sigma(x) = (1 + tanh(x/2)) / 2
#pragma unroll
    for (int ii = 0; ii < 8; ++ii) {
      const float2 gh = __fmul2_rn(bf2_at(raw + RAW_G * RAW_TILE + roff(ii)), make_float2(0.5f, 0.5f));
      const float2 e = __ffma2_rn(make_float2(hl, hl),
                                  make_float2(tanh_approx(gh.x), tanh_approx(gh.y)),
                                  make_float2(hl, hl));
      a[ii].x = ex2_approx(e.x);
      a[ii].y = ex2_approx(e.y);
      Pl[ii] = ii ? __fmul2_rn(Pl[ii - 1], a[ii]) : a[ii];
    }
  }
  S.hx[w][l] = Pl[7];  // read by the other token half after the pair barrier
  {
    // diagonal: lane (g = l >> 2, c = l & 3) holds columns 8 nt + 2c, +1 of
    // rows g (acc 0, 1) and g + 8 (acc 2, 3) of column tile nt; the two warps
    // of a matrix add their halves of the channels
    const int g = l >> 2, e = g - 2 * (l & 3);
    if (e == 0 || e == 1) {
      S.g2[w][g] = e ? gacc[0][1] : gacc[0][0];
      S.g2[w][g + 8] = e ? gacc[1][3] : gacc[1][2];
    }
    if (w < 2)
      named_bar(3, 64);  // the q pair
    else
      named_bar(4, 64);  // the k pair
    if ((w & 1) == 0 && l < 16) {
      const float s2 = S.g2[w][l] + S.g2[w + 1][l];
      if (nx == RAW_Q)
      {
        const float r = scale * rsqrtf(s2 + eps);  // the read scale is folded into q's norm
        S.rq[l] = r;
        *reinterpret_cast<float*>(rec + OFF_RQ + 4 * l) = r;
      }
      else
        S.rk[l] = rsqrtf(s2 + eps);
    }
  }
  // products over the other half, from lane l ^ 1 of warp w ^ 1 (written
  // before the pair barrier above)
  const float2 Hh = Pl[7];
  const float2 Ho = S.hx[w ^ 1][l ^ 1];
  float2 Qu[8];  // q P of this thread's tokens (Qdec; rq is applied to the outputs)
  {
    const float2 one = make_float2(1.f, 1.f);
    const float2 dl = hf ? __fmul2_rn(Ho, Hh) : __fmul2_rn(Hh, Ho);  // same product in both lanes
    float2 sfx = hf ? one : Ho;  // prod over the tokens after the one being processed
    // midpoint m = P_7 (first half's product) and Q_7 = dlast / m (second half's):
    // P_i / m = Pl_i / Hh in the first half and Pl_i in the second
    const float2 h1 = hf ? Ho : Hh, h2 = hf ? Hh : Ho;
    const float2 rel = hf ? one : make_float2(rcp_approx(Hh.x), rcp_approx(Hh.y));
    const float2 inv_q7 = make_float2(rcp_approx(h2.x), rcp_approx(h2.y));
    if (hf == 0) {
      *reinterpret_cast<float2*>(rec + OFF_DL + d0 * 4) = dl;
      *reinterpret_cast<float2*>(&S.pm[d0]) = h1;
    }
    // packed bf16 words, [token pair m] for channel d0 (x) and d0+1 (y)
    uint32_t qx[4], qy[4], kx[4], ky[4], ix[4], iy[4];
    float ex[8], ey[8];  // kQ of channels d0, d0 + 1
#pragma unroll
    for (int m = 3; m >= 0; --m) {
      float2 Kd[2], Ki[2], Qm[2];
#pragma unroll
      for (int o = 1; o >= 0; --o) {
        const int ii = 2 * m + o;
        const float2 Q = sfx;
        sfx = __fmul2_rn(sfx, a[ii]);
        const float2 Pm = __fmul2_rn(Pl[ii], rel);  // P_i / m
        const float2 qv = bf2_at(raw + RAW_Q * RAW_TILE + roff(ii));
        const float2 kv = bf2_at(raw + RAW_K * RAW_TILE + roff(ii));
        Qm[o] = __fmul2_rn(qv, Pm);
        Qu[ii] = __fmul2_rn(Qm[o], h1);  // q P_i = (q P_i / m) m
        Kd[o] = __fmul2_rn(kv, Pm);
        const float2 Ke = __fmul2_rn(kv, Q);
        Ki[o] = __fmul2_rn(Ke, inv_q7);
        ex[ii] = Ke.x;
        ey[ii] = Ke.y;
      }
      qx[m] = pack_bf16(Qm[0].x, Qm[1].x);
      qy[m] = pack_bf16(Qm[0].y, Qm[1].y);
      kx[m] = pack_bf16(Kd[0].x, Kd[1].x);
      ky[m] = pack_bf16(Kd[0].y, Kd[1].y);
      ix[m] = pack_bf16(Ki[0].x, Ki[1].x);
      iy[m] = pack_bf16(Ki[0].y, Ki[1].y);
    }
    const int ox = drv_off(d0, hf), oy = drv_off(d0 + 1, hf);
    *reinterpret_cast<uint4*>(S.qd + ox) = make_uint4(qx[0], qx[1], qx[2], qx[3]);
    *reinterpret_cast<uint4*>(S.qd + oy) = make_uint4(qy[0], qy[1], qy[2], qy[3]);
    *reinterpret_cast<uint4*>(S.kd + ox) = make_uint4(kx[0], kx[1], kx[2], kx[3]);
    *reinterpret_cast<uint4*>(S.kd + oy) = make_uint4(ky[0], ky[1], ky[2], ky[3]);
    *reinterpret_cast<uint4*>(S.ki + ox) = make_uint4(ix[0], ix[1], ix[2], ix[3]);
    *reinterpret_cast<uint4*>(S.ki + oy) = make_uint4(iy[0], iy[1], iy[2], iy[3]);
    // Kend': this half's 8 tokens are one K=8 tile row, two 16-byte pieces
    *reinterpret_cast<float4*>(rec + kend_offset(d0, hf * 8)) = make_float4(ex[0], ex[1], ex[2], ex[3]);
    *reinterpret_cast<float4*>(rec + kend_offset(d0, hf * 8 + 4)) = make_float4(ex[4], ex[5], ex[6], ex[7]);
    *reinterpret_cast<float4*>(rec + kend_offset(d0 + 1, hf * 8)) = make_float4(ey[0], ey[1], ey[2], ey[3]);
    *reinterpret_cast<float4*>(rec + kend_offset(d0 + 1, hf * 8 + 4)) = make_float4(ey[4], ey[5], ey[6], ey[7]);
  }
  chunk_sync();
  // q, k and g_raw of this chunk are no longer read
  next_qkg();

  // ---- Mkk (warps 0,1) -> -R'^T, Mqk (warps 2,3) -> Aqk'; Qdec -> record ----
  {
    const int mat = w >> 1, nt = w & 1;
    float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};  // even / odd k-steps
    const int mi = l >> 3;
    // channel rows kk*16 + r of the tiles are drv_off(r, h) + 512 kk
    const uint32_t abase = smem_u32(mat ? S.qd : S.kd) + drv_off((l & 7) + (mi >> 1) * 8, mi & 1);
    const uint32_t bbase = smem_u32(S.ki) + drv_off((l & 7) + (mi & 1) * 8, nt);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t ar[4], br[2];
      ldsm_x4_t_at(ar, abase + kk * 512);
      ldsm_x2_t_at(br, bbase + kk * 512);
      mma16816(acc2[kk & 1], ar, br[0], br[1]);
    }
    // Qdec = qP, bf16 rows 0..15 of [Qdec ; W'] (this thread's pairs)
#pragma unroll
    for (int ii = 0; ii < 8; ++ii)
      *reinterpret_cast<uint32_t*>(rec + b1_offset(hf * 8 + ii, d0)) = pack_bf16(Qu[ii].x, Qu[ii].y);
    float acc[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] = acc2[0][e] + acc2[1][e];
    const int r0 = l >> 2, c0 = nt * 8 + (l & 3) * 2;
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int i = r0 + h2 * 8;
      if (mat == 0) {
        const float rki = S.rk[i];
        const float f = -(S.beta[i] * rki * rki);
#pragma unroll
        for (int o = 0; o < 2; ++o) {
          const int m = c0 + o;
          S.Rt[m][i] = m < i ? f * acc[2 * h2 + o] : 0.f;
        }
      } else {
#pragma unroll
        for (int o = 0; o < 2; ++o) {
          const int j = c0 + o;
          *reinterpret_cast<float*>(rec + aqk_offset(i, j)) = j <= i ? acc[2 * h2 + o] : 0.f;
        }
      }
    }
  }
  chunk_sync();

  // ---- A' = (I + R')^-1 by fp32 forward substitution in warp 0: lane j (and
  // j + 16, which repeats it) carries column j; after column m of R' has been
  // applied, entry m is final.  Writes A' diag(beta rk^2) (lanes 0-15) and
  // A' diag(beta rk) (lanes 16-31). ----
  if (w == 0) {
    const int j = l & 15;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
    for (int m = 0; m < 15; ++m) {
#pragma unroll
      for (int i4 = (m + 1) >> 2; i4 < 4; ++i4) {
        const float4 r = *reinterpret_cast<const float4*>(&S.Rt[m][4 * i4]);
        const float rv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (4 * i4 + e > m) x[4 * i4 + e] = fmaf(rv[e], x[m], x[4 * i4 + e]);
      }
    }
    const float rkj = S.rk[j];
    const float cu = S.beta[j] * rkj, cw = cu * rkj;
    // lanes 0-15 write column j of A' diag(beta rk^2), lanes 16-31 (which
    // computed the same column) that of A' diag(beta rk)
    {
      float* dst = l < 16 ? &S.Aw[0][j] : &S.Au[0][j];
      const float f = l < 16 ? cw : cu;
#pragma unroll
      for (int i = 0; i < 16; ++i) dst[i * AS] = x[i] * f;
    }
  }
  // this chunk's v tile (a timeout latches the error and the record is
  // finished on whatever is there; the caller sees the error word)
  if (rs.next_ready)
    *rs.next_ready = rs.next_qkg_bar && mbar_test_wait(rs.next_qkg_bar, rs.next_qkg_parity);
  if (!u_zero) {
    raw_wait(rs.v_bar, rs.v_parity, rs.abort, rs.err);
    if (nc < kChunk) fill_rows_past_end(vt, nc, 0u, t);
  }
  chunk_sync();

  // ---- W' = A' diag(beta rk^2) kP, U' = A' diag(beta rk) V (warp w: channels 32w..32w+31) ----
  {
    const int mi = l >> 3, g = l >> 2, q2 = (l & 3) * 2;
    auto ld2 = [](const float* p) { return *reinterpret_cast<const float2*>(p); };
    // W' [i][c] = m_c (A' diag(beta rk^2) kM)[i][c]: A = A' diag(beta rk^2) [i][j]
    // (bf16), B = kM^T tile [c][j] ([n][k] order)
    uint32_t ah[4];
    {
      const float2 f0 = ld2(&S.Aw[g][q2]), f1 = ld2(&S.Aw[g + 8][q2]);
      const float2 f2 = ld2(&S.Aw[g][q2 + 8]), f3 = ld2(&S.Aw[g + 8][q2 + 8]);
      ah[0] = pack_bf16(f0.x, f0.y);
      ah[1] = pack_bf16(f1.x, f1.y);
      ah[2] = pack_bf16(f2.x, f2.y);
      ah[3] = pack_bf16(f3.x, f3.y);
    }
#pragma unroll
    for (int pair = 0; pair < 2; ++pair) {
      const int n0 = w * 32 + pair * 16;
      uint32_t bk[4], wf[4];
      ldsm_x4(bk, S.kd + drv_off(n0 + (l & 7) + (mi >> 1) * 8, mi & 1));
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float wacc[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816(wacc, ah, bk[2 * half], bk[2 * half + 1]);
        const float2 mc = *reinterpret_cast<const float2*>(&S.pm[n0 + half * 8 + q2]);
        wf[2 * half] = pack_bf16(wacc[0] * mc.x, wacc[1] * mc.y);      // rows g
        wf[2 * half + 1] = pack_bf16(wacc[2] * mc.x, wacc[3] * mc.y);  // rows g + 8
      }
      if constexpr (kRecShared) {
        // the four 8 x 8 bf16 tiles (W' rows 0-7 / 8-15 x channels n0.. /
        // n0+8..) in one stmatrix: lane l gives the address of row (l & 7) of
        // tile l >> 3, a 16-byte piece of the swizzled [Qdec ; W'] tile
        stsm_x4(rec + b1_offset(16 + (l & 7) + 8 * (mi & 1), n0 + 8 * (mi >> 1)), wf);
      } else {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int c = n0 + half * 8 + q2;
          *reinterpret_cast<uint32_t*>(rec + b1_offset(16 + g, c)) = wf[2 * half];
          *reinterpret_cast<uint32_t*>(rec + b1_offset(24 + g, c)) = wf[2 * half + 1];
        }
      }
    }
    // U'^T [c][i] = V^T (A' diag(beta rk))^T: A = V^T from the raw v tile
    // (transposed load), B[j][i] = (A' diag(beta rk))[i][j] as high and low
    // bf16 parts; each lane then holds two consecutive tokens of one channel
    if (u_zero) return true;
    uint32_t bh[4], bl[4];
    split2(ld2(&S.Au[g][q2]), bh[0], bl[0]);
    split2(ld2(&S.Au[g][q2 + 8]), bh[1], bl[1]);
    split2(ld2(&S.Au[g + 8][q2]), bh[2], bl[2]);
    split2(ld2(&S.Au[g + 8][q2 + 8]), bh[3], bl[3]);
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const int m0 = w * 32 + mt * 16;
      const int j = (l & 7) + (mi >> 1) * 8;
      uint32_t av[4];
      ldsm_x4_t(av, vt + raw_off(j, m0 + 8 * (mi & 1)));
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        float u[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816(u, av, bh[2 * nt], bh[2 * nt + 1]);
        mma16816(u, av, bl[2 * nt], bl[2 * nt + 1]);
        *reinterpret_cast<float2*>(rec + u_offset(m0 + g, nt * 8 + q2)) = make_float2(u[0], u[1]);
        *reinterpret_cast<float2*>(rec + u_offset(m0 + g + 8, nt * 8 + q2)) = make_float2(u[2], u[3]);
      }
    }
  }
  return true;
}

// Locate record slot `slot`: the sequence n with slot0(n) <= slot < slot0(n+1)
// and the chunk index c inside it.  Returns false for an unused slot.
__device__ __forceinline__ bool locate_slot(const int32_t* cu, int64_t T_total, int N,
                                            int64_t slot, int& n, int64_t& bos, int64_t& eos,
                                            int64_t& c) {
  int lo = 0, hi = N - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    int64_t b, e;
    seq_bounds(cu, T_total, N, mid, b, e);
    if (b / kChunk + mid <= slot)
      lo = mid;
    else
      hi = mid - 1;
  }
  n = lo;
  seq_bounds(cu, T_total, N, n, bos, eos);
  c = slot - (bos / kChunk + n);
  return c >= 0 && c * kChunk < (eos - bos);
}

}  // namespace kda
