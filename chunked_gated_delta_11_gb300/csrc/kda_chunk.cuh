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
//   |q_i|^2, |k_i|^2 from the raw bf16 rows (tensor-core Gram diagonals)
//   Qdec_i = s q_i P_i / |q_i|, Kdec_i = k_i P_i / |k_i|, Kend_i = k_i Q_i / |k_i|,
//   Kinv_i = Kend_i / dlast
//   Mkk = Kdec Kinv^T, Mqk = Qdec Kinv^T              (16 x 16, K = 128)
//   R = strictly-lower(diag(beta) Mkk), Aqk = lower(Mqk)  (rho and chi of sec. 6.3/6.5)
//   A = (I + R)^-1 = (I - R)(I + R^2)(I + R^4)(I + R^8)  (finite Neumann series)
//   W = A diag(beta) Kdec,  U = A diag(beta) V
// Decay factors are prefix/suffix products of per-token retention factors, so
// their range is that of D_{0:i} itself: with lower_bound >= -5 and 16 tokens
// every factor and its inverse stays a normal fp32 number.
//
// Precision.  The norms are exact fp32 sums: the raw rows are bf16, so their
// products are exact in the bf16 tensor-core MMA with fp32 accumulation.  The
// intra-chunk products Mkk, Mqk and W take bf16 operands with fp32
// accumulation, as FlashKDA's chunk kernel does ("FlashKDA v1: A Deep Dive",
// sec. 3).  U keeps A diag(beta) as a bf16 high part plus remainder (two
// products) because its rounding would go straight into the state.  The
// inverse runs as bf16 tensor-core products of high/low operand splits (about
// 16 significant bits per operand) with fp32 accumulation and fp32 additive
// terms.  The record holds Qdec and W as bf16 (the recurrence's first MMA
// reads a bf16 snapshot of the state, as FlashKDA's bf16 state does) and Kend,
// Aqk, U, dlast as fp32 (the tf32 MMAs read their tf32 part).
//
// Raw input tiles (16 rows of 128 bf16, 4 KB each) live in shared buffers of
// the caller: q, k, g_raw of a chunk in one 12 KB buffer (in that order), v in
// a 4 KB one; rows of 256 bytes whose 16-byte pieces are XOR-swizzled by
// (row & 7).  They arrive as two cp.async groups: q, k, g_raw (issued during an
// earlier build, once that build's gate phase is done with its own buffer) and
// v (issued at the start of the chunk's own build, once the previous U
// products are done with the v buffer).
#pragma once

#include "kda_common.cuh"

namespace kda {

constexpr int AS = 24;  // bf16 row stride of the 16 x 16 A diag(beta) tiles (48 B)

enum { RAW_Q = 0, RAW_K = 1, RAW_G = 2 };
constexpr int QKG_BYTES = 3 * 4096;  // one chunk's q, k, g_raw tiles
constexpr int V_BYTES = 4096;        // one chunk's v tile

// Per-group scratch.  Derived operand tiles are bf16, stored transposed,
// [128 channels][16 tokens] (32 B per channel), 16-byte halves swizzled by
// bit 2 of the channel, which keeps the ldmatrix reads conflict-free.
struct ChunkSmem {
  uint8_t kd[4096];  // Kdec
  uint8_t ki[4096];  // Kinv
  uint8_t qd[4096];  // Qdec
  float Rf[16][20];  // R = strictly-lower(diag(beta) Mkk), fp32, rows of 20 floats
  __nv_bfloat16 abh[16 * AS];  // A diag(beta), high
  __nv_bfloat16 abl[16 * AS];  // A diag(beta), low
  float rq[16], rk[16], beta[16];
  float2 hx[2][64];  // per channel pair: prod of a over tokens 0-7, over tokens 8-15
};

__device__ __forceinline__ uint8_t* raw_row(uint8_t* raw, int x, int i) {
  return raw + x * 4096 + i * 256;
}
// byte offset of 16-byte piece c of raw row i
__device__ __forceinline__ int raw_piece(int i, int c) { return (c ^ (i & 7)) << 4; }
// byte offset of (channel d, token-half p) in a derived tile
__device__ __forceinline__ int drv_off(int d, int p) { return d * 32 + ((p ^ ((d >> 2) & 1)) << 4); }

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t (&r)[2], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(x);
  lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}

__device__ __forceinline__ float2 bf2_at(const uint8_t* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}

// Barrier over the 128 threads that build records (named barrier 1, so that a
// larger CTA can run other warps beside them).
__device__ __forceinline__ void chunk_sync() { named_bar(1, 128); }

// The raw-tile loads of one thread, set up once: thread t copies 16-byte piece
// (t & 15) of rows (t >> 4) and (t >> 4) + 8 of every tile with cp.async; rows
// past a chunk's end get `fill` (two bf16 per word) by plain stores instead.
struct TileLoader {
  uint32_t soff;     // shared offset of the piece in row (t >> 4) (row + 8: + 2048)
  int64_t goff;      // element offset of the piece from the chunk's first token
  int64_t rstride8;  // elements between a row and the row 8 further
  int row;
  __device__ __forceinline__ TileLoader(int t, int64_t row_stride) {
    row = t >> 4;
    const int c = t & 15;
    soff = static_cast<uint32_t>(row * 256 + ((c ^ (row & 7)) << 4));
    goff = row * row_stride + c * 8;
    rstride8 = row_stride * 8;
  }
  // tile: shared base of one 16-row tile; src: the chunk's first token, head h
  __device__ __forceinline__ void load(uint8_t* tile, const __nv_bfloat16* src, int nc,
                                       uint32_t fill) const {
    uint8_t* d = tile + soff;
    const __nv_bfloat16* s0 = src + goff;
    if (row < nc)
      cp_async16(d, s0);
    else
      *reinterpret_cast<uint4*>(d) = make_uint4(fill, fill, fill, fill);
    if (row + 8 < nc)
      cp_async16(d + 2048, s0 + rstride8);
    else
      *reinterpret_cast<uint4*>(d + 2048) = make_uint4(fill, fill, fill, fill);
  }
};
// Scalar gate (one g_raw per token and head, broadcast over the key channels):
// the g tile is written with plain stores.  gs points at the chunk's first
// token, head h; its token stride is `gstride` elements.
__device__ __forceinline__ void broadcast_gate_tile(const TileLoader& L, uint8_t* tile,
                                                    const __nv_bfloat16* gs, int64_t gstride,
                                                    int nc) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int row = L.row + 8 * half;
    uint32_t w = 0xFF80FF80u;
    if (row < nc) {
      const uint32_t b = __bfloat16_as_ushort(gs[row * gstride]);
      w = b | (b << 16);
    }
    *reinterpret_cast<uint4*>(tile + L.soff + 2048 * half) = make_uint4(w, w, w, w);
  }
}
// q, k and g_raw of one chunk (pointers at its first token, head h): the first
// cp.async group of its raw tiles.  gstride > 0: g_raw is one value per token
// and head (token stride gstride), broadcast over the key channels.
__device__ __forceinline__ void issue_qkg_loads(const TileLoader& L, uint8_t* raw,
                                                const __nv_bfloat16* q, const __nv_bfloat16* k,
                                                const __nv_bfloat16* g, int nc,
                                                int64_t gstride = 0) {
  L.load(raw + RAW_Q * 4096, q, nc, 0u);
  L.load(raw + RAW_K * 4096, k, nc, 0u);
  // g_raw rows past the end hold -inf: sigma(-inf) = 0 gives a = 2^0 = 1 exactly,
  // so those tokens neither decay nor change the running products
  if (gstride > 0)
    broadcast_gate_tile(L, raw + RAW_G * 4096, g, gstride, nc);
  else
    L.load(raw + RAW_G * 4096, g, nc, 0xFF80FF80u);
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// v of one chunk into a v buffer: the second group
__device__ __forceinline__ void issue_v_loads(const TileLoader& L, uint8_t* vt,
                                              const __nv_bfloat16* v, int nc) {
  L.load(vt, v, nc, 0u);
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// ---- 16 x 16 matrix products inside one warp (the triangular inverse) ----
// A 16 x 16 fp32 matrix M lives in the accumulator layout of two m16n8 tiles:
// lane (g = l / 4, q = l % 4) holds m[nt][e] = M[g + 8 (e >> 1)][8 nt + 2q + (e & 1)].
// Packed to bf16 pairs, those registers are exactly the A-operand fragment of
// an m16n8k16 product (a0 = m[0][0..1], a1 = m[0][2..3], a2 = m[1][0..1],
// a3 = m[1][2..3]); the B-operand fragments of M are the 8 x 8 transposes of
// the same four blocks (movmatrix).  Every operand is split into a bf16 high
// part and remainder and each product takes high*high + high*low + low*high
// (about 16 significant bits per operand) with fp32 accumulation.
struct Mat16 {
  float m[2][4];
};
struct OpA {
  uint32_t hi[4], lo[4];
};
struct OpB {
  uint32_t hi[4], lo[4];  // n-tile nt: {x[2 nt], x[2 nt + 1]}
};
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}
__device__ __forceinline__ OpA as_a(const Mat16& M) {
  OpA A;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const float x0 = M.m[r >> 1][(r & 1) * 2], x1 = M.m[r >> 1][(r & 1) * 2 + 1];
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 lo = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    A.hi[r] = *reinterpret_cast<const uint32_t*>(&h);
    A.lo[r] = *reinterpret_cast<const uint32_t*>(&lo);
  }
  return A;
}
__device__ __forceinline__ OpB as_b(const OpA& A) {
  OpB B;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    B.hi[r] = movmatrix_t(A.hi[r]);
    B.lo[r] = movmatrix_t(A.lo[r]);
  }
  return B;
}
// C = Init + X Y (Init may be null)
__device__ __forceinline__ Mat16 mat_mul(const OpA& X, const OpB& Y, const Mat16* Init) {
  Mat16 C;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    float acc[4], acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] = Init ? Init->m[nt][e] : 0.f;
    mma16816(acc2, X.lo, Y.hi[2 * nt], Y.hi[2 * nt + 1]);
    mma16816(acc2, X.hi, Y.lo[2 * nt], Y.lo[2 * nt + 1]);
    mma16816(acc, X.hi, Y.hi[2 * nt], Y.hi[2 * nt + 1]);
#pragma unroll
    for (int e = 0; e < 4; ++e) C.m[nt][e] = acc[e] + acc2[e];
  }
  return C;
}

// Zero the A diag(beta) tiles once (the inverse rewrites them in full).
__device__ __forceinline__ void clear_chunk_workspace(ChunkSmem& S, int t) {
  uint16_t* b = reinterpret_cast<uint16_t*>(S.abh);
  for (int e = t; e < 2 * 16 * AS; e += 128) b[e] = 0;
  named_bar(1, 128);
}

// Build the record of one chunk whose q, k, g_raw tiles were issued into `raw`
// with issue_qkg_loads (this call waits for them; `newer_qkg` says whether the
// q, k, g_raw group of a later chunk was issued after them, and may still be
// pending).  Its v tile goes to `vt`.  All 128 threads of the group must call
// it.  beta_raw_bits: thread t < 16 holds the bf16 bits of token t's
// beta_raw (any value for t >= nc).  `rec` is the record base (global or
// shared memory).  Hooks, each run by
// all 128 threads:
//   may_write()  before the first write to the record; returns, uniformly,
//                whether to go on (the fused kernel waits there until the
//                previous record of this stage is consumed).  Includes a
//                barrier of the group.  On false nothing is written.
//   load_v()     right after may_write: issue this chunk's v tile (issue_v_loads).
//   next_qkg()   once the gate phase is done with `raw`: issue a later chunk's
//                q, k, g_raw tiles (into `raw` or another buffer); returns
//                whether it issued them.
// Returns may_write().
template <class MayWrite, class LoadV, class NextQKG>
__device__ __forceinline__ bool build_chunk_record(ChunkSmem& S, uint8_t* raw, uint8_t* vt,
                                                   bool newer_qkg, uint32_t beta_raw_bits,
                                                   int nc, float scale,
                                                   float lb_log2e, float eps, uint8_t* rec, int t,
                                                   MayWrite&& may_write, LoadV&& load_v,
                                                   NextQKG&& next_qkg) {
  const int w = t >> 5, l = t & 31;
  if (newer_qkg)
    asm volatile("cp.async.wait_group 1;" ::: "memory");
  else
    asm volatile("cp.async.wait_group 0;" ::: "memory");
  if (t < 16) {
    const float br = __bfloat162float(__ushort_as_bfloat16(static_cast<unsigned short>(beta_raw_bits)));
    S.beta[t] = (t < nc) ? sigmoid_fast(br) : 0.f;
  }
  if (!may_write()) return false;  // includes a barrier of the 128 threads
  load_v();

  // Channel pair and token half of this thread in the gate phases.
  const int p = t & 63, hf = t >> 6, d0 = 2 * p;
  const int gpc = p >> 2, gsub = (p & 3) * 4;  // 16-byte piece and byte inside it

  // ---- phase 1: squared norms (tensor cores) and retention factors ----
  // warp w: Gram tile G[i][j] = sum_d X[i][d] X[j][d] of X = q (w < 2) or k,
  // columns j = 8 (w & 1) .. +7; only its diagonal is kept.  Two accumulator
  // chains (even / odd k-steps); the gate math below fills their latency.
  const int nx = (w >> 1) ? RAW_K : RAW_Q, ntn = w & 1;
  float gacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  {
    const int mi = l >> 3;
    const int arow = (l & 7) + (mi & 1) * 8;
    const int brow = ntn * 8 + (l & 7);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t a[4], b[2];
      ldsm_x4(a, raw_row(raw, nx, arow) + raw_piece(arow, 2 * kk + (mi >> 1)));
      ldsm_x2(b, raw_row(raw, nx, brow) + raw_piece(brow, 2 * kk + (mi & 1)));
      mma16816(gacc[kk & 1], a, b[0], b[1]);
    }
  }
  // retention factors of this thread's 8 tokens, two channels each, and their
  // running products inside the half
  float2 a[8], Pl[8];
  {
    const float hl = 0.5f * lb_log2e;  // a = 2^(lb log2e sigma(x)), sigma(x) = (1 + tanh(x/2)) / 2
#pragma unroll
    for (int ii = 0; ii < 8; ++ii) {
      const int i = hf * 8 + ii;
      const float2 gh = __fmul2_rn(bf2_at(raw_row(raw, RAW_G, i) + raw_piece(i, gpc) + gsub),
                                   make_float2(0.5f, 0.5f));
      const float2 e = __ffma2_rn(make_float2(hl, hl),
                                  make_float2(tanh_approx(gh.x), tanh_approx(gh.y)),
                                  make_float2(hl, hl));
      a[ii].x = ex2_approx(e.x);
      a[ii].y = ex2_approx(e.y);
      Pl[ii] = ii ? __fmul2_rn(Pl[ii - 1], a[ii]) : a[ii];
    }
    S.hx[hf][p] = Pl[7];
  }
  {
    // diagonal: lane (g = l >> 2, c = l & 3) holds columns 2c, 2c+1 of rows g
    // (acc 0, 1) and g + 8 (acc 2, 3) of the tile
    const int g = l >> 2, e = g - 2 * (l & 3);
    if (e == 0 || e == 1) {
      const float s2 = ntn ? (e ? gacc[0][3] + gacc[1][3] : gacc[0][2] + gacc[1][2])
                           : (e ? gacc[0][1] + gacc[1][1] : gacc[0][0] + gacc[1][0]);
      const int i = ntn * 8 + g;
      if (nx == RAW_Q)
        S.rq[i] = scale * rsqrtf(s2 + eps);  // the read scale is folded into q's norm
      else
        S.rk[i] = rsqrtf(s2 + eps);
    }
  }
  chunk_sync();

  // ---- phase 2: decayed factors -> record (Qdec, Kend, dlast) and tiles ----
  {
    const float2 h0 = S.hx[0][p], h1 = S.hx[1][p];
    const float2 dl = __fmul2_rn(h0, h1);
    const float2 pre = hf ? h0 : make_float2(1.f, 1.f);   // prod over tokens before the half
    const float2 post = hf ? make_float2(1.f, 1.f) : h1;  // prod over tokens after the half
    const float2 inv_dl = make_float2(rcp_approx(dl.x), rcp_approx(dl.y));
    if (hf == 0) *reinterpret_cast<float2*>(rec + OFF_DL + d0 * 4) = dl;
    const float4 rq0 = *reinterpret_cast<const float4*>(&S.rq[hf * 8]);
    const float4 rq1 = *reinterpret_cast<const float4*>(&S.rq[hf * 8 + 4]);
    const float4 rk0 = *reinterpret_cast<const float4*>(&S.rk[hf * 8]);
    const float4 rk1 = *reinterpret_cast<const float4*>(&S.rk[hf * 8 + 4]);
    const float rqv[8] = {rq0.x, rq0.y, rq0.z, rq0.w, rq1.x, rq1.y, rq1.z, rq1.w};
    const float rkv[8] = {rk0.x, rk0.y, rk0.z, rk0.w, rk1.x, rk1.y, rk1.z, rk1.w};
    // packed bf16 words, [token pair m] for channel d0 (x) and d0+1 (y)
    uint32_t qx[4], qy[4], kx[4], ky[4], ix[4], iy[4];
    float ex[8], ey[8];  // Kend of channels d0, d0 + 1
    float2 sfx = post;  // prod over the tokens after the one being processed
#pragma unroll
    for (int m = 3; m >= 0; --m) {
      float2 Qd[2], Kd[2], Ke[2], Ki[2];
#pragma unroll
      for (int o = 1; o >= 0; --o) {
        const int ii = 2 * m + o, i = hf * 8 + ii;
        const float2 Q = sfx;
        sfx = __fmul2_rn(sfx, a[ii]);
        const float2 P = __fmul2_rn(pre, Pl[ii]);
        const int off = raw_piece(i, gpc) + gsub;
        const float2 qv = bf2_at(raw_row(raw, RAW_Q, i) + off);
        const float2 kv = bf2_at(raw_row(raw, RAW_K, i) + off);
        Qd[o] = __fmul2_rn(__fmul2_rn(qv, make_float2(rqv[ii], rqv[ii])), P);
        const float2 kr = __fmul2_rn(kv, make_float2(rkv[ii], rkv[ii]));
        Kd[o] = __fmul2_rn(kr, P);
        Ke[o] = __fmul2_rn(kr, Q);
        Ki[o] = __fmul2_rn(Ke[o], inv_dl);
        *reinterpret_cast<uint32_t*>(rec + b1_offset(i, d0)) = pack_bf16(Qd[o].x, Qd[o].y);
      }
      qx[m] = pack_bf16(Qd[0].x, Qd[1].x);
      qy[m] = pack_bf16(Qd[0].y, Qd[1].y);
      kx[m] = pack_bf16(Kd[0].x, Kd[1].x);
      ky[m] = pack_bf16(Kd[0].y, Kd[1].y);
      ix[m] = pack_bf16(Ki[0].x, Ki[1].x);
      iy[m] = pack_bf16(Ki[0].y, Ki[1].y);
      ex[2 * m] = Ke[0].x;
      ex[2 * m + 1] = Ke[1].x;
      ey[2 * m] = Ke[0].y;
      ey[2 * m + 1] = Ke[1].y;
    }
    const int ox = drv_off(d0, hf), oy = drv_off(d0 + 1, hf);
    *reinterpret_cast<uint4*>(S.qd + ox) = make_uint4(qx[0], qx[1], qx[2], qx[3]);
    *reinterpret_cast<uint4*>(S.qd + oy) = make_uint4(qy[0], qy[1], qy[2], qy[3]);
    *reinterpret_cast<uint4*>(S.kd + ox) = make_uint4(kx[0], kx[1], kx[2], kx[3]);
    *reinterpret_cast<uint4*>(S.kd + oy) = make_uint4(ky[0], ky[1], ky[2], ky[3]);
    *reinterpret_cast<uint4*>(S.ki + ox) = make_uint4(ix[0], ix[1], ix[2], ix[3]);
    *reinterpret_cast<uint4*>(S.ki + oy) = make_uint4(iy[0], iy[1], iy[2], iy[3]);
    // Kend: this half's 8 tokens are one K=8 tile row, two 16-byte pieces
    *reinterpret_cast<float4*>(rec + kend_offset(d0, hf * 8)) = make_float4(ex[0], ex[1], ex[2], ex[3]);
    *reinterpret_cast<float4*>(rec + kend_offset(d0, hf * 8 + 4)) = make_float4(ex[4], ex[5], ex[6], ex[7]);
    *reinterpret_cast<float4*>(rec + kend_offset(d0 + 1, hf * 8)) = make_float4(ey[0], ey[1], ey[2], ey[3]);
    *reinterpret_cast<float4*>(rec + kend_offset(d0 + 1, hf * 8 + 4)) = make_float4(ey[4], ey[5], ey[6], ey[7]);
  }
  chunk_sync();
  // q, k and g_raw of this chunk are no longer read
  const bool prefetched = next_qkg();

  // ---- phase 3: Mkk (warps 0,1), Mqk (warps 2,3); R, I - R, Aqk from the
  // accumulators ----
  {
    const int mat = w >> 1, nt = w & 1;
    const uint8_t* A = mat ? S.qd : S.kd;
    float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};  // even / odd k-steps
    const int mi = l >> 3;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int arow = kk * 16 + (l & 7) + (mi >> 1) * 8;  // channel
      const int brow = kk * 16 + (l & 7) + (mi & 1) * 8;
      uint32_t ar[4], br[2];
      ldsm_x4_t(ar, A + drv_off(arow, mi & 1));
      ldsm_x2_t(br, S.ki + drv_off(brow, nt));
      mma16816(acc2[kk & 1], ar, br[0], br[1]);
    }
    float acc[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] = acc2[0][e] + acc2[1][e];
    const int r0 = l >> 2, c0 = nt * 8 + (l & 3) * 2;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = r0 + (e >> 1) * 8, j = c0 + (e & 1);
      if (mat == 0) {
        S.Rf[i][j] = j < i ? S.beta[i] * acc[e] : 0.f;
      } else {
        *reinterpret_cast<float*>(rec + aqk_offset(i, j)) = j <= i ? acc[e] : 0.f;
      }
    }
  }
  chunk_sync();

  // ---- A = (I - R)(I + R^2)(I + R^4)(I + R^8): four dependent levels of
  // register-resident tensor-core products in warp 0, no shared memory or
  // barriers between them; it writes A diag(beta) as bf16 high / low ----
  if (w == 0) {
    const int g = l >> 2, q2 = (l & 3) * 2;
    Mat16 R, P0;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int i = g + 8 * h2, j = 8 * nt + q2;
        const float2 r = *reinterpret_cast<const float2*>(&S.Rf[i][j]);
        R.m[nt][2 * h2] = r.x;
        R.m[nt][2 * h2 + 1] = r.y;
        P0.m[nt][2 * h2] = (i == j ? 1.f : 0.f) - r.x;
        P0.m[nt][2 * h2 + 1] = (i == j + 1 ? 1.f : 0.f) - r.y;
      }
    const OpA Ra = as_a(R);
    const Mat16 R2 = mat_mul(Ra, as_b(Ra), nullptr);                     // R^2
    const OpA R2a = as_a(R2);
    const OpB R2b = as_b(R2a);
    const Mat16 P1 = mat_mul(as_a(P0), R2b, &P0);                        // (I-R)(I+R^2)
    const Mat16 R4 = mat_mul(R2a, R2b, nullptr);                         // R^4
    const OpA R4a = as_a(R4);
    const OpB R4b = as_b(R4a);
    const Mat16 P2 = mat_mul(as_a(P1), R4b, &P1);                        // P1 (I+R^4)
    const Mat16 R8 = mat_mul(R4a, R4b, nullptr);                         // R^8
    const Mat16 A = mat_mul(as_a(P2), as_b(as_a(R8)), &P2);              // P2 (I+R^8)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int j = 8 * nt + q2;
      const float b0 = S.beta[j], b1 = S.beta[j + 1];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int i = g + 8 * h2;
        const float x0 = A.m[nt][2 * h2] * b0, x1 = A.m[nt][2 * h2 + 1] * b1;
        const __nv_bfloat162 hi = __floats2bfloat162_rn(x0, x1);
        const float2 hf = __bfloat1622float2(hi);
        *reinterpret_cast<__nv_bfloat162*>(S.abh + i * AS + j) = hi;
        *reinterpret_cast<__nv_bfloat162*>(S.abl + i * AS + j) =
            __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
      }
    }
  }
  // this chunk's v tile (the older of at most two pending groups)
  if (prefetched)
    asm volatile("cp.async.wait_group 1;" ::: "memory");
  else
    asm volatile("cp.async.wait_group 0;" ::: "memory");
  chunk_sync();

  // ---- W = A diag(beta) Kdec, U = A diag(beta) V (warp w: channels 32w..32w+31) ----
  {
    const int mi = l >> 3, g = l >> 2, q2 = (l & 3) * 2;
    // W [i][c]: A = (A diag beta)_hi [i][j], B = Kdec^T tile [c][j] ([n][k] order)
    uint32_t ah[4];
    ldsm_x4(ah, S.abh + (l & 15) * AS + (l >> 4) * 8);
#pragma unroll
    for (int pair = 0; pair < 2; ++pair) {
      const int n0 = w * 32 + pair * 16;
      uint32_t bk[4];
      ldsm_x4(bk, S.kd + drv_off(n0 + (l & 7) + (mi >> 1) * 8, mi & 1));
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float wacc[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816(wacc, ah, bk[2 * half], bk[2 * half + 1]);
        const int c = n0 + half * 8 + q2;
        *reinterpret_cast<uint32_t*>(rec + b1_offset(16 + g, c)) = pack_bf16(wacc[0], wacc[1]);
        *reinterpret_cast<uint32_t*>(rec + b1_offset(24 + g, c)) = pack_bf16(wacc[2], wacc[3]);
      }
    }
    // U^T [c][i] = V^T (A diag beta)^T: A = V^T from the raw v tile (transposed
    // load), B = (A diag beta) rows [i][j] ([n][k] order), high and low parts;
    // each lane then holds two consecutive tokens of one channel
    uint32_t bh[4], bl[4];
    const int boff = ((l & 7) + (l >> 4) * 8) * AS + ((l >> 3) & 1) * 8;
    ldsm_x4(bh, S.abh + boff);
    ldsm_x4(bl, S.abl + boff);
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const int m0 = w * 32 + mt * 16;
      const int j = (l & 7) + (mi >> 1) * 8;
      uint32_t av[4];
      ldsm_x4_t(av, raw_row(vt, 0, j) + raw_piece(j, (m0 >> 3) + (mi & 1)));
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
