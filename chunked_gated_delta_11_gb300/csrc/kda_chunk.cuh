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
//   q^ = q / sqrt(|q|^2 + eps), k^ likewise
//   Qdec_i = s q^_i P_i, Kdec_i = k^_i P_i, Kend_i = k^_i Q_i, Kinv_i = Kend_i / dlast
//   Mkk = Kdec Kinv^T, Mqk = Qdec Kinv^T              (16 x 16, K = 128)
//   R = strictly-lower(diag(beta) Mkk), Aqk = lower(Mqk)  (rho and chi of sec. 6.3/6.5)
//   A = (I + R)^-1 = (I - R)(I + R^2)(I + R^4)(I + R^8)  (finite Neumann series)
//   W = A diag(beta) Kdec,  U = A diag(beta) V
// Decay factors are prefix/suffix products of per-token retention factors, so
// their range is that of D_{0:i} itself: with lower_bound >= -5 and 16 tokens
// every factor and its inverse stays a normal fp32 number.
//
// Precision: the 16 x 16 and 16 x 128 products run on mma.sync (bf16 in, fp32
// accumulate) with each fp32 operand split into a bf16 high part and a bf16
// remainder (three products per tile), which keeps ~16 mantissa bits; the
// inverse runs in fp32.  W and Qdec are stored as tf32 (the recurrence reads
// them with tf32 MMAs), U as fp32, Kend and Aqk as bf16 high/low pairs.
//
// Raw input tiles (q, k, v, g_raw: 16 rows of 128 bf16) live in shared memory
// wherever the caller puts them (RawTiles), rows of 256 bytes whose 16-byte
// pieces are XOR-swizzled by (row & 7).  The fused kernel places them in the
// W/U area of the record stage they belong to and loads them one chunk ahead;
// W and U are written only after every thread has finished reading them.
#pragma once

#include "kda_common.cuh"

namespace kda {

constexpr int AS = 24;  // bf16 row stride of the 16 x 16 tiles (48 B)

// Per-group scratch.  Derived operand tiles are stored transposed, [128
// channels][16 tokens] bf16 (32 B per channel), 16-byte halves swizzled by
// bit 2 of the channel, so each thread writes its channel with two 16-byte
// stores and ldmatrix reads are conflict-free.
struct ChunkSmem {
  uint8_t kdh[4096];  // Kdec high
  uint8_t kdl[4096];  // Kdec low
  uint8_t kih[4096];  // Kinv high
  uint8_t kil[4096];  // Kinv low
  uint8_t qdh[4096];  // Qdec high
  uint8_t qdl[4096];  // Qdec low
  float M[2][16][17];    // Mkk, Mqk
  // inverse workspace, rows of 20 floats (16-byte aligned, conflict-free):
  // row-major copies (X role) and transposed copies (Y role) of the factors
  float Rr[16][20];   // R, later R^4 (rows)
  float RT[16][20];   // R^T, later (R^8)^T
  float R2r[16][20];  // R^2 (rows)
  float R2T[16][20];  // (R^2)^T
  float R4T[16][20];  // (R^4)^T
  float P0[16][20];   // I - R, later P2 = (I-R)(I+R^2)(I+R^4)
  float P1[16][20];   // P1 = (I-R)(I+R^2), later A = P2 (I+R^8)
  __nv_bfloat16 abh[16 * AS];  // A diag(beta), high
  __nv_bfloat16 abl[16 * AS];  // A diag(beta), low
  float rq[16], rk[16], beta[16];
};

// Where the four raw tiles live: rows 0-7 of tile x at lo[x], rows 8-15 at hi[x].
struct RawTiles {
  uint8_t* lo[4];
  uint8_t* hi[4];
};
enum { RAW_Q = 0, RAW_K = 1, RAW_V = 2, RAW_G = 3 };

__device__ __forceinline__ uint8_t* raw_row(const RawTiles& R, int x, int i) {
  return (i < 8 ? R.lo[x] : R.hi[x]) + (i & 7) * 256;
}
// byte offset of 16-byte piece c of raw row i
__device__ __forceinline__ int raw_piece(int i, int c) { return (c ^ (i & 7)) << 4; }
// byte offset of (channel d, token-half p) in a derived tile
__device__ __forceinline__ int drv_off(int d, int p) { return d * 32 + ((p ^ ((d >> 2) & 1)) << 4); }

// Raw tiles placed in the W/U area of a record (the fused kernel): U^T holds
// q and k; the W rows (first 2 KB of each 4 KB block of [W ; Qdec]) hold v, g.
__device__ __forceinline__ RawTiles raw_tiles_in_record(uint8_t* rec) {
  RawTiles R;
  R.lo[RAW_Q] = rec + OFF_U;
  R.hi[RAW_Q] = rec + OFF_U + 2048;
  R.lo[RAW_K] = rec + OFF_U + 4096;
  R.hi[RAW_K] = rec + OFF_U + 6144;
  R.lo[RAW_V] = rec + OFF_B1;
  R.hi[RAW_V] = rec + OFF_B1 + 4096;
  R.lo[RAW_G] = rec + OFF_B1 + 8192;
  R.hi[RAW_G] = rec + OFF_B1 + 12288;
  return R;
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

__device__ __forceinline__ float bf16_at(const uint8_t* p) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
}

// Barrier over the 128 threads that build records (named barrier 1, so that a
// larger CTA can run other warps beside them).
__device__ __forceinline__ void chunk_sync() { named_bar(1, 128); }

// Issue the loads of one chunk's four raw tiles (rows past nc are zeroed) as
// one cp.async group.  q..g point at token t0, head h (row stride
// `row_stride` elements).
__device__ __forceinline__ void issue_raw_loads(const RawTiles& R,
                                                const __nv_bfloat16* __restrict__ q,
                                                const __nv_bfloat16* __restrict__ k,
                                                const __nv_bfloat16* __restrict__ v,
                                                const __nv_bfloat16* __restrict__ g,
                                                int64_t row_stride, int nc, int t) {
  const __nv_bfloat16* src[4] = {q, k, v, g};
#pragma unroll
  for (int x = 0; x < 4; ++x) {
#pragma unroll
    for (int rep = 0; rep < 2; ++rep) {
      const int p = t + rep * 128;
      const int row = p >> 4, c = p & 15;
      uint8_t* d = raw_row(R, x, row) + raw_piece(row, c);
      if (row < nc)
        cp_async16(d, src[x] + row * row_stride + c * 8);
      else
        *reinterpret_cast<uint4*>(d) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Order of the 136 lower-triangle entries (i >= j) by decreasing i - j, so that
// the threads of one warp get similar loop lengths in the triangular products.
struct EntryTable {
  uint8_t ij[136];
};
__host__ __device__ constexpr EntryTable make_entry_table() {
  EntryTable t{};
  int e = 0;
  for (int dl = 15; dl >= 0; --dl)
    for (int j = 0; j + dl < 16; ++j) t.ij[e++] = static_cast<uint8_t>(((j + dl) << 4) | j);
  return t;
}
__constant__ EntryTable kEntries = make_entry_table();

// Entry (i, j), i >= j, of C = B + X Y for 16 x 16 lower-triangular X, Y whose
// never-written triangles hold zeros: a dense 16-term dot product of row i of
// X with column j of Y (read as row j of Y^T), all loads issued up front.
// Writes C[i][j] and, if CT, CT[j][i].
__device__ __forceinline__ void tri_entry(const float (*X)[20], const float (*YT)[20],
                                          const float (*B)[20], float (*Cm)[20], float (*CT)[20],
                                          int i, int j) {
  const float4* xr = reinterpret_cast<const float4*>(X[i]);
  const float4* yr = reinterpret_cast<const float4*>(YT[j]);
  float4 x[4], y[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    x[q] = xr[q];
    y[q] = yr[q];
  }
  float a0 = B ? B[i][j] : 0.f, a1 = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    a0 = fmaf(x[q].x, y[q].x, a0);
    a1 = fmaf(x[q].y, y[q].y, a1);
    a0 = fmaf(x[q].z, y[q].z, a0);
    a1 = fmaf(x[q].w, y[q].w, a1);
  }
  const float c = a0 + a1;
  Cm[i][j] = c;
  if (CT) CT[j][i] = c;
}
// Thread t of 128 computes entry e1 = kEntries[t] and, on lanes 0 and 1 of
// each warp, e2 = kEntries[128 + 2 (t / 32) + lane] (packed (i << 4) | j,
// loaded once per chunk), so the eight extra entries are spread over the warps.
__device__ __forceinline__ bool has_second_entry(int t) { return (t & 31) < 2; }
__device__ __forceinline__ int second_entry_index(int t) { return 128 + (t >> 5) * 2 + (t & 31); }
__device__ __forceinline__ void tri_product(const float (*X)[20], const float (*YT)[20],
                                            const float (*B)[20], float (*Cm)[20],
                                            float (*CT)[20], int e1, int e2, int t) {
  tri_entry(X, YT, B, Cm, CT, e1 >> 4, e1 & 15);
  if (has_second_entry(t)) tri_entry(X, YT, B, Cm, CT, e2 >> 4, e2 & 15);
}

// Zero the inverse workspace once (its unwritten triangles must stay zero).
__device__ __forceinline__ void clear_inverse_workspace(ChunkSmem& S, int t) {
  float* p = &S.Rr[0][0];
  const int n = static_cast<int>(7 * 16 * 20);
  for (int e = t; e < n; e += 128) p[e] = 0.f;
}

// Build the record of one chunk from raw tiles already issued with
// issue_raw_loads (this call waits for them).  All 128 threads of the group
// must call it.  beta_raw_bits: thread t < 16 holds the bf16 bits of token t's
// beta_raw (any value for t >= nc).  `rec` is the record base (global or
// shared).  `may_write()` runs on all threads before the first write to the
// record and returns, uniformly, whether to go on (the fused kernel waits there
// until the previous record in this stage is consumed); on false nothing is
// written.  `after_d` runs on all threads in the middle of the build (the
// fused kernel issues the next chunk's loads there).  Returns may_write().
template <class MayWrite, class Hook>
__device__ __forceinline__ bool build_chunk_record(ChunkSmem& S, const RawTiles& R,
                                                   uint32_t beta_raw_bits, int nc, float scale,
                                                   float lb_log2e, float eps, uint8_t* rec,
                                                   int t, MayWrite&& may_write, Hook&& after_d) {
  const int w = t >> 5, l = t & 31;
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  if (t < 16) {
    const float br = __bfloat162float(__ushort_as_bfloat16(static_cast<unsigned short>(beta_raw_bits)));
    S.beta[t] = (t < nc) ? sigmoid_fast(br) : 0.f;
  }
  if (!may_write()) return false;  // includes a barrier of the 128 threads

  // ---- per-token inverse norms (warp w: tokens 4w .. 4w+3), all eight sums
  // reduced together so the shuffle latencies overlap ----
  {
    float sq[4], sk[4];
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
      const int i = w * 4 + ii;
      const int off = raw_piece(i, l >> 1) + (l & 1) * 8;
      const uint2 qv = *reinterpret_cast<const uint2*>(raw_row(R, RAW_Q, i) + off);
      const uint2 kv = *reinterpret_cast<const uint2*>(raw_row(R, RAW_K, i) + off);
      const float2 q0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qv.x));
      const float2 q1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qv.y));
      const float2 k0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kv.x));
      const float2 k1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&kv.y));
      sq[ii] = q0.x * q0.x + q0.y * q0.y + q1.x * q1.x + q1.y * q1.y;
      sk[ii] = k0.x * k0.x + k0.y * k0.y + k1.x * k1.x + k1.y * k1.y;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int ii = 0; ii < 4; ++ii) {
        sq[ii] += __shfl_xor_sync(0xffffffffu, sq[ii], o);
        sk[ii] += __shfl_xor_sync(0xffffffffu, sk[ii], o);
      }
    }
    if (l < 4) {
      // the read scale is folded into the query norm: rq = scale / |q|
      S.rq[w * 4 + l] =
          scale * rsqrtf((l == 0 ? sq[0] : l == 1 ? sq[1] : l == 2 ? sq[2] : sq[3]) + eps);
      S.rk[w * 4 + l] = rsqrtf((l == 0 ? sk[0] : l == 1 ? sk[1] : l == 2 ? sk[2] : sk[3]) + eps);
    }
  }
  chunk_sync();

  // ---- gates, decayed factors (thread t = key channel d) ----
  // forward pass: prefix products P_i -> Qdec, Kdec; backward pass: suffix
  // products Q_i -> Kend, Kinv.  Eight tokens are packed and stored at a time.
  {
    const int d = t;
    const int dp = d >> 3, db = (d & 7) * 2;
    float a[16];
    // a = 2^(lb log2e sigma(x)), sigma(x) = 1/2 + tanh(x/2)/2
    const float hl = 0.5f * lb_log2e;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float gv = bf16_at(raw_row(R, RAW_G, i) + raw_piece(i, dp) + db);
      a[i] = (i < nc) ? ex2_approx(fmaf(hl, tanh_approx(0.5f * gv), hl)) : 1.f;
    }
    float p = 1.f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t qh[4], ql[4], kh[4], kl[4];
#pragma unroll
      for (int i2 = 0; i2 < 4; ++i2) {
        const int i = half * 8 + i2 * 2;  // tokens i, i + 1 as one packed pair
        const int o0 = raw_piece(i, dp) + db, o1 = raw_piece(i + 1, dp) + db;
        float2 P;
        p *= a[i];
        P.x = p;
        p *= a[i + 1];
        P.y = p;
        const float2 qr = make_float2(bf16_at(raw_row(R, RAW_Q, i) + o0),
                                      bf16_at(raw_row(R, RAW_Q, i + 1) + o1));
        const float2 kr = make_float2(bf16_at(raw_row(R, RAW_K, i) + o0),
                                      bf16_at(raw_row(R, RAW_K, i + 1) + o1));
        const float2 Qd = mul2(mul2(qr, make_float2(S.rq[i], S.rq[i + 1])), P);
        const float2 Kd = mul2(mul2(kr, make_float2(S.rk[i], S.rk[i + 1])), P);
        *reinterpret_cast<float*>(rec + b1_offset(16 + i, d)) = to_tf32(Qd.x);
        *reinterpret_cast<float*>(rec + b1_offset(17 + i, d)) = to_tf32(Qd.y);
        split_pair2(Qd.x, Qd.y, qh[i2], ql[i2]);
        split_pair2(Kd.x, Kd.y, kh[i2], kl[i2]);
      }
      const int o = drv_off(d, half);
      *reinterpret_cast<uint4*>(S.qdh + o) = make_uint4(qh[0], qh[1], qh[2], qh[3]);
      *reinterpret_cast<uint4*>(S.qdl + o) = make_uint4(ql[0], ql[1], ql[2], ql[3]);
      *reinterpret_cast<uint4*>(S.kdh + o) = make_uint4(kh[0], kh[1], kh[2], kh[3]);
      *reinterpret_cast<uint4*>(S.kdl + o) = make_uint4(kl[0], kl[1], kl[2], kl[3]);
    }
    const float dlast = p;
    const float inv_dl = rcp_approx(dlast);
    reinterpret_cast<float*>(rec + OFF_DL)[d] = dlast;
    float sfx = 1.f;  // prod_{m > i} a_m while token i is processed
#pragma unroll
    for (int half = 1; half >= 0; --half) {
      uint32_t eh[4], el[4], ih[4], il[4];
#pragma unroll
      for (int i2 = 3; i2 >= 0; --i2) {
        const int i = half * 8 + i2 * 2;  // tokens i, i + 1 as one packed pair
        float2 Q;
        Q.y = sfx;
        sfx *= a[i + 1];
        Q.x = sfx;
        sfx *= a[i];
        const float2 kr =
            make_float2(bf16_at(raw_row(R, RAW_K, i) + raw_piece(i, dp) + db),
                        bf16_at(raw_row(R, RAW_K, i + 1) + raw_piece(i + 1, dp) + db));
        const float2 Ke = mul2(mul2(kr, make_float2(S.rk[i], S.rk[i + 1])), Q);
        const float2 Ki = mul2(Ke, make_float2(inv_dl, inv_dl));
        split_pair2(Ke.x, Ke.y, eh[i2], el[i2]);
        split_pair2(Ki.x, Ki.y, ih[i2], il[i2]);
      }
      const int o = drv_off(d, half);
      *reinterpret_cast<uint4*>(S.kih + o) = make_uint4(ih[0], ih[1], ih[2], ih[3]);
      *reinterpret_cast<uint4*>(S.kil + o) = make_uint4(il[0], il[1], il[2], il[3]);
      const int ko = kend_offset(KDA_KEND_LAYOUT, d, half * 8);
      *reinterpret_cast<uint4*>(rec + OFF_KH + ko) = make_uint4(eh[0], eh[1], eh[2], eh[3]);
      *reinterpret_cast<uint4*>(rec + OFF_KL + ko) = make_uint4(el[0], el[1], el[2], el[3]);
    }
  }
  chunk_sync();

  // ---- Mkk (warps 0,1) and Mqk (warps 2,3), split-bf16 mma.sync over 8 k-steps ----
  {
    const int mat = w >> 1, nt = w & 1;
    const uint8_t* Ah = mat ? S.qdh : S.kdh;
    const uint8_t* Al = mat ? S.qdl : S.kdl;
    // three independent accumulator chains (high*high, high*low, low*high)
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f},
          acc2[4] = {0.f, 0.f, 0.f, 0.f};
    const int mi = l >> 3;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int arow = kk * 16 + (l & 7) + (mi >> 1) * 8;   // channel
      const int aoff = drv_off(arow, mi & 1);                // token half
      const int brow = kk * 16 + (l & 7) + ((l >> 3) & 1) * 8;
      const int boff = drv_off(brow, nt);
      uint32_t ah[4], al[4], bh[2], bl[2];
      ldsm_x4_t(ah, Ah + aoff);
      ldsm_x4_t(al, Al + aoff);
      ldsm_x2_t(bh, S.kih + boff);
      ldsm_x2_t(bl, S.kil + boff);
      mma16816(acc, ah, bh[0], bh[1]);
      mma16816(acc1, ah, bl[0], bl[1]);
      mma16816(acc2, al, bh[0], bh[1]);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] += acc1[e] + acc2[e];
    const int r0 = l >> 2, c0 = nt * 8 + (l & 3) * 2;
    S.M[mat][r0][c0] = acc[0];
    S.M[mat][r0][c0 + 1] = acc[1];
    S.M[mat][r0 + 8][c0] = acc[2];
    S.M[mat][r0 + 8][c0 + 1] = acc[3];
  }
  chunk_sync();

  // ---- R, I - R, Aqk ----
  {
    const int i = t >> 3, j0 = (t & 7) * 2;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int j = j0 + jj;
      const float r = (j < i) ? S.beta[i] * S.M[0][i][j] : 0.f;
      S.Rr[i][j] = r;
      S.RT[j][i] = r;
      S.P0[i][j] = ((i == j) ? 1.f : 0.f) - r;
      __nv_bfloat16 ah, al;
      split_bf16((j <= i) ? S.M[1][i][j] : 0.f, ah, al);
      *reinterpret_cast<__nv_bfloat16*>(rec + OFF_AQK + aqk_offset(i, j)) = ah;
      *reinterpret_cast<__nv_bfloat16*>(rec + OFF_AQK + 512 + aqk_offset(i, j)) = al;
    }
  }
  after_d();
  chunk_sync();

  // ---- A = (I - R)(I + R^2)(I + R^4)(I + R^8) in four dependent steps ----
  {
    const int e1 = kEntries.ij[t], e2 = has_second_entry(t) ? kEntries.ij[second_entry_index(t)] : 0;
    tri_product(S.Rr, S.RT, nullptr, S.R2r, S.R2T, e1, e2, t);   // R^2
    chunk_sync();
    tri_product(S.P0, S.R2T, S.P0, S.P1, nullptr, e1, e2, t);    // P1 = (I-R)(I+R^2)
    tri_product(S.R2r, S.R2T, nullptr, S.Rr, S.R4T, e1, e2, t);  // R^4 (rows into Rr)
    chunk_sync();
    tri_product(S.P1, S.R4T, S.P1, S.P0, nullptr, e1, e2, t);    // P2 = P1 (I+R^4)
    tri_product(S.Rr, S.R4T, nullptr, S.R2r, S.RT, e1, e2, t);   // R^8 (only R8^T kept)
    chunk_sync();
    tri_product(S.P0, S.RT, S.P0, S.P1, nullptr, e1, e2, t);     // A = P2 (I+R^8)
    chunk_sync();
  }

  // ---- A diag(beta), split into bf16 high / low ----
  {
    const int i = t >> 3, j0 = (t & 7) * 2;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int j = j0 + jj;
      __nv_bfloat16 hi, lo;
      split_bf16((j <= i) ? S.P1[i][j] * S.beta[j] : 0.f, hi, lo);
      S.abh[i * AS + j] = hi;
      S.abl[i * AS + j] = lo;
    }
  }
  chunk_sync();

  // ---- W = A diag(beta) Kdec, U = A diag(beta) V (warp w: channels 32w..32w+31) ----
  float wa[4][4], ua[4][4];
  {
    uint32_t ah[4], al[4];
    const int aoff = (l & 15) * AS + (l >> 4) * 8;
    ldsm_x4(ah, S.abh + aoff);
    ldsm_x4(al, S.abl + aoff);
    const int mi = l >> 3;
#pragma unroll
    for (int pair = 0; pair < 2; ++pair) {
      const int n0 = w * 32 + pair * 16;
      // Kdec^T tile [d][j] is B in [n][k] order: plain ldmatrix
      const int koff = drv_off(n0 + (l & 7) + (mi >> 1) * 8, mi & 1);
      // raw V [j][d] is B in [k][n] order: transposed ldmatrix
      const int vrow = (l & 7) + (mi & 1) * 8;
      const uint8_t* vaddr = raw_row(R, RAW_V, vrow) + raw_piece(vrow, (n0 >> 3) + (mi >> 1));
      uint32_t bkh[4], bkl[4], bv[4];
      ldsm_x4(bkh, S.kdh + koff);
      ldsm_x4(bkl, S.kdl + koff);
      ldsm_x4_t(bv, vaddr);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float* W4 = wa[pair * 2 + half];
        float* U4 = ua[pair * 2 + half];
        float wacc[4] = {0.f, 0.f, 0.f, 0.f}, uacc[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816(wacc, ah, bkh[2 * half], bkh[2 * half + 1]);
        mma16816(wacc, ah, bkl[2 * half], bkl[2 * half + 1]);
        mma16816(wacc, al, bkh[2 * half], bkh[2 * half + 1]);
        mma16816(uacc, ah, bv[2 * half], bv[2 * half + 1]);
        mma16816(uacc, al, bv[2 * half], bv[2 * half + 1]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          W4[e] = wacc[e];
          U4[e] = uacc[e];
        }
      }
    }
  }
  chunk_sync();  // every read of the raw tiles is done: W and U may overwrite them
  {
    const int r0 = l >> 2;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int c = w * 32 + nt * 8 + (l & 3) * 2;
      *reinterpret_cast<float2*>(rec + b1_offset(r0, c)) =
          make_float2(to_tf32(wa[nt][0]), to_tf32(wa[nt][1]));
      *reinterpret_cast<float2*>(rec + b1_offset(r0 + 8, c)) =
          make_float2(to_tf32(wa[nt][2]), to_tf32(wa[nt][3]));
      float* U = reinterpret_cast<float*>(rec + OFF_U);
      U[c * 16 + r0] = ua[nt][0];
      U[(c + 1) * 16 + r0] = ua[nt][1];
      U[c * 16 + r0 + 8] = ua[nt][2];
      U[(c + 1) * 16 + r0 + 8] = ua[nt][3];
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
