// kda_chunk.cuh -- the per-chunk work of the chunkwise KDA forward pass
// ("You Could Have Come Up with Kimi Delta Attention", sec. 6.1-6.6; gates and
// norms as in "FlashKDA Delta Attention Algorithm", Core Architecture), done
// by one 128-thread group for one (chunk, head) and written as one record
// (layout in kda_common.cuh).  Used by the token-parallel chunk kernel (K1).
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
// them with tf32 MMAs), U and Aqk as fp32, Kend as a bf16 high/low pair.
#pragma once

#include "kda_common.cuh"

namespace kda {

constexpr int TS = 136;  // bf16 row stride of the 16 x 128 tiles (272 B: no ldmatrix conflicts)
constexpr int AS = 24;   // bf16 row stride of the 16 x 16 tiles (48 B)

struct ChunkSmem {
  __nv_bfloat16 q[16 * TS];    // raw q, then Qdec high
  __nv_bfloat16 k[16 * TS];    // raw k, then Kdec high
  __nv_bfloat16 v[16 * TS];    // raw v (exact bf16 operand of U)
  __nv_bfloat16 g[16 * TS];    // raw g_raw, then Qdec low
  __nv_bfloat16 kdl[16 * TS];  // Kdec low
  __nv_bfloat16 kih[16 * TS];  // Kinv high
  __nv_bfloat16 kil[16 * TS];  // Kinv low
  float M[2][16][17];          // Mkk, Mqk
  float mat[4][16][17];        // inverse workspace
  __nv_bfloat16 abh[16 * AS];  // A diag(beta), high
  __nv_bfloat16 abl[16 * AS];  // A diag(beta), low
  float rq[16], rk[16], beta[16];
};

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

// C = P * (I + Q) or P * Q for lower-triangular 16 x 16 P, Q (fp32, smem);
// thread t of 128 writes entries (t / 8, 2 (t % 8) + {0, 1}).
__device__ __forceinline__ void lower_mul(const float (*P)[17], const float (*Q)[17],
                                          float (*Cm)[17], bool plus_identity, int t) {
  const int i = t >> 3, j0 = (t & 7) * 2;
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {
    const int j = j0 + jj;
    float acc = 0.f;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      if (m >= j && m <= i) {
        const float qv = Q[m][j] + ((plus_identity && m == j) ? 1.f : 0.f);
        acc = fmaf(P[i][m], qv, acc);
      }
    }
    Cm[i][j] = (j <= i) ? acc : 0.f;
  }
}

// Barrier over the 128 threads that build records (named barrier 1, so that a
// larger CTA can run other warps beside them).
__device__ __forceinline__ void chunk_sync() { named_bar(1, 128); }

// Build the record of one chunk.  All 128 threads of the group must call it.
// q..g point at token t0, head h of [T, H, 128] bf16 tensors (row stride
// `row_stride` elements); beta_raw points at [t0][h] (stride H).  `rec` is the
// record base (global or shared).  Ends with the group's shared memory free.
__device__ __forceinline__ void build_chunk_record(
    ChunkSmem& S, const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
    const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ g,
    const __nv_bfloat16* __restrict__ beta_raw, int64_t row_stride, int64_t beta_stride, int nc,
    float scale, float lb_log2e, float eps, uint8_t* __restrict__ rec, int t) {
  const int w = t >> 5, l = t & 31;

  // ---- load the four 16 x 128 tiles (rows past nc are zero) ----
  {
    const __nv_bfloat16* src[4] = {q, k, v, g};
    __nv_bfloat16* dst[4] = {S.q, S.k, S.v, S.g};
#pragma unroll
    for (int x = 0; x < 4; ++x) {
#pragma unroll
      for (int rep = 0; rep < 2; ++rep) {
        const int p = t + rep * 128;
        const int row = p >> 4, col = (p & 15) * 8;
        __nv_bfloat16* d = dst[x] + row * TS + col;
        if (row < nc)
          cp_async16(d, src[x] + row * row_stride + col);
        else
          *reinterpret_cast<uint4*>(d) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
  }
  if (t < 16) {
    S.beta[t] = (t < nc) ? sigmoid_fast(__bfloat162float(beta_raw[t * beta_stride])) : 0.f;
  }
  chunk_sync();

  // ---- per-token inverse norms (warp w: tokens 4w .. 4w+3) ----
#pragma unroll
  for (int ii = 0; ii < 4; ++ii) {
    const int i = w * 4 + ii;
    const __nv_bfloat162* qr = reinterpret_cast<const __nv_bfloat162*>(S.q + i * TS + l * 4);
    const __nv_bfloat162* kr = reinterpret_cast<const __nv_bfloat162*>(S.k + i * TS + l * 4);
    float2 q0 = __bfloat1622float2(qr[0]), q1 = __bfloat1622float2(qr[1]);
    float2 k0 = __bfloat1622float2(kr[0]), k1 = __bfloat1622float2(kr[1]);
    float sq = q0.x * q0.x + q0.y * q0.y + q1.x * q1.x + q1.y * q1.y;
    float sk = k0.x * k0.x + k0.y * k0.y + k1.x * k1.x + k1.y * k1.y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
      sk += __shfl_xor_sync(0xffffffffu, sk, o);
    }
    if (l == 0) {
      S.rq[i] = rsqrtf(sq + eps);
      S.rk[i] = rsqrtf(sk + eps);
    }
  }
  chunk_sync();

  // ---- gates, decayed factors (thread t = key channel d) ----
  {
    const int d = t;
    float a[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float gv = __bfloat162float(S.g[i * TS + d]);
      a[i] = (i < nc) ? ex2_approx(lb_log2e * sigmoid_fast(gv)) : 1.f;
    }
    float P[16], Qs[16];
    float p = 1.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      p *= a[i];
      P[i] = p;
    }
    const float dlast = p;
    const float inv_dl = rcp_approx(dlast);
    float sfx = 1.f;
#pragma unroll
    for (int i = 15; i >= 0; --i) {
      Qs[i] = sfx;
      sfx *= a[i];
    }
    uint32_t kh[8], kl[8];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float qv = __bfloat162float(S.q[i * TS + d]) * S.rq[i];
      const float kv = __bfloat162float(S.k[i * TS + d]) * S.rk[i];
      const float Qd = scale * qv * P[i];
      const float Kd = kv * P[i];
      const float Ke = kv * Qs[i];
      const float Ki = Ke * inv_dl;
      *reinterpret_cast<float*>(rec + b1_offset(16 + i, d)) = to_tf32(Qd);
      __nv_bfloat16 hi, lo;
      split_bf16(Qd, hi, lo);
      S.q[i * TS + d] = hi;
      S.g[i * TS + d] = lo;
      split_bf16(Kd, hi, lo);
      S.k[i * TS + d] = hi;
      S.kdl[i * TS + d] = lo;
      split_bf16(Ki, hi, lo);
      S.kih[i * TS + d] = hi;
      S.kil[i * TS + d] = lo;
      split_bf16(Ke, hi, lo);
      const uint32_t hb = __bfloat16_as_ushort(hi), lbits = __bfloat16_as_ushort(lo);
      if (i & 1) {
        kh[i >> 1] |= hb << 16;
        kl[i >> 1] |= lbits << 16;
      } else {
        kh[i >> 1] = hb;
        kl[i >> 1] = lbits;
      }
    }
#pragma unroll
    for (int piece = 0; piece < 2; ++piece) {
      const int off = kend_offset(KDA_KEND_LAYOUT, d, piece * 8);
      *reinterpret_cast<uint4*>(rec + OFF_KH + off) =
          make_uint4(kh[piece * 4], kh[piece * 4 + 1], kh[piece * 4 + 2], kh[piece * 4 + 3]);
      *reinterpret_cast<uint4*>(rec + OFF_KL + off) =
          make_uint4(kl[piece * 4], kl[piece * 4 + 1], kl[piece * 4 + 2], kl[piece * 4 + 3]);
    }
    reinterpret_cast<float*>(rec + OFF_DL)[d] = dlast;
  }
  chunk_sync();

  // ---- Mkk (warps 0,1) and Mqk (warps 2,3), split-bf16 mma.sync ----
  {
    const int mat = w >> 1, nt = w & 1;
    const __nv_bfloat16* Ah = mat ? S.q : S.k;
    const __nv_bfloat16* Al = mat ? S.g : S.kdl;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t ah[4], al[4], bh[2], bl[2];
      const int aoff = (l & 15) * TS + kk * 16 + (l >> 4) * 8;
      const int boff = (nt * 8 + (l & 7)) * TS + kk * 16 + ((l >> 3) & 1) * 8;
      ldsm_x4(ah, Ah + aoff);
      ldsm_x4(al, Al + aoff);
      ldsm_x2(bh, S.kih + boff);
      ldsm_x2(bl, S.kil + boff);
      mma16816(acc, ah, bh[0], bh[1]);
      mma16816(acc, ah, bl[0], bl[1]);
      mma16816(acc, al, bh[0], bh[1]);
    }
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
      S.mat[0][i][j] = r;
      S.mat[1][i][j] = ((i == j) ? 1.f : 0.f) - r;
      reinterpret_cast<float*>(rec + OFF_AQK)[i * 16 + j] = (j <= i) ? S.M[1][i][j] : 0.f;
    }
  }
  chunk_sync();

  // ---- A = (I - R)(I + R^2)(I + R^4)(I + R^8) ----
  lower_mul(S.mat[0], S.mat[0], S.mat[2], false, t);  // R^2
  chunk_sync();
  lower_mul(S.mat[1], S.mat[2], S.mat[3], true, t);   // (I - R)(I + R^2)
  chunk_sync();
  lower_mul(S.mat[2], S.mat[2], S.mat[0], false, t);  // R^4
  chunk_sync();
  lower_mul(S.mat[3], S.mat[0], S.mat[1], true, t);   // ... (I + R^4)
  chunk_sync();
  lower_mul(S.mat[0], S.mat[0], S.mat[2], false, t);  // R^8
  chunk_sync();
  lower_mul(S.mat[1], S.mat[2], S.mat[3], true, t);   // ... (I + R^8) = A
  chunk_sync();

  // ---- A diag(beta), split into bf16 high / low ----
  {
    const int i = t >> 3, j0 = (t & 7) * 2;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int j = j0 + jj;
      __nv_bfloat16 hi, lo;
      split_bf16(S.mat[3][i][j] * S.beta[j], hi, lo);
      S.abh[i * AS + j] = hi;
      S.abl[i * AS + j] = lo;
    }
  }
  chunk_sync();

  // ---- W = A diag(beta) Kdec, U = A diag(beta) V (warp w: channels 32w..32w+31) ----
  {
    uint32_t ah[4], al[4];
    const int aoff = (l & 15) * AS + (l >> 4) * 8;
    ldsm_x4(ah, S.abh + aoff);
    ldsm_x4(al, S.abl + aoff);
#pragma unroll
    for (int pair = 0; pair < 2; ++pair) {
      const int n0 = w * 32 + pair * 16;
      const int boff = ((l & 7) + ((l >> 3) & 1) * 8) * TS + n0 + (l >> 4) * 8;
      uint32_t bkh[4], bkl[4], bv[4];
      ldsm_x4_t(bkh, S.k + boff);
      ldsm_x4_t(bkl, S.kdl + boff);
      ldsm_x4_t(bv, S.v + boff);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float wa[4] = {0.f, 0.f, 0.f, 0.f}, ua[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816(wa, ah, bkh[2 * half], bkh[2 * half + 1]);
        mma16816(wa, ah, bkl[2 * half], bkl[2 * half + 1]);
        mma16816(wa, al, bkh[2 * half], bkh[2 * half + 1]);
        mma16816(ua, ah, bv[2 * half], bv[2 * half + 1]);
        mma16816(ua, al, bv[2 * half], bv[2 * half + 1]);
        const int r0 = l >> 2, c = n0 + half * 8 + (l & 3) * 2;
        *reinterpret_cast<float2*>(rec + b1_offset(r0, c)) =
            make_float2(to_tf32(wa[0]), to_tf32(wa[1]));
        *reinterpret_cast<float2*>(rec + b1_offset(r0 + 8, c)) =
            make_float2(to_tf32(wa[2]), to_tf32(wa[3]));
        float* U = reinterpret_cast<float*>(rec + OFF_U);
        U[c * 16 + r0] = ua[0];
        U[(c + 1) * 16 + r0] = ua[1];
        U[c * 16 + r0 + 8] = ua[2];
        U[(c + 1) * 16 + r0 + 8] = ua[3];
      }
    }
  }
  chunk_sync();
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
