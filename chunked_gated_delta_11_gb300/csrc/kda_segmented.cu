// kda_segmented.cu -- the forward pass with every sequence cut into P pieces
// that run at the same time, for few long sequences whose (sequence, head)
// units alone would leave most SMs idle.
//
// Each token step of the recurrence is an affine map of the state, with a
// diagonal-plus-low-rank linear part ("You Could Have Come Up with Kimi Delta
// Attention", sec. 4.1; rows = value index):
//   S_t = S_{t-1} A_t + B_t,   A_t = Diag(alpha_t) (I - beta_t k_t k_t^T),
//                              B_t = beta_t v_t k_t^T,
// so a segment of tokens maps its starting state S_0 to S_0 M + X, where
// M = A_1 ... A_n and X is the segment's state from a zero start.  Inside the
// segment S_t = S_0 M_t + X_t, hence o_t = S_t (s q_t) = X_t (s q_t) + S_0 y_t
// with y_t = M_t (s q_t).  The scan of these maps is the exchange step that a
// context-parallel split of a long sequence needs; here all pieces run on one
// GPU:
//   1. seg_plan_kernel      segment boundaries (chunk-aligned) and the fix-up
//                           work list;
//   2. fused_kernel         one launch with two CTAs per (segment, head)
//                           (SegArgs in kda_common.cuh): X role (the segment
//                           from zero, or from the sequence's initial state for
//                           its first segment) -> out, X; M role (v = 0 from
//                           the identity: its state is M_t, its output y_t);
//   3. affine_scan_kernel   per (sequence, head): S_0 of every later segment
//                           and the final state (fp32 or bf16), S <- S M_j + X_j
//                           in fp32;
//   4. seg_fixup_kernel     out_t += S_0 y_t for the tokens of later segments
//                           (bf16 tensor-core MMA, fp32 accumulation).
#include "kda_chunk.cuh"

namespace kda {

constexpr int SG_BLOCK = 64;   // tokens per fix-up work item (4 warps x 16)
constexpr int SG_ROW = 272;    // padded byte stride of a 128 x bf16 row in shared memory

// Segment j of sequence n covers chunks [nch j / P, nch (j + 1) / P) of the
// sequence's nch chunks (floor division), so every boundary but the last is a
// chunk boundary and segments differ in length by at most one chunk (empty
// segments when nch < P).  cu_seg [N P + 1] holds the boundaries as a packed
// cu_seqlens over the same token array; blk [N P + 1] the exclusive prefix
// over segments of their fix-up work items (first segments have none).
// One CTA.
__global__ void seg_plan_kernel(const int32_t* __restrict__ cu, int64_t T_total, int N, int P,
                                int32_t* __restrict__ cu_seg, int32_t* __restrict__ blk) {
  grid_dep_launch();  // the fused launch may be scheduled now; it waits for this kernel
  for (int n = threadIdx.x; n < N; n += blockDim.x) {
    int64_t bos, eos;
    seq_bounds(cu, T_total, N, n, bos, eos);
    const int64_t nch = (eos - bos + kChunk - 1) / kChunk;
    for (int j = 0; j < P; ++j) {
      const int64_t b = bos + kChunk * ((nch * j) / P);
      int64_t e = bos + kChunk * ((nch * (j + 1)) / P);
      if (e > eos) e = eos;
      cu_seg[static_cast<int64_t>(n) * P + j] = static_cast<int32_t>(b);
      blk[static_cast<int64_t>(n) * P + j + 1] =
          j == 0 ? 0 : static_cast<int32_t>((e - b + SG_BLOCK - 1) / SG_BLOCK);
    }
    if (n == N - 1) cu_seg[static_cast<int64_t>(N) * P] = static_cast<int32_t>(eos);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    blk[0] = 0;
    const int64_t ns = static_cast<int64_t>(N) * P;
    for (int64_t s = 0; s < ns; ++s) blk[s + 1] += blk[s];
  }
}

// ---------------------------------------------------------------------------
// The scan.  Rows of S M + X depend only on the same rows of S, so each
// (sequence, head) is split over 128 / ROWS CTAs of ROWS value rows (the
// launcher takes the smallest ROWS whose grid fits one CTA per SM: few units,
// more CTAs per unit and shorter steps).  The steps are serial and short, so
// the kernel is bound by latency; its warps are arranged so that M_j is read
// from shared memory once per CTA and step while 16 warps cover each other's
// latency:
//   - RW row warps own RA = 4 rows each (8 when ROWS >= 64) and, lane l, key
//     columns 4 l .. 4 l + 3;
//   - KS = 16 / RW warps share each row block, warp ks taking the
//     contraction indices ks 128 / KS .. (ks + 1) 128 / KS - 1; the KS - 1
//     partial sums go through shared memory to the ks = 0 warp at the end of
//     the step.
// The rows are kept transposed in shared memory (St[k][v], row stride ROWS +
// 4 floats) so that a thread's values of one key column are contiguous.
// Everything a step reads arrives during the step before: M_{j+1} by cp.async
// into the second of two buffers, and the ks = 0 threads' elements of X_{j+1}
// into registers.  xs holds the X role's final states [N P, H, V, K]; for
// every later segment j its entry is replaced by that segment's starting
// state S_0 (read by the fix-up).
// ---------------------------------------------------------------------------
template <int ROWS>
struct ScanShape {
  static constexpr int RA = ROWS >= 64 ? 8 : 4;  // rows per thread
  static constexpr int RW = ROWS / RA;            // row warps
  static constexpr int KS = 16 / RW;              // warps per row block
  static constexpr int NT = 32 * RW * KS;         // 512 threads
  static constexpr int LD = ROWS + 4;             // St row stride (floats)
  // floats: St, two M buffers, the KS - 1 partial tiles
  static constexpr int SMEM = (kDim * LD + 2 * kDim * kDim + (KS - 1) * ROWS * kDim) * 4;
};

template <int NT>
__device__ __forceinline__ void sc_stage_m(float* dst, const float* src, int t) {
#pragma unroll 4
  for (int i = t; i < kDim * kDim / 4; i += NT)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst + 4 * i)),
                 "l"(src + 4 * i)
                 : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int ROWS>
__global__ void __launch_bounds__(ScanShape<ROWS>::NT)
affine_scan_kernel(float* __restrict__ xs, const float* __restrict__ ms, int N, int P, int H,
                   void* __restrict__ final_state, bool final_bf16,
                   __nv_bfloat16* __restrict__ s0_bf16) {
  grid_dep_wait();  // the fused launch's states
  grid_dep_launch();
  using SS = ScanShape<ROWS>;
  constexpr int NT = SS::NT, RA = SS::RA, RW = SS::RW, KS = SS::KS, LD = SS::LD;
  constexpr int SPLIT = kDim / ROWS, KC = kDim / KS;
  extern __shared__ float4 sc_smem4[];
  float* St = reinterpret_cast<float*>(sc_smem4);
  float* Mbuf = St + kDim * LD;          // two [128][128] buffers
  float* Red = Mbuf + 2 * kDim * kDim;   // [KS - 1][ROWS][128] partial sums
  const int unit = blockIdx.x / SPLIT, part = blockIdx.x - unit * SPLIT;
  const int n = unit / H, h = unit - (unit / H) * H;
  const int t = threadIdx.x, wi = t >> 5;
  const int rw = wi % RW, ks = wi / RW;
  const int rv = rw * RA, ck = (t & 31) * 4;  // local value rows rv.., key columns ck..
  const int k0 = ks * KC;                     // this warp's contraction indices k0..
  const int64_t row0 = static_cast<int64_t>(part) * ROWS * kDim;  // first row of the part
  auto base = [&](int64_t s) { return (s * H + h) * kDim * kDim; };
  const int64_t s0 = static_cast<int64_t>(n) * P;
  // this thread's elements of X_j (rows rv.., columns ck..; ks = 0 only)
  auto load_x = [&](float4 (&x)[RA], int j) {
    const float* xj = xs + base(s0 + j) + row0;
#pragma unroll
    for (int a = 0; a < RA; ++a) x[a] = __ldcg(reinterpret_cast<const float4*>(xj + (rv + a) * kDim + ck));
  };
  float4 xn[RA];
  if (P > 1) {
    sc_stage_m<NT>(Mbuf, ms + base(s0 + 1), t);
    if (ks == 0) load_x(xn, 1);
  }
  {
    const float* x0 = xs + base(s0) + row0;
    for (int i = t; i < ROWS * kDim; i += NT) St[(i & 127) * LD + (i >> 7)] = x0[i];
  }
  for (int j = 1; j < P; ++j) {
    const float* Ms = Mbuf + ((j - 1) & 1) * kDim * kDim;
    float* xj = xs + base(s0 + j) + row0;
    float acc[RA][4];
#pragma unroll
    for (int a = 0; a < RA; ++a) {
      if (ks == 0) {
        acc[a][0] = xn[a].x; acc[a][1] = xn[a].y; acc[a][2] = xn[a].z; acc[a][3] = xn[a].w;
      } else {
        acc[a][0] = acc[a][1] = acc[a][2] = acc[a][3] = 0.f;
      }
    }
    // M_j has arrived; its other buffer was last read in step j - 1, which
    // every thread has finished (barrier at the end of the previous step)
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    if (j + 1 < P) {
      sc_stage_m<NT>(Mbuf + (j & 1) * kDim * kDim, ms + base(s0 + j + 1), t);
      if (ks == 0) load_x(xn, j + 1);  // used by the next step; its latency overlaps this one
    }
#pragma unroll 4
    for (int kk = k0; kk < k0 + KC; ++kk) {
      float sv[RA];
#pragma unroll
      for (int a = 0; a < RA; ++a) sv[a] = St[kk * LD + rv + a];
      const float4 ma = *reinterpret_cast<const float4*>(Ms + kk * kDim + ck);
      const float mv[4] = {ma.x, ma.y, ma.z, ma.w};
#pragma unroll
      for (int a = 0; a < RA; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(sv[a], mv[b], acc[a][b]);
    }
    if (ks == 0) {
      // segment j starts from the S before this step (X_j was read a step
      // ago); the fix-up's bf16 copy of it, if asked for, beside it
      __nv_bfloat16* bj = s0_bf16 ? s0_bf16 + base(s0 + j) + row0 : nullptr;
#pragma unroll
      for (int a = 0; a < RA; ++a) {
        const float4 sj = make_float4(St[ck * LD + rv + a], St[(ck + 1) * LD + rv + a],
                                      St[(ck + 2) * LD + rv + a], St[(ck + 3) * LD + rv + a]);
        *reinterpret_cast<float4*>(xj + (rv + a) * kDim + ck) = sj;
        if (bj)
          *reinterpret_cast<uint2*>(bj + (rv + a) * kDim + ck) =
              make_uint2(pack_bf16(sj.x, sj.y), pack_bf16(sj.z, sj.w));
      }
    } else {
      float* r = Red + (ks - 1) * ROWS * kDim;
#pragma unroll
      for (int a = 0; a < RA; ++a)
        *reinterpret_cast<float4*>(r + (rv + a) * kDim + ck) =
            make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
    }
    __syncthreads();  // every read of St and of this M buffer is done; partials written
    if (ks == 0) {
#pragma unroll
      for (int q = 1; q < KS; ++q) {
        const float* r = Red + (q - 1) * ROWS * kDim;
#pragma unroll
        for (int a = 0; a < RA; ++a) {
          const float4 p4 = *reinterpret_cast<const float4*>(r + (rv + a) * kDim + ck);
          acc[a][0] += p4.x; acc[a][1] += p4.y; acc[a][2] += p4.z; acc[a][3] += p4.w;
        }
      }
#pragma unroll
      for (int a = 0; a < RA; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) St[(ck + b) * LD + rv + a] = acc[a][b];
    }
  }
  __syncthreads();
  if (final_state) {
    const int64_t f0 = (static_cast<int64_t>(n) * H + h) * kDim * kDim + row0;
    if (final_bf16) {
      __nv_bfloat16* f = static_cast<__nv_bfloat16*>(final_state) + f0;
      for (int i = t; i < ROWS * kDim; i += NT)
        f[i] = __float2bfloat16_rn(St[(i & 127) * LD + (i >> 7)]);
    } else {
      float* f = static_cast<float*>(final_state) + f0;
      for (int i = t; i < ROWS * kDim; i += NT) f[i] = St[(i & 127) * LD + (i >> 7)];
    }
  }
}

// ---------------------------------------------------------------------------
// The fix-up: out[t, h, :] += S_0 y[t, h, :] for the tokens of every later
// segment.  Work item = (head, 64-token block of one segment), numbered head
// major so that a CTA's contiguous range of items mostly shares one (segment,
// head) and converts its S_0 once: S_0 (fp32) -> bf16 [v][k] in shared memory,
// read as B fragments (ldmatrix).  The item's rows of y and out arrive by
// cp.async into padded shared tiles (coalesced 16-byte pieces; y rows past the
// segment end are zero-filled), y is read as A fragments (ldmatrix), the sums
// are added to the out tile in the accumulator layout, and the tile goes back
// in 16-byte pieces.  Warp w: tokens 16 w .. +15 of the block, 16 column tiles
// of 8 values, K = 128.
// ---------------------------------------------------------------------------
constexpr int FX_THREADS = 128;
constexpr int FX_S_BYTES = kDim * SG_ROW;        // S_0, bf16 [128][128], padded rows
constexpr int FX_T_BYTES = SG_BLOCK * SG_ROW;    // one [64][128] bf16 tile, padded rows
constexpr int FX_SMEM = FX_S_BYTES + 2 * FX_T_BYTES;

__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, bool pred) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(pred ? 16 : 0)
               : "memory");
}

__global__ void __launch_bounds__(FX_THREADS, 3)
seg_fixup_kernel(const int32_t* __restrict__ cu_seg, const int32_t* __restrict__ blk, int Nseg,
                 int H, const float* __restrict__ sstart, const __nv_bfloat16* __restrict__ sstart16,
                 const __nv_bfloat16* __restrict__ y, __nv_bfloat16* __restrict__ out) {
  grid_dep_wait();  // the scan's starting states
  extern __shared__ __align__(16) uint8_t fx_smem[];
  uint8_t* sb = fx_smem;
  uint8_t* yt = fx_smem + FX_S_BYTES;
  uint8_t* ot = yt + FX_T_BYTES;
  const int t = threadIdx.x, w = t >> 5, l = t & 31;
  const int64_t nblk = __ldg(blk + Nseg);
  const int64_t total = nblk * H;
  const int64_t per = (total + gridDim.x - 1) / gridDim.x;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * per;
  const int64_t i1 = (i0 + per < total) ? i0 + per : total;
  const int64_t row_stride = static_cast<int64_t>(H) * kDim;
  int cur_s = -1, cur_h = -1;
  for (int64_t it = i0; it < i1; ++it) {
    const int h = static_cast<int>(it / nblk);
    const int gb = static_cast<int>(it - static_cast<int64_t>(h) * nblk);
    // the segment s with blk[s] <= gb < blk[s + 1]
    int lo = 0, hi = Nseg - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(blk + mid) <= gb)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int s = lo;
    const int64_t t0 = __ldg(cu_seg + s) + static_cast<int64_t>(gb - __ldg(blk + s)) * SG_BLOCK;
    const int64_t rem = __ldg(cu_seg + s + 1) - t0;
    const int nt = static_cast<int>(rem < SG_BLOCK ? rem : SG_BLOCK);
    __syncthreads();  // the previous item's tiles (and S_0) are no longer read
    // this item's y and out rows: 16 pieces of 16 bytes per row
    const __nv_bfloat16* ybase = y + t0 * row_stride + static_cast<int64_t>(h) * kDim;
    __nv_bfloat16* obase = out + t0 * row_stride + static_cast<int64_t>(h) * kDim;
#pragma unroll
    for (int k = 0; k < SG_BLOCK * 16 / FX_THREADS; ++k) {
      const int i = t + k * FX_THREADS, r = i >> 4, c = i & 15;
      const bool in = r < nt;
      const int64_t go = (in ? r : 0) * row_stride + c * 8;
      cp_async16_zfill(yt + r * SG_ROW + c * 16, ybase + go, in);
      cp_async16_zfill(ot + r * SG_ROW + c * 16, obase + go, in);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    if (s != cur_s || h != cur_h) {
      const int64_t s0off = (static_cast<int64_t>(s) * H + h) * kDim * kDim;
      if (sstart16) {
        // the scan's bf16 copy: 16 pieces of 16 bytes per row, with the tiles
        const __nv_bfloat16* src = sstart16 + s0off;
#pragma unroll 4
        for (int i = t; i < kDim * 16; i += FX_THREADS)
          cp_async16_zfill(sb + (i >> 4) * SG_ROW + (i & 15) * 16, src + (i >> 4) * kDim + (i & 15) * 8,
                           true);
        asm volatile("cp.async.commit_group;" ::: "memory");
      } else {
        const float2* src = reinterpret_cast<const float2*>(sstart + s0off);
        for (int i = t; i < kDim * kDim / 2; i += FX_THREADS) {
          const float2 x = __ldg(src + i);
          const int v = i >> 6, kp = i & 63;
          *reinterpret_cast<uint32_t*>(sb + v * SG_ROW + kp * 4) = pack_bf16(x.x, x.y);
        }
      }
      cur_s = s;
      cur_h = h;
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    const int rbase = 16 * w;
    if (rbase < nt) {
      uint32_t a[8][4];
      const uint8_t* arow = yt + (rbase + (l & 7) + ((l >> 3) & 1) * 8) * SG_ROW + (l >> 4) * 16;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) ldsm_x4(a[kk], arow + kk * 32);
      const int g = l >> 2, q2 = 2 * (l & 3);
#pragma unroll 2
      for (int n8 = 0; n8 < 16; ++n8) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const uint8_t* brow = sb + (n8 * 8 + (l & 7)) * SG_ROW + (l >> 3) * 16;
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
          uint32_t b[4];
          ldsm_x4(b, brow + k2 * 64);
          mma16816(acc, a[2 * k2], b[0], b[1]);
          mma16816(acc, a[2 * k2 + 1], b[2], b[3]);
        }
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          uint32_t* p = reinterpret_cast<uint32_t*>(ot + (rbase + g + 8 * hr) * SG_ROW +
                                                    (n8 * 8 + q2) * 2);
          const uint32_t o32 = *p;
          const float2 o = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&o32));
          *p = pack_bf16(o.x + acc[2 * hr], o.y + acc[2 * hr + 1]);
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < SG_BLOCK * 16 / FX_THREADS; ++k) {
      const int i = t + k * FX_THREADS, r = i >> 4, c = i & 15;
      if (r < nt)
        *reinterpret_cast<uint4*>(obase + r * row_stride + c * 8) =
            *reinterpret_cast<const uint4*>(ot + r * SG_ROW + c * 16);
    }
  }
}

cudaError_t launch_seg_plan(const int32_t* cu, int64_t T_total, int N, int P, int32_t* cu_seg,
                            int32_t* blk, cudaStream_t stream) {
  seg_plan_kernel<<<1, 1024, 0, stream>>>(cu, T_total, N, P, cu_seg, blk);
  return cudaGetLastError();
}

template <int ROWS>
cudaError_t launch_affine_scan_t(float* xs, const float* ms, int N, int P, int H,
                                 void* final_state, bool final_bf16, __nv_bfloat16* s0_bf16,
                                 cudaStream_t stream) {
  static std::atomic<uint64_t> smem_set{0};
  if (const cudaError_t e = ensure_smem_limit(
          reinterpret_cast<const void*>(affine_scan_kernel<ROWS>), ScanShape<ROWS>::SMEM, smem_set);
      e != cudaSuccess)
    return e;
  const int64_t ctas = static_cast<int64_t>(N) * H * (kDim / ROWS);
  return launch_pdl(affine_scan_kernel<ROWS>, dim3(static_cast<unsigned>(ctas)),
                    dim3(ScanShape<ROWS>::NT), ScanShape<ROWS>::SMEM, stream, xs, ms, N, P, H,
                    final_state, final_bf16, s0_bf16);
}

cudaError_t launch_affine_scan(float* xs, const float* ms, int N, int P, int H,
                               void* final_state, bool final_bf16, int sm_count,
                               cudaStream_t stream, void* s0_bf16) {
  const int64_t units = static_cast<int64_t>(N) * H;
  if (units == 0) return cudaSuccess;
  __nv_bfloat16* bf = static_cast<__nv_bfloat16*>(s0_bf16);
  // the most CTAs per (sequence, head) that still fit one per SM
  const int64_t slots = sm_count;
  if (units * 16 <= slots)
    return launch_affine_scan_t<8>(xs, ms, N, P, H, final_state, final_bf16, bf, stream);
  if (units * 8 <= slots)
    return launch_affine_scan_t<16>(xs, ms, N, P, H, final_state, final_bf16, bf, stream);
  if (units * 4 <= slots)
    return launch_affine_scan_t<32>(xs, ms, N, P, H, final_state, final_bf16, bf, stream);
  if (units * 2 <= slots)
    return launch_affine_scan_t<64>(xs, ms, N, P, H, final_state, final_bf16, bf, stream);
  return launch_affine_scan_t<128>(xs, ms, N, P, H, final_state, final_bf16, bf, stream);
}

cudaError_t launch_seg_fixup(const int32_t* cu_seg, const int32_t* blk, int Nseg, int H,
                             const float* sstart, const void* y, void* out, int sm_count,
                             cudaStream_t stream, const void* sstart16) {
  static std::atomic<uint64_t> smem_set{0};
  if (const cudaError_t e =
          ensure_smem_limit(reinterpret_cast<const void*>(seg_fixup_kernel), FX_SMEM, smem_set);
      e != cudaSuccess)
    return e;
  if (Nseg == 0) return cudaSuccess;
  return launch_pdl(seg_fixup_kernel, dim3(static_cast<unsigned>(3 * sm_count)), dim3(FX_THREADS),
                    FX_SMEM, stream, cu_seg, blk, Nseg, H, sstart,
                    static_cast<const __nv_bfloat16*>(sstart16), static_cast<const __nv_bfloat16*>(y),
                    static_cast<__nv_bfloat16*>(out));
}

}  // namespace kda
