// kda_decode.cu -- the recurrent (decode) schedule of the KDA forward pass: the
// token-by-token recurrence of "You Could Have Come Up with Kimi Delta
// Attention" (sec. 4, boxed; sec. 5 "The fused recurrent Triton kernel" for the
// decode regime), for short sequences and stateful serving, where the state
// read and write dominate and there are no 16-token chunks to batch.
//
// One CTA per (sequence, head, 32 value rows): 256 threads, thread
// (row r = t / 8, slice s = t % 8) keeps the 16 entries S[32 b + r][4 (8 j + s) + e]
// (j, e = 0..3; fp32) in registers for the whole call: four groups of four
// channels, interleaved over the slices so that the eight slices of a row read
// eight consecutive 16-byte words of the per-token vectors (no bank conflicts)
// and their state loads stay coalesced.  Per token:
//   threads 0-127 (channel c = t): q_c, k_c, g_c -> alpha_c = 2^(lb log2e sigma(g_c));
//     squared norms reduced over the CTA; k^_c, s q^_c, alpha_c -> shared memory
//   every thread, on its 16 entries:  S *= alpha  (forget)
//     pred = sum S k^ (8-lane shuffle reduction), e = beta (v_r - pred)  (predict, correct)
//     S += e k^  (write),  o_r = sum S (s q^) (read), stored as bf16 by slice 0.
// The states are fp32 (or bf16, converted at load and store); the final state
// may overwrite the initial state in place (every thread reads its entries
// before it writes them, and no two threads share an entry).
#include "kda_common.cuh"

namespace kda {

constexpr int DEC_THREADS = 256;
constexpr int DEC_ROWS = 32;  // value rows per CTA

__global__ void __launch_bounds__(DEC_THREADS)
decode_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
              const __nv_bfloat16* __restrict__ v, const __nv_bfloat16* __restrict__ g,
              const __nv_bfloat16* __restrict__ beta_raw, float scale, float lb_log2e,
              float eps, const void* init, const int32_t* __restrict__ cu, int64_t T_total,
              int H, int N, __nv_bfloat16* __restrict__ out, void* final_state, FwdOpts opts) {
  // this launch may start while the previous kernel on the stream (say, the
  // previous decode step, whose final state is this one's initial state)
  // runs: wait for it before the first read
  grid_dep_wait();
  grid_dep_launch();
  __shared__ float4 sk4[kDim / 4], sq4[kDim / 4], sa4[kDim / 4];
  __shared__ float red[2][4];
  const int t = threadIdx.x, l = t & 31, w = t >> 5;
  const int tile = blockIdx.x & 3;
  const int unit = blockIdx.x >> 2;
  const int n = unit / H, h = unit - (unit / H) * H;
  const int r = t >> 3, sl = t & 7;
  const int vrow = tile * DEC_ROWS + r;
  int64_t bos, eos;
  seq_bounds(cu, T_total, N, n, bos, eos);
  const int64_t sbase = ((static_cast<int64_t>(n) * H + h) * kDim + vrow) * kDim + sl * 4;
  // entries 4 j .. 4 j + 3 of s[] are channels 4 (8 j + sl) .. + 3: element offset 32 j

  float s[16];
  if (init && opts.state_bf16) {
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(init) + sbase;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint2 b = *reinterpret_cast<const uint2*>(src + 32 * j);
      const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b.x));
      const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b.y));
      s[4 * j] = lo.x;
      s[4 * j + 1] = lo.y;
      s[4 * j + 2] = hi.x;
      s[4 * j + 3] = hi.y;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 x = init ? *reinterpret_cast<const float4*>(static_cast<const float*>(init) + sbase + 32 * j)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
      s[4 * j] = x.x;
      s[4 * j + 1] = x.y;
      s[4 * j + 2] = x.z;
      s[4 * j + 3] = x.w;
    }
  }
  const float hl = 0.5f * lb_log2e;
  for (int64_t tok = bos; tok < eos; ++tok) {
    const int64_t row = (tok * H + h) * kDim;
    float qc = 0.f, kc = 0.f;
    if (t < kDim) {
      qc = __bfloat162float(q[row + t]);
      kc = __bfloat162float(k[row + t]);
      const float gc = __bfloat162float(opts.gate_scalar ? g[tok * H + h] : g[row + t]);
      reinterpret_cast<float*>(sa4)[t] = ex2_approx(fmaf(hl, tanh_approx(0.5f * gc), hl));
      float sqq = qc * qc, skk = kc * kc;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sqq += __shfl_xor_sync(0xffffffffu, sqq, o);
        skk += __shfl_xor_sync(0xffffffffu, skk, o);
      }
      if (l == 0) {
        red[0][w] = sqq;
        red[1][w] = skk;
      }
    }
    const float beta = sigmoid_fast(__bfloat162float(beta_raw[tok * H + h]));
    const float vv = __bfloat162float(v[row + vrow]);
    __syncthreads();
    if (t < kDim) {
      const float rq = scale * rsqrtf(red[0][0] + red[0][1] + red[0][2] + red[0][3] + eps);
      const float rk = rsqrtf(red[1][0] + red[1][1] + red[1][2] + red[1][3] + eps);
      reinterpret_cast<float*>(sq4)[t] = qc * rq;
      reinterpret_cast<float*>(sk4)[t] = kc * rk;
    }
    __syncthreads();
    float pred = 0.f;
#pragma unroll
    for (int i4 = 0; i4 < 4; ++i4) {
      const float4 a = sa4[i4 * 8 + sl], kk = sk4[i4 * 8 + sl];
      s[4 * i4] *= a.x;
      s[4 * i4 + 1] *= a.y;
      s[4 * i4 + 2] *= a.z;
      s[4 * i4 + 3] *= a.w;
      pred = fmaf(s[4 * i4], kk.x, pred);
      pred = fmaf(s[4 * i4 + 1], kk.y, pred);
      pred = fmaf(s[4 * i4 + 2], kk.z, pred);
      pred = fmaf(s[4 * i4 + 3], kk.w, pred);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) pred += __shfl_xor_sync(0xffffffffu, pred, o);
    const float e = beta * (vv - pred);
    float o_acc = 0.f;
#pragma unroll
    for (int i4 = 0; i4 < 4; ++i4) {
      const float4 kk = sk4[i4 * 8 + sl], qq = sq4[i4 * 8 + sl];
      s[4 * i4] = fmaf(e, kk.x, s[4 * i4]);
      s[4 * i4 + 1] = fmaf(e, kk.y, s[4 * i4 + 1]);
      s[4 * i4 + 2] = fmaf(e, kk.z, s[4 * i4 + 2]);
      s[4 * i4 + 3] = fmaf(e, kk.w, s[4 * i4 + 3]);
      o_acc = fmaf(s[4 * i4], qq.x, o_acc);
      o_acc = fmaf(s[4 * i4 + 1], qq.y, o_acc);
      o_acc = fmaf(s[4 * i4 + 2], qq.z, o_acc);
      o_acc = fmaf(s[4 * i4 + 3], qq.w, o_acc);
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) o_acc += __shfl_xor_sync(0xffffffffu, o_acc, o);
    if (sl == 0) out[row + vrow] = __float2bfloat16_rn(o_acc);
    __syncthreads();  // shared q^, k^, alpha of this token are no longer read
  }
  if (final_state && opts.state_bf16) {
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(final_state) + sbase;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<uint2*>(dst + 32 * j) =
          make_uint2(pack_bf16(s[4 * j], s[4 * j + 1]), pack_bf16(s[4 * j + 2], s[4 * j + 3]));
  } else if (final_state) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<float4*>(static_cast<float*>(final_state) + sbase + 32 * j) =
          make_float4(s[4 * j], s[4 * j + 1], s[4 * j + 2], s[4 * j + 3]);
  }
}

cudaError_t launch_decode(const void* q, const void* k, const void* v, const void* g,
                          const void* beta_raw, float scale, float lower_bound, float eps,
                          const void* init, const int32_t* cu, int64_t T_total, int H, int N,
                          void* out, void* final_state, FwdOpts opts, cudaStream_t stream) {
  const int64_t ctas = static_cast<int64_t>(N) * H * (kDim / DEC_ROWS);
  if (ctas == 0) return cudaSuccess;
  return launch_pdl(decode_kernel, dim3(static_cast<unsigned>(ctas)), dim3(DEC_THREADS), 0, stream,
                    static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
                    static_cast<const __nv_bfloat16*>(v), static_cast<const __nv_bfloat16*>(g),
                    static_cast<const __nv_bfloat16*>(beta_raw), scale,
                    lower_bound * 1.4426950408889634f, eps, init, cu, T_total, H, N,
                    static_cast<__nv_bfloat16*>(out), final_state, opts);
}

}  // namespace kda
