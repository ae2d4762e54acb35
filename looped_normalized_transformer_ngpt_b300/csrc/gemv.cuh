// gemv.cuh - projections for few rows (decode: M = batch <= 16).
//
// With M <= 16 rows the projections stream weights (2 M FLOP per 2-byte
// weight): the bound is HBM bandwidth and load latency, not the tensor cores.
// One warp owns one output feature (or, for SwiGLU, the pair of W_up and W_sl
// rows of one feature) and one K segment of J x 256 elements: every lane
// issues all J 16-byte non-caching weight loads of its segment before using
// any, multiplies with the M activation rows (L2 resident) in fp32 and reduces
// across the warp; the S segments of a row (S = 1, 2, 4 or 8, chosen so that
// J <= 8) are summed through shared memory.  A CTA is 8 warps = 8 / S
// features, so even N = 1024 spreads over 128 to 1024 CTAs with up to
// 8 KB of weight loads in flight per warp.
//
//   Y[m, n] = scale[n] * sum_k X[m, k] W[n, k]                 (fp32 out)
//   SwiGLU:  m_out[m, n] = u * SiLU(v),  u = X W_up[n]^T, v = X W_sl[n]^T
//
// The q/k/v/gate math of the tensor-core epilogue runs on Y in a small row
// kernel: RoPE + per-head L2 norm + s_qk for q and k, copy for v, sigmoid for
// the gate ("Dory1.0-4B: A Looped Normalized-GPT", Architecture).
#pragma once
#include "ptx.cuh"

namespace dory {

constexpr int kGemvMaxM = 16;
constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;
constexpr int kGemvMaxK = kGemvWarps * 8 * 256;     // S <= 8 segments of J <= 8 chunks

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// K must be a multiple of 8; X rows are ldx elements apart (16-byte aligned).
// SWIGLU: W holds [W_up; W_sl] and feature n uses rows n and n + pair_off.
template <int MM, int J, bool SWIGLU>
__global__ void __launch_bounds__(kGemvThreads)
    gemv_kernel(const __nv_bfloat16* X, int ldx, int M, const __nv_bfloat16* W, int N, int K,
                int S, float* Y, int ldy, const float* col_scale, int pair_off,
                __nv_bfloat16* m_out, int ldm) {
  constexpr int R = SWIGLU ? 2 : 1;
  __shared__ float red[kGemvWarps][R][MM];
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows_per_cta = kGemvWarps / S;
  const int n = blockIdx.x * rows_per_cta + warp / S;
  const int seg = warp % S;
  const bool valid = n < N;
  const int kbase = seg * (J * 256) + lane * 8;

  uint4 w[R][J];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const __nv_bfloat16* wr = W + (long long)(valid ? n + r * pair_off : 0) * K;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int k = kbase + j * 256;
      w[r][j] = (valid && k < K) ? ld_stream16(wr + k) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  float acc[R][MM];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < MM; ++m) acc[r][m] = 0.f;
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int k = kbase + j * 256;
    if (valid && k < K) {
      float fw[R][8];
#pragma unroll
      for (int r = 0; r < R; ++r) bf16x8_to_f32(w[r][j], fw[r]);
#pragma unroll
      for (int m = 0; m < MM; ++m) {
        if (m < M) {
          float fx[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(X + (long long)m * ldx + k), fx);
#pragma unroll
          for (int r = 0; r < R; ++r)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[r][m] = fmaf(fw[r][i], fx[i], acc[r][m]);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < MM; ++m) {
      const float v = warp_sum(acc[r][m]);
      if (lane == 0) red[warp][r][m] = v;
    }
  __syncthreads();
  const int t = threadIdx.x;
  if (t < rows_per_cta * MM) {
    const int rl = t / MM, m = t % MM;
    const int nn = blockIdx.x * rows_per_cta + rl;
    if (nn < N && m < M) {
      float s0 = 0.f, s1 = 0.f;
      for (int sg = 0; sg < S; ++sg) {
        s0 += red[rl * S + sg][0][m];
        if (SWIGLU) s1 += red[rl * S + sg][R - 1][m];
      }
      if (SWIGLU)
        m_out[(long long)m * ldm + nn] = __float2bfloat16_rn(s0 * (s1 / (1.0f + __expf(-s1))));
      else
        Y[(long long)m * ldy + nn] = s0 * (col_scale ? col_scale[nn] : 1.f);
    }
  }
}

// q/k/v/gate post-processing of a fp32 projection Y [M, (2 n_q + 2 n_kv) dh]
// (row = token).  grid = (M, n_q + n_kv + n_kv + n_q), block = max(32, dh / 2);
// thread i < dh / 2 owns columns i and i + dh / 2 of its head.
__global__ void qkvg_post_kernel(const float* Y, int M, int n_q, int n_kv, int dh,
                                 const float* s_qk, const float2* rope, int rows_per_seq,
                                 __nv_bfloat16* q, __nv_bfloat16* k, __nv_bfloat16* v,
                                 __nv_bfloat16* g) {
  __shared__ float red[8];
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x, head = blockIdx.y;
  const int half = dh / 2, i = threadIdx.x;
  const bool own = i < half;
  const int N = (2 * n_q + 2 * n_kv) * dh;
  const float* y = Y + (long long)row * N + (long long)head * dh;
  float x1 = own ? y[i] : 0.f, x2 = own ? y[i + half] : 0.f;
  if (head < n_q + n_kv) {
    float ss = warp_sum(x1 * x1 + x2 * x2);
    const int w = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    if ((threadIdx.x & 31) == 0) red[w] = ss;
    __syncthreads();
    ss = 0.f;
    for (int j = 0; j < nw; ++j) ss += red[j];
    const float inv = 1.0f / sqrtf(fmaxf(ss, 1e-12f));
    if (rope && own) {
      const float2 cs = rope[(long long)(row % rows_per_seq) * half + i];
      const float y1 = x1 * cs.x - x2 * cs.y, y2 = x2 * cs.x + x1 * cs.y;
      x1 = y1;
      x2 = y2;
    }
    if (!own) return;
    x1 *= inv * s_qk[i];
    x2 *= inv * s_qk[i + half];
    __nv_bfloat16* dst = head < n_q ? q + ((long long)row * n_q + head) * dh
                                    : k + ((long long)row * n_kv + head - n_q) * dh;
    dst[i] = __float2bfloat16_rn(x1);
    dst[i + half] = __float2bfloat16_rn(x2);
  } else if (!own) {
    return;
  } else if (head < n_q + 2 * n_kv) {
    __nv_bfloat16* dst = v + ((long long)row * n_kv + head - n_q - n_kv) * dh;
    dst[i] = __float2bfloat16_rn(x1);
    dst[i + half] = __float2bfloat16_rn(x2);
  } else {
    __nv_bfloat16* dst = g + ((long long)row * n_q + head - n_q - 2 * n_kv) * dh;
    dst[i] = __float2bfloat16_rn(1.0f / (1.0f + __expf(-x1)));
    dst[i + half] = __float2bfloat16_rn(1.0f / (1.0f + __expf(-x2)));
  }
}

}  // namespace dory
