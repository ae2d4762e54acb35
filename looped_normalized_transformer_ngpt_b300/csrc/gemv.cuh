// gemv.cuh - projections for few rows (decode: M = batch <= 16).
//
// With M <= 16 the projections are weight-streaming (8 to 16 FLOP per weight
// byte): the bound is HBM bandwidth, not the tensor cores.  Each warp owns
// two weight rows, reads them once with 16-byte non-caching loads (all K
// chunks issued before use), multiplies with the M activation rows (L1/L2
// resident) in fp32 and reduces across the warp; one CTA = 4 warps = 8 output
// features, so even N = 1024 spreads over 128 CTAs.
//
//   Y[m, n] = scale[n] * sum_k X[m, k] W[n, k]     (fp32 out)
//
// The per-projection math of the tensor-core epilogues then runs as small row
// kernels on Y: RoPE + per-head L2 norm + s_qk for q/k, copy for v, sigmoid
// for the gate ("Dory1.0-4B: A Looped Normalized-GPT", Architecture), and
// m = u * SiLU(v) for the SwiGLU MLP.
#pragma once
#include "ptx.cuh"

namespace dory {

constexpr int kGemvMaxM = 16;
constexpr int kGemvRowsPerWarp = 2;
constexpr int kGemvWarps = 4;
constexpr int kGemvRowsPerCta = kGemvRowsPerWarp * kGemvWarps;

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

// K must be a multiple of 8; X rows are ldx elements apart.
template <int MM>
__global__ void __launch_bounds__(kGemvWarps * 32) gemv_kernel(const __nv_bfloat16* X, int ldx,
                                                               int M, const __nv_bfloat16* W,
                                                               int N, int K, float* Y, int ldy,
                                                               const float* col_scale) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = (blockIdx.x * kGemvWarps + warp) * kGemvRowsPerWarp;
  if (r0 >= N) return;
  const bool has1 = r0 + 1 < N;
  float acc[kGemvRowsPerWarp][MM];
#pragma unroll
  for (int r = 0; r < kGemvRowsPerWarp; ++r)
#pragma unroll
    for (int m = 0; m < MM; ++m) acc[r][m] = 0.f;
  const __nv_bfloat16* w0 = W + (long long)r0 * K;
  const __nv_bfloat16* w1 = W + (long long)(has1 ? r0 + 1 : r0) * K;
  constexpr int U = 4;   // K chunks of 256 elements in flight per lane
  for (int kb = lane * 8; kb < K; kb += 256 * U) {
    uint4 a[U], b[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int k = kb + u * 256;
      if (k < K) {
        a[u] = ld_stream16(w0 + k);
        b[u] = ld_stream16(w1 + k);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int k = kb + u * 256;
      if (k < K) {
        float fa[8], fb[8];
        bf16x8_to_f32(a[u], fa);
        bf16x8_to_f32(b[u], fb);
#pragma unroll
        for (int m = 0; m < MM; ++m) {
          if (m < M) {
            float fx[8];
            bf16x8_to_f32(*reinterpret_cast<const uint4*>(X + (long long)m * ldx + k), fx);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              acc[0][m] = fmaf(fa[i], fx[i], acc[0][m]);
              acc[1][m] = fmaf(fb[i], fx[i], acc[1][m]);
            }
          }
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kGemvRowsPerWarp; ++r)
#pragma unroll
    for (int m = 0; m < MM; ++m) acc[r][m] = warp_sum(acc[r][m]);
  if (lane == 0) {
#pragma unroll
    for (int r = 0; r < kGemvRowsPerWarp; ++r) {
      const int n = r0 + r;
      if (n >= N) break;
      const float sc = col_scale ? col_scale[n] : 1.f;
#pragma unroll
      for (int m = 0; m < MM; ++m)
        if (m < M) Y[(long long)m * ldy + n] = acc[r][m] * sc;
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

// m = u * SiLU(v) from Y [M, 2F] = [u | v] (fp32) to bf16 [M, F].
__global__ void swiglu_post_kernel(const float* Y, int M, int F, __nv_bfloat16* m_out) {
  const long long n = (long long)M * F;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long r = idx / F, c = idx % F;
    const float u = Y[r * 2 * F + c], s = Y[r * 2 * F + F + c];
    m_out[idx] = __float2bfloat16_rn(u * (s / (1.0f + __expf(-s))));
  }
}

}  // namespace dory
