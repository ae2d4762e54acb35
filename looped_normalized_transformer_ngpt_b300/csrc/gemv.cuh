// gemv.cuh - projections for few rows (M <= 16: prefill chunks, the
// verifier's rows, the quantised one-sequence decode).
//
// With M <= 16 rows the projections stream weights (2 M FLOP per 2-byte
// weight): the bound is HBM bandwidth and load latency, not the tensor cores.
// One warp owns one output feature (or, for SwiGLU, the pair of W_up and W_sl
// rows of one feature) and one K segment of J x 256 elements: every lane
// issues all J 16-byte non-caching weight loads of its segment before using
// any, multiplies with the M activation rows in fp32 and reduces across the
// warp; the S segments of a row (S = 1, 2, 4 or 8, chosen so that J <= 8) are
// summed through shared memory.  A CTA iteration covers 8 / S features; CTAs
// stride over the iterations.
//
// Weights never change during a forward pass, so each CTA loads its first
// iteration's weights BEFORE waiting on the previous kernel (programmatic
// dependent launch): the weight stream of this projection overlaps the tail
// of the kernel before it.  Later iterations prefetch the next weights into a
// second register set while the current ones are multiplied.
//
//   Y[m, n] = scale[n] * sum_k X[m, k] W[n, k]                 (fp32 out)
//   SwiGLU:  m_out[m, n] = u * SiLU(v),  u = X W_up[n]^T, v = X W_sl[n]^T
//
// PRE variant (fused nGPT step, "Dory1.0-4B: A Looped Normalized-GPT",
// Architecture): the activation rows are not read from memory but formed by
// every CTA from the previous sublayer's projection output y and the hidden
// state h:  x = N(h + alpha * (N(y) - h)),  kept in shared memory as bf16.
// CTA 0 also stores x (fp32) as the next hidden state.  This removes the
// separate residual-update kernel between two projections.
#pragma once
#include "ptx.cuh"

namespace dory {

constexpr int kGemvMaxM = 16;
constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;
constexpr int kGemvMaxK = kGemvWarps * 8 * 256;     // S <= 8 segments of J <= 8 chunks
constexpr int kGemvPreMaxD = 2048;                  // PRE: d <= 2048 (8 chunks per lane)
constexpr int kGemvStageMax = kGemvMaxM * kGemvPreMaxD * 2;   // shared-memory rows, bytes

struct GemvArgs {
  const __nv_bfloat16* X;   // activations [M, ldx] (not PRE)
  int ldx;
  int M;
  const __nv_bfloat16* W;   // weights [N (+ pair rows), K]
  int N, K, S, n_iters;
  int pair_off;             // SwiGLU: W_sl row of feature n is n + pair_off
  float* Y;                 // fp32 [M, ldy]
  int ldy;
  const float* col_scale;   // may be null
  __nv_bfloat16* m_out;     // SwiGLU bf16 [M, ldm]
  int ldm;
  // PRE: x = N(h_in + alpha * (N(y_in) - h_in)), rows of length K (= d)
  const float* h_in;
  const float* y_in;
  const float* alpha;
  float* h_out;             // written by CTA 0 (a different buffer from h_in)
  int stage_x;              // not PRE: copy X to shared memory first (M * K * 2 bytes)
  // weight-only quantised weights (quant.cuh) instead of W when qfmt != 0
  int qfmt;
  const uint8_t* Wq;        // codes
  const uint8_t* Ws;        // block scales
  const float* Wr;          // per-row scales (may be null)
};

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

__device__ __forceinline__ void ld8f(const float* p, float* v) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// The fused nGPT step of the PRE variant: warp w forms rows w, w + 8, ...
// (lane owns 8-element chunks lane, lane + 32, ...), keeping the row in
// registers between the two normalisations.
__device__ __forceinline__ void gemv_pre_rows(const GemvArgs& a, __nv_bfloat16* xs) {
  constexpr int MAXC = kGemvPreMaxD / 256;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = a.K, nch = d / 8;
  const bool store = blockIdx.x == 0 && a.h_out != nullptr;
  for (int m = warp; m < a.M; m += kGemvWarps) {
    float u[MAXC][8];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < MAXC; ++j) {
      const int ch = lane + 32 * j;
      if (ch < nch) {
        ld8f(a.y_in + (long long)m * d + ch * 8, u[j]);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss += u[j][i] * u[j][i];
      }
    }
    const float inv_y = 1.0f / sqrtf(fmaxf(warp_sum(ss), 1e-12f));
    float su = 0.f;
#pragma unroll
    for (int j = 0; j < MAXC; ++j) {
      const int ch = lane + 32 * j;
      if (ch < nch) {
        float h[8], al[8];
        ld8f(a.h_in + (long long)m * d + ch * 8, h);
        ld8f(a.alpha + ch * 8, al);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          u[j][i] = h[i] + al[i] * (u[j][i] * inv_y - h[i]);
          su += u[j][i] * u[j][i];
        }
      }
    }
    const float inv_u = 1.0f / sqrtf(fmaxf(warp_sum(su), 1e-12f));
#pragma unroll
    for (int j = 0; j < MAXC; ++j) {
      const int ch = lane + 32 * j;
      if (ch < nch) {
#pragma unroll
        for (int i = 0; i < 8; ++i) u[j][i] *= inv_u;
        uint4 p;
        p.x = pack_bf16x2(u[j][0], u[j][1]);
        p.y = pack_bf16x2(u[j][2], u[j][3]);
        p.z = pack_bf16x2(u[j][4], u[j][5]);
        p.w = pack_bf16x2(u[j][6], u[j][7]);
        *reinterpret_cast<uint4*>(xs + (long long)m * d + ch * 8) = p;
        if (store) {
          float4* o = reinterpret_cast<float4*>(a.h_out + (long long)m * d + ch * 8);
          o[0] = make_float4(u[j][0], u[j][1], u[j][2], u[j][3]);
          o[1] = make_float4(u[j][4], u[j][5], u[j][6], u[j][7]);
        }
      }
    }
  }
}

// K must be a multiple of 8; X rows are 16-byte aligned.  Dynamic shared
// memory (PRE, or stage_x): M * K bf16.
template <int MM, int J, bool SWIGLU, bool PRE>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(const GemvArgs a) {
  constexpr int R = SWIGLU ? 2 : 1;
  extern __shared__ __align__(16) uint8_t gemv_smem[];
  __shared__ float red[kGemvWarps][R][MM];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.S;
  const int fpi = kGemvWarps / S;                 // features per iteration
  const int seg = warp % S;
  const int kbase = seg * (J * 256) + lane * 8;

  uint4 w[R][J], wn[R][J];
  auto load_w = [&](uint4 (&dst)[R][J], int it) {
    const int n = it * fpi + warp / S;
    const bool valid = it < a.n_iters && n < a.N;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const __nv_bfloat16* wr = a.W + (long long)(valid ? n + r * a.pair_off : 0) * a.K;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int k = kbase + j * 256;
        dst[r][j] = (valid && k < a.K) ? ld_stream16(wr + k) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
  };

  int it = blockIdx.x;
  load_w(w, it);                                  // weights: safe before the wait
  pdl_wait();
  pdl_trigger();

  const __nv_bfloat16* X = a.X;
  int ldx = a.ldx;
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(gemv_smem);
  if (PRE) {
    gemv_pre_rows(a, xs);
    __syncthreads();
    X = xs;
    ldx = a.K;
  } else if (a.stage_x) {
    // the activation rows (written by the previous kernel) staged once with
    // coalesced 16-byte loads, instead of one dependent L2 round trip per
    // weight chunk inside the loop below
    const int cpr = a.K / 8;
    for (int i = threadIdx.x; i < a.M * cpr; i += kGemvThreads) {
      const int m = i / cpr, c = i % cpr;
      *reinterpret_cast<uint4*>(xs + (long long)m * a.K + c * 8) =
          *reinterpret_cast<const uint4*>(a.X + (long long)m * a.ldx + c * 8);
    }
    __syncthreads();
    X = xs;
    ldx = a.K;
  }

  for (; it < a.n_iters; it += gridDim.x) {
    const int nxt = it + gridDim.x;
    if (nxt < a.n_iters) load_w(wn, nxt);
    const int n = it * fpi + warp / S;
    const bool valid = n < a.N;
    float acc[R][MM];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MM; ++m) acc[r][m] = 0.f;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int k = kbase + j * 256;
      if (valid && k < a.K) {
        float fw[R][8];
#pragma unroll
        for (int r = 0; r < R; ++r) bf16x8_to_f32(w[r][j], fw[r]);
#pragma unroll
        for (int m = 0; m < MM; ++m) {
          if (m < a.M) {
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
    if (t < fpi * MM) {
      const int rl = t / MM, m = t % MM;
      const int nn = it * fpi + rl;
      if (nn < a.N && m < a.M) {
        float s0 = 0.f, s1 = 0.f;
        for (int sg = 0; sg < S; ++sg) {
          s0 += red[rl * S + sg][0][m];
          if (SWIGLU) s1 += red[rl * S + sg][R - 1][m];
        }
        if (SWIGLU)
          a.m_out[(long long)m * a.ldm + nn] = __float2bfloat16_rn(s0 * (s1 / (1.0f + __expf(-s1))));
        else
          a.Y[(long long)m * a.ldy + nn] = s0 * (a.col_scale ? a.col_scale[nn] : 1.f);
      }
    }
    __syncthreads();
    if (nxt < a.n_iters) {
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int j = 0; j < J; ++j) w[r][j] = wn[r][j];
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
