// quant.cuh - weight-only quantised projection weights (MXFP8, NVFP4):
// the quantisers and the few-row projection (decode GEMV) that streams them.
//
// "Dory1.0-4B: A Looped Normalized-GPT", Quantization (Post-Training
// Quantization): every weight matrix except the token embeddings and the LM
// head is quantised, weights only; MXFP8 with maximum scaling, NVFP4 with
// each block's E4M3 scale chosen to minimise the block's squared error over
// all 126 positive finite E4M3 values.
//
// Formats (row-major [rows, K], blocks of consecutive elements along K):
//   MXFP8: codes  uint8 [rows, K]       E4M3 (sign bit 7)
//          scales uint8 [rows, K / 32]  E8M0: 2^(s - 127);  x ~ code * 2^(s-127)
//   NVFP4: codes  uint8 [rows, K / 2]   E2M1, element 2i in the low nibble
//          scales uint8 [rows, K / 16]  E4M3 block scale s
//          row_scale float [rows]       the tensor's scale s_g on every row;
//                                       x ~ code * s * s_g
// Maximum scaling (MXFP8): e = floor(log2 max|x|) - 8 clamped to [-127, 127]
// (-127 for a block whose maximum is 0 or subnormal), element = x / 2^e
// rounded to nearest even E4M3, saturating at 448.  NVFP4: s_g = max|x| /
// (6 * 448) over the tensor (1 if it is all zero); each block tries the
// candidates in increasing order with the float32 expression
//   d = s * s_g,  v = x / d,  q = E2M1(v) (nearest, ties to even, at most 6),
//   err += (x - q * d)^2      (elements in order, every operation rounded)
// and keeps the first smallest error.  The decision is an integer taken from
// floating point, so its expression and order are fixed (no contraction:
// the __f*_rn intrinsics).
//
// The GEMV (gemv_q_kernel) has the shape of gemv_kernel (gemv.cuh): one warp
// per output feature and K segment, every lane's 16-byte weight loads issued
// before any is used (the first before the wait on the previous kernel),
// activations from shared memory, the same PRE (fused nGPT step) and SwiGLU
// variants.  A 16-byte chunk holds 16 (MXFP8) or 32 (NVFP4) weights, so the
// bytes streamed per weight drop to 1/2 or 1/4 of bf16, plus one scale byte
// per 32 or 16 weights.  Codes are expanded with the hardware conversions
// (cvt.rn.f16x2.e4m3x2 / .e2m1x2, exact); the products with the activations
// are summed in fp32 per 16 weights and then multiplied by the block scale.
#pragma once
#include <cuda_fp16.h>
#include "gemv.cuh"
#include "gemv_tma.cuh"

namespace dory {

enum QuantFmt : int { QF_NONE = 0, QF_MXFP8 = 1, QF_NVFP4 = 2 };

// ---------------------------------------------------------------- codes
// four E4M3 codes (byte i = element i) -> four floats
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float* f) {
  uint32_t h0, h1;
  asm("{\n\t.reg .b16 a0, a1;\n\tmov.b32 {a0, a1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a0;\n\tcvt.rn.f16x2.e4m3x2 %1, a1;\n\t}"
      : "=r"(h0), "=r"(h1)
      : "r"(w));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h0));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&h1));
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
}

// eight E2M1 codes (nibble i = element i) -> eight floats
__device__ __forceinline__ void e2m1x8_to_f32(uint32_t w, float* f) {
  uint32_t h[4];
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&h[i]));
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// E8M0 scale code -> 2^(c - 127) (code 0 is the subnormal 2^-127)
__device__ __forceinline__ float e8m0_to_f32(uint32_t c) {
  return c ? __uint_as_float(c << 23) : __uint_as_float(0x00400000u);
}

// one E4M3 code (low byte) -> float
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
  float f[4];
  e4m3x4_to_f32(c & 0xFFu, f);
  return f[0];
}

// two floats -> two E4M3 codes (lo in the low byte), nearest even, saturating
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// E2M1 magnitude code (0..7) of a >= 0: nearest of 0 .5 1 1.5 2 3 4 6, ties
// to the even code (midpoints .25 .75 1.25 1.75 2.5 3.5 5), saturating
__device__ __forceinline__ int e2m1_code(float a) {
  return a <= 0.25f ? 0 : a < 0.75f ? 1 : a <= 1.25f ? 2 : a < 1.75f ? 3
       : a <= 2.5f ? 4 : a < 3.5f ? 5 : a <= 5.0f ? 6 : 7;
}

__device__ __forceinline__ float e2m1_mag(int c) {
  return c < 4 ? 0.5f * c : (c < 6 ? (float)(c - 2) : 2.0f * (c - 4));
}

// ---------------------------------------------------------------- quantisers
// max |W| over n bf16 values (n a multiple of 8) -> atomicMax on the float
// bits in *amax (the caller zeroes it first)
__global__ void quant_amax_kernel(const __nv_bfloat16* W, long long n, unsigned* amax) {
  unsigned m = 0;
  const uint4* p = reinterpret_cast<const uint4*>(W);
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n / 8;
       i += (long long)gridDim.x * blockDim.x) {
    const uint4 v = p[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) m = max(m, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
  }
  m = __reduce_max_sync(0xffffffffu, m);
  if ((threadIdx.x & 31) == 0 && m) atomicMax(amax, m << 16);
}

// s_g = amax / (6 * 448) (1 if amax = 0) written to every row; row_scale[0]
// holds the amax bits on entry.  One CTA.
__global__ void quant_gscale_kernel(float* row_scale, int rows) {
  __shared__ float sg;
  if (threadIdx.x == 0) {
    const float amax = row_scale[0];
    sg = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 2688.0f);
  }
  __syncthreads();
  for (int r = threadIdx.x; r < rows; r += blockDim.x) row_scale[r] = sg;
}

// one thread per block of 32: codes, E8M0 scale, bf16 dequantised values
// (deq may alias W: every thread reads its block before writing it)
__global__ void quant_mxfp8_kernel(const __nv_bfloat16* W, long long n_blocks, uint8_t* codes,
                                   uint8_t* scales, __nv_bfloat16* deq, float* row_scale, int K) {
  const long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (b >= n_blocks) return;
  const uint4* src = reinterpret_cast<const uint4*>(W) + b * 4;
  uint4 v[4];
  unsigned amax = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[i] = src[i];
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) amax = max(amax, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
  }
  const int expo = (int)(amax >> 7) & 0xFF;                 // bf16 exponent field
  const int e = expo == 0 ? -127 : max(expo - 127 - 8, -127);
  const float inv = __uint_as_float((uint32_t)(127 - e) << 23);   // 2^-e (e <= 119)
  const float sc = e8m0_to_f32((uint32_t)(e + 127));
  uint32_t c[8];
  uint4 dq[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float x[8];
    bf16x8_to_f32(v[i], x);
    c[2 * i] = f32x2_to_e4m3x2(x[0] * inv, x[1] * inv) | (f32x2_to_e4m3x2(x[2] * inv, x[3] * inv) << 16);
    c[2 * i + 1] =
        f32x2_to_e4m3x2(x[4] * inv, x[5] * inv) | (f32x2_to_e4m3x2(x[6] * inv, x[7] * inv) << 16);
    float y[8];
    e4m3x4_to_f32(c[2 * i], y);
    e4m3x4_to_f32(c[2 * i + 1], y + 4);
    dq[i].x = pack_bf16x2(y[0] * sc, y[1] * sc);
    dq[i].y = pack_bf16x2(y[2] * sc, y[3] * sc);
    dq[i].z = pack_bf16x2(y[4] * sc, y[5] * sc);
    dq[i].w = pack_bf16x2(y[6] * sc, y[7] * sc);
  }
  uint4* cd = reinterpret_cast<uint4*>(codes) + b * 2;
  cd[0] = make_uint4(c[0], c[1], c[2], c[3]);
  cd[1] = make_uint4(c[4], c[5], c[6], c[7]);
  scales[b] = (uint8_t)(e + 127);
  if (deq) {
    uint4* dd = reinterpret_cast<uint4*>(deq) + b * 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) dd[i] = dq[i];
  }
  if (row_scale && (b * 32) % K == 0) row_scale[b * 32 / K] = 1.0f;
}

// one thread per block of 16: the squared-error scale search
__global__ void __launch_bounds__(128) quant_nvfp4_kernel(const __nv_bfloat16* W,
                                                          long long n_blocks, int K,
                                                          const float* row_scale, uint8_t* codes,
                                                          uint8_t* scales, __nv_bfloat16* deq) {
  __shared__ float cand[128];
  if (threadIdx.x < 126) cand[threadIdx.x] = e4m3_to_f32(threadIdx.x + 1);
  __syncthreads();
  const long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (b >= n_blocks) return;
  const float s_g = row_scale[b * 16 / K];
  const uint4* src = reinterpret_cast<const uint4*>(W) + b * 2;
  float x[16];
  bf16x8_to_f32(src[0], x);
  bf16x8_to_f32(src[1], x + 8);
  float best = __int_as_float(0x7f800000);                  // +inf
  int bc = 0;
  for (int c = 0; c < 126; ++c) {
    const float d = __fmul_rn(cand[c], s_g);
    float err = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float v = __fdiv_rn(x[i], d);
      const float q = copysignf(e2m1_mag(e2m1_code(fabsf(v))), v);
      const float e = __fsub_rn(x[i], __fmul_rn(q, d));
      err = __fadd_rn(err, __fmul_rn(e, e));
    }
    if (err < best) {
      best = err;
      bc = c;
    }
  }
  const float s = cand[bc];
  const float d = __fmul_rn(s, s_g);
  uint32_t packed[2] = {0u, 0u};
  uint32_t dq[8];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float v = __fdiv_rn(x[i], d);
    const int mc = e2m1_code(fabsf(v));
    const uint32_t code = (uint32_t)mc | (signbit(v) ? 8u : 0u);
    packed[i / 8] |= code << (4 * (i % 8));
    x[i] = __fmul_rn(copysignf(e2m1_mag(mc), v) * s, s_g);   // q * s exact, then * s_g
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) dq[i] = pack_bf16x2(x[2 * i], x[2 * i + 1]);
  reinterpret_cast<uint2*>(codes)[b] = make_uint2(packed[0], packed[1]);
  scales[b] = (uint8_t)(bc + 1);
  if (deq) {
    uint4* dd = reinterpret_cast<uint4*>(deq) + b * 2;
    dd[0] = make_uint4(dq[0], dq[1], dq[2], dq[3]);
    dd[1] = make_uint4(dq[4], dq[5], dq[6], dq[7]);
  }
}

// ---------------------------------------------------------------- GEMV
// GemvArgs with qfmt != 0: Wq (codes), Ws (block scales), Wr (row scales or
// null) replace W.  K a multiple of 32; code rows 16-byte aligned.
template <int FMT, int MM, int J, bool SWIGLU, bool PRE>
__global__ void __launch_bounds__(kGemvThreads) gemv_q_kernel(const GemvArgs a) {
  constexpr int R = SWIGLU ? 2 : 1;
  constexpr int E = FMT == QF_MXFP8 ? 16 : 32;     // weights per 16-byte chunk
  constexpr int G = E / 16;                        // groups of 16 weights per chunk
  extern __shared__ __align__(16) uint8_t gemv_smem[];
  __shared__ float red[kGemvWarps][R][MM];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.S;
  const int fpi = kGemvWarps / S;
  const int seg = warp % S;
  const int kbase = seg * (J * 32 * E) + lane * E;
  const long long row_bytes = FMT == QF_MXFP8 ? a.K : a.K / 2;
  const int spr = FMT == QF_MXFP8 ? a.K / 32 : a.K / 16;   // scale bytes per row

  uint4 w[R][J], wn[R][J];
  uint32_t sc[R][J], scn[R][J];
  auto load_w = [&](uint4 (&dst)[R][J], uint32_t (&ds)[R][J], int it) {
    const int n = it * fpi + warp / S;
    const bool valid = it < a.n_iters && n < a.N;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const long long row = valid ? n + r * a.pair_off : 0;
      const uint8_t* wr = a.Wq + row * row_bytes;
      const uint8_t* sr = a.Ws + row * spr;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int k = kbase + j * 32 * E;
        if (valid && k < a.K) {
          dst[r][j] = ld_stream16(wr + (FMT == QF_MXFP8 ? k : k / 2));
          ds[r][j] = FMT == QF_MXFP8 ? (uint32_t)__ldg(sr + k / 32)
                                     : (uint32_t)__ldg(reinterpret_cast<const unsigned short*>(sr + k / 16));
        } else {
          dst[r][j] = make_uint4(0u, 0u, 0u, 0u);
          ds[r][j] = 0u;
        }
      }
    }
  };

  int it = blockIdx.x;
  load_w(w, sc, it);                               // weights: safe before the wait
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
    if (nxt < a.n_iters) load_w(wn, scn, nxt);
    const int n = it * fpi + warp / S;
    const bool valid = n < a.N;
    float acc[R][MM];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MM; ++m) acc[r][m] = 0.f;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int k = kbase + j * 32 * E;
      if (valid && k < a.K) {
#pragma unroll
        for (int g = 0; g < G; ++g) {              // 16 weights sharing one scale
          float fw[R][16], bs[R];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const uint32_t* wv = reinterpret_cast<const uint32_t*>(&w[r][j]);
            if (FMT == QF_MXFP8) {
#pragma unroll
              for (int q = 0; q < 4; ++q) e4m3x4_to_f32(wv[q], fw[r] + 4 * q);
              bs[r] = e8m0_to_f32(sc[r][j]);
            } else {
              e2m1x8_to_f32(wv[2 * g], fw[r]);
              e2m1x8_to_f32(wv[2 * g + 1], fw[r] + 8);
              bs[r] = e4m3_to_f32(sc[r][j] >> (8 * g));
            }
          }
#pragma unroll
          for (int m = 0; m < MM; ++m) {
            if (m < a.M) {
              float fx[16];
              const __nv_bfloat16* xr = X + (long long)m * ldx + k + 16 * g;
              bf16x8_to_f32(*reinterpret_cast<const uint4*>(xr), fx);
              bf16x8_to_f32(*reinterpret_cast<const uint4*>(xr + 8), fx + 8);
#pragma unroll
              for (int r = 0; r < R; ++r) {
                float p = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) p = fmaf(fw[r][i], fx[i], p);
                acc[r][m] = fmaf(p, bs[r], acc[r][m]);
              }
            }
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
        if (a.Wr) {
          s0 *= a.Wr[nn];
          if (SWIGLU) s1 *= a.Wr[nn + a.pair_off];
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
        for (int j = 0; j < J; ++j) {
          w[r][j] = wn[r][j];
          sc[r][j] = scn[r][j];
        }
    }
  }
}

// ---------------------------------------------------------------- bulk-copy GEMV
// Up to 4 activation rows: the bulk-copy design of gemv_tma.cuh for packed
// weights.  Each CTA (one per SM) owns a contiguous range of features, so
// its code rows and its scale rows are two contiguous byte ranges (four for
// SwiGLU); warp 8 copies them stage by stage with cp.async.bulk into a
// shared-memory ring, issuing the first stages before the wait on the
// previous kernel.  Warps 0-7 take one feature each per stage: lane l
// decodes 16-byte chunks l, l + 32, ... of the code row and multiplies them
// with the activations, which are held in shared memory as fp32 in a
// chunk-interleaved order (float4 q of chunk c at [q][c]) so that the warp's
// loads of one instruction are consecutive.
constexpr int kGvqStageMax = 16384;

struct GvqGeom {
  int rb, sb;         // code / scale bytes of one row
  int per_stage;      // features per stage (<= 8)
  int stage_bytes;
  int stages;
  int xf_off;         // fp32 activations (M * K * 4 bytes)
  int ring_off;
};

__host__ __device__ inline GvqGeom gvq_geom(int fmt, int M, int K, bool swiglu, bool pre) {
  GvqGeom g;
  g.rb = fmt == QF_MXFP8 ? K : K / 2;
  g.sb = fmt == QF_MXFP8 ? K / 32 : K / 16;
  const int unit = (swiglu ? 2 : 1) * (g.rb + g.sb);
  const int r = kGvqStageMax / unit;
  g.per_stage = r < 1 ? 1 : (r > 8 ? 8 : r);
  g.stage_bytes = g.per_stage * unit;
  g.xf_off = pre ? (M * K * 2 + 1023) / 1024 * 1024 : 0;   // PRE: bf16 rows first
  g.ring_off = g.xf_off + (M * K * 4 + 1023) / 1024 * 1024;
  const int s = (kGvtSmem - g.ring_off - 1024) / g.stage_bytes;
  g.stages = s > 16 ? 16 : s;
  return g;
}

template <int FMT, int MM, bool SWIGLU, bool PRE>
__global__ void __launch_bounds__(kGvtThreads, 1) gemv_tma_q_kernel(const GemvArgs a, int* status) {
  constexpr int R = SWIGLU ? 2 : 1;
  constexpr int E = FMT == QF_MXFP8 ? 16 : 32;     // weights per 16-byte chunk
  constexpr int Q = E / 4;                         // float4 activations per chunk
  extern __shared__ __align__(1024) uint8_t gvq_smem[];
  const GvqGeom geo = gvq_geom(FMT, a.M, a.K, SWIGLU, PRE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = gvq_smem + geo.ring_off;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + geo.stages * geo.stage_bytes);
  uint64_t* empty = full + geo.stages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + geo.stages);
  const int f0 = (int)((long long)blockIdx.x * a.N / gridDim.x);
  const int f1 = (int)((long long)(blockIdx.x + 1) * a.N / gridDim.x);
  const int nf = f1 - f0;
  const int ps = geo.per_stage;
  const int n_stages = (nf + ps - 1) / ps;
  // stage layout: codes [ps][rb] (+ pair codes), then scales [ps][sb] (+ pair)
  const int off_s = R * ps * geo.rb;

  if (threadIdx.x == 0) {
    for (int s = 0; s < geo.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], ps);                  // one arrival per feature of the stage
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 8) {
    // ------------------------------------------------ producer: packed rows
    pdl_trigger();
    if (lane == 0) {
      for (int s = 0; s < n_stages && !*abort_flag; ++s) {
        const int slot = s % geo.stages;
        if (s >= geo.stages &&
            !mbar_wait_bounded(&empty[slot], ((s / geo.stages) - 1) & 1, status, DEV_GEMV_PRODUCER)) {
          *abort_flag = 1;
          break;
        }
        const long long u0 = f0 + s * ps;
        const int nu = min(ps, f1 - (int)u0);
        uint8_t* dst = ring + slot * geo.stage_bytes;
        const uint32_t cbytes = (uint32_t)(nu * geo.rb), sbytes = (uint32_t)(nu * geo.sb);
        mbar_arrive_expect_tx(&full[slot], R * (cbytes + sbytes));
        bulk_load(dst, a.Wq + u0 * geo.rb, cbytes, &full[slot]);
        bulk_load(dst + off_s, a.Ws + u0 * geo.sb, sbytes, &full[slot]);
        if (SWIGLU) {
          bulk_load(dst + ps * geo.rb, a.Wq + (u0 + a.pair_off) * geo.rb, cbytes, &full[slot]);
          bulk_load(dst + off_s + ps * geo.sb, a.Ws + (u0 + a.pair_off) * geo.sb, sbytes,
                    &full[slot]);
        }
      }
    }
    return;
  }

  // ------------------------------------------------ consumers (warps 0-7)
  pdl_wait();
  pdl_trigger();
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(gvq_smem);
  float4* xf = reinterpret_cast<float4*>(gvq_smem + geo.xf_off);
  const int nch = geo.rb / 16;                   // chunks per row
  if (PRE) gemv_pre_rows(a, xs);                 // warps 0-7
  named_bar(1, 256);
  // fp32 activations, chunk-interleaved: float4 q of chunk c of row m at
  // [m][q][c]
  for (int i = threadIdx.x; i < a.M * a.K / 4; i += 256) {
    const int m = i / (a.K / 4), qc = i % (a.K / 4);
    const int q = qc / nch, c = qc % nch;        // consecutive threads: consecutive c
    const int e4 = c * Q + q;
    const __nv_bfloat16* src = PRE ? xs + (long long)m * a.K + 4 * e4
                                   : a.X + (long long)m * a.ldx + 4 * e4;
    const uint2 v = *reinterpret_cast<const uint2*>(src);
    xf[((long long)m * Q + q) * nch + c] =
        make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                    __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
  }
  named_bar(1, 256);

  for (int j = warp; j < nf; j += 8) {
    const int s = j / ps, r = j % ps;
    const int slot = s % geo.stages;
    const bool ok = !*abort_flag && mbar_wait_bounded(&full[slot], (s / geo.stages) & 1, status,
                                                      DEV_GEMV_CONSUMER);
    if (!__all_sync(0xffffffffu, ok)) {
      *abort_flag = 1;
      break;
    }
    const uint8_t* stage = ring + slot * geo.stage_bytes;
    float acc[R][MM];
#pragma unroll
    for (int rr = 0; rr < R; ++rr)
#pragma unroll
      for (int m = 0; m < MM; ++m) acc[rr][m] = 0.f;
    for (int c = lane; c < nch; c += 32) {
#pragma unroll
      for (int rr = 0; rr < R; ++rr) {
        const uint8_t* crow = stage + (rr * ps + r) * geo.rb;
        const uint8_t* srow = stage + off_s + (rr * ps + r) * geo.sb;
        const uint4 wv = *reinterpret_cast<const uint4*>(crow + 16 * c);
        const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
        float bs[E / 16];
        if (FMT == QF_MXFP8) {
          bs[0] = e8m0_to_f32(srow[c >> 1]);
        } else {
          const uint32_t s2 = *reinterpret_cast<const unsigned short*>(srow + 2 * c);
          bs[0] = e4m3_to_f32(s2 & 0xFFu);
          bs[E / 16 - 1] = e4m3_to_f32(s2 >> 8);
        }
#pragma unroll
        for (int g = 0; g < E / 16; ++g) {       // 16 weights sharing one scale
          float fw[16];
          if (FMT == QF_MXFP8) {
#pragma unroll
            for (int q = 0; q < 4; ++q) e4m3x4_to_f32(w4[q], fw + 4 * q);
          } else {
            e2m1x8_to_f32(w4[2 * g], fw);
            e2m1x8_to_f32(w4[2 * g + 1], fw + 8);
          }
#pragma unroll
          for (int m = 0; m < MM; ++m) {
            if (m < a.M) {
              float p = 0.f;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float4 x = xf[((long long)m * Q + 4 * g + q) * nch + c];
                p = fmaf(fw[4 * q], x.x, p);
                p = fmaf(fw[4 * q + 1], x.y, p);
                p = fmaf(fw[4 * q + 2], x.z, p);
                p = fmaf(fw[4 * q + 3], x.w, p);
              }
              acc[rr][m] = fmaf(p, bs[g], acc[rr][m]);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);    // this feature's rows are consumed
    const int n = f0 + j;
#pragma unroll
    for (int m = 0; m < MM; ++m) {
      if (m < a.M) {
        float u = warp_sum(acc[0][m]);
        if (SWIGLU) {
          float v = warp_sum(acc[R - 1][m]);
          if (lane == 0) {
            if (a.Wr) {
              u *= a.Wr[n];
              v *= a.Wr[n + a.pair_off];
            }
            a.m_out[(long long)m * a.ldm + n] = __float2bfloat16_rn(u * (v / (1.0f + __expf(-v))));
          }
        } else if (lane == 0) {
          a.Y[(long long)m * a.ldy + n] =
              u * (a.Wr ? a.Wr[n] : 1.f) * (a.col_scale ? a.col_scale[n] : 1.f);
        }
      }
    }
  }
  if (*abort_flag) {
    for (int k = 0; k < 64; ++k) __nanosleep(1000);   // let in-flight copies land
  }
}

}  // namespace dory
