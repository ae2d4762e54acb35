// rowops.cuh - per-token kernels of the looped nGPT forward pass (HBM-bound):
// embedding gather + normalisation, the nGPT residual step, loop-boundary
// transforms, the KV-cache writer, the RoPE table and the greedy argmax.
//
// One CTA (128 threads) per token row; each thread owns up to 4 chunks of 8
// consecutive elements (d <= 4096), loaded and stored as 16/32-byte vectors;
// row sums of squares are reduced with warp shuffles and one shared-memory
// step.  Normalisation: N(v) = v / sqrt(max(sum v^2, 1e-12)).
#pragma once
#include "ptx.cuh"

namespace dory {

constexpr int kRowThreads = 128;
constexpr int kRowMaxChunks = 4;

enum : int { DEV_BAD_TOKEN = 0x21 };

__device__ __forceinline__ float block_sum128(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  return red[0] + red[1] + red[2] + red[3];
}

__device__ __forceinline__ void load8(const float* p, float* v) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void store8(float* p, const float* v) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void load8_bf16(const __nv_bfloat16* p, float* v) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void store8_bf16(__nv_bfloat16* p, const float* v) {
  uint4 u;
  u.x = pack_bf16x2(v[0], v[1]);
  u.y = pack_bf16x2(v[2], v[3]);
  u.z = pack_bf16x2(v[4], v[5]);
  u.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = u;
}

// h = N(E_in[token]); tokens [B, ld_tok], row = b * C + t.
__global__ void __launch_bounds__(kRowThreads) embed_kernel(const int32_t* tokens, int ld_tok,
                                                            int C, const __nv_bfloat16* E, int V,
                                                            int d, float* h32, __nv_bfloat16* hb,
                                                            int* status) {
  __shared__ float red[4];
  pdl_wait();
  pdl_trigger();
  const long long row = blockIdx.x;
  const int b = (int)(row / C), t = (int)(row % C);
  int tok = tokens[(long long)b * ld_tok + t];
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0 && status) atomicCAS(status, 0, DEV_BAD_TOKEN);
    tok = 0;
  }
  const int nch = d / 8;
  float v[kRowMaxChunks][8];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kRowMaxChunks; ++j) {
    const int ch = threadIdx.x + j * kRowThreads;
    if (ch < nch) {
      load8_bf16(E + (long long)tok * d + ch * 8, v[j]);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss += v[j][i] * v[j][i];
    }
  }
  const float inv = 1.0f / sqrtf(fmaxf(block_sum128(ss, red), 1e-12f));
#pragma unroll
  for (int j = 0; j < kRowMaxChunks; ++j) {
    const int ch = threadIdx.x + j * kRowThreads;
    if (ch < nch) {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[j][i] *= inv;
      store8(h32 + row * d + ch * 8, v[j]);
      store8_bf16(hb + row * d + ch * 8, v[j]);
    }
  }
}

// nGPT residual step ("Dory1.0-4B: A Looped Normalized-GPT", Architecture):
// h <- N(h + alpha * (N(y) - h)), y = the sublayer's projection output (the
// sum of n_parts partial sums part_stride apart; one part unless the
// projection was split along K).
__global__ void __launch_bounds__(kRowThreads) ngpt_update_kernel(float* h32, __nv_bfloat16* hb,
                                                                  const float* y,
                                                                  const float* alpha, int d,
                                                                  int n_parts,
                                                                  long long part_stride) {
  __shared__ float red[4];
  pdl_wait();
  pdl_trigger();
  const long long row = blockIdx.x;
  const int nch = d / 8;
  float yv[kRowMaxChunks][8];
  // h and alpha are loaded with y (one memory round trip before the first
  // reduction instead of two around it)
  float hv[kRowMaxChunks][8], av[kRowMaxChunks][8];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kRowMaxChunks; ++j) {
    const int ch = threadIdx.x + j * kRowThreads;
    if (ch < nch) {
      load8(h32 + row * d + ch * 8, hv[j]);
      load8(alpha + ch * 8, av[j]);
      load8(y + row * d + ch * 8, yv[j]);
      for (int p = 1; p < n_parts; ++p) {
        float t[8];
        load8(y + p * part_stride + row * d + ch * 8, t);
#pragma unroll
        for (int i = 0; i < 8; ++i) yv[j][i] += t[i];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) ss += yv[j][i] * yv[j][i];
    }
  }
  const float inv_y = 1.0f / sqrtf(fmaxf(block_sum128(ss, red), 1e-12f));
  float su = 0.f;
#pragma unroll
  for (int j = 0; j < kRowMaxChunks; ++j) {
    const int ch = threadIdx.x + j * kRowThreads;
    if (ch < nch) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float u = hv[j][i] + av[j][i] * (yv[j][i] * inv_y - hv[j][i]);
        yv[j][i] = u;
        su += u * u;
      }
    }
  }
  const float inv_u = 1.0f / sqrtf(fmaxf(block_sum128(su, red), 1e-12f));
#pragma unroll
  for (int j = 0; j < kRowMaxChunks; ++j) {
    const int ch = threadIdx.x + j * kRowThreads;
    if (ch < nch) {
#pragma unroll
      for (int i = 0; i < 8; ++i) yv[j][i] *= inv_u;
      store8(h32 + row * d + ch * 8, yv[j]);
      store8_bf16(hb + row * d + ch * 8, yv[j]);
    }
  }
}

// SwiGLU of split-K partial sums: y = [u | v] per row (2F columns, n_parts
// partials part_stride apart); m = u * SiLU(v) as bf16 [rows, F].
// grid = (ceil(F / 1024), rows), 128 threads x 8 columns.
__global__ void __launch_bounds__(kRowThreads) swiglu_parts_kernel(const float* y, int F,
                                                                   int n_parts,
                                                                   long long part_stride,
                                                                   __nv_bfloat16* m) {
  pdl_wait();
  pdl_trigger();
  const long long row = blockIdx.y;
  const int c0 = (blockIdx.x * kRowThreads + threadIdx.x) * 8;
  if (c0 >= F) return;
  float u[8], v[8];
  load8(y + row * 2 * F + c0, u);
  load8(y + row * 2 * F + F + c0, v);
  for (int p = 1; p < n_parts; ++p) {
    float tu[8], tv[8];
    load8(y + p * part_stride + row * 2 * F + c0, tu);
    load8(y + p * part_stride + row * 2 * F + F + c0, tv);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      u[i] += tu[i];
      v[i] += tv[i];
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) u[i] *= v[i] / (1.0f + __expf(-v[i]));
  store8_bf16(m + row * F + c0, u);
}

// Loop-boundary transforms ("Dory1.0-4B: A Looped Normalized-GPT", Training
// with Loops): the state starts as x; before each pass of the shared block
// the block input is N(s + x); the state after a pass is the normalised block
// output; the output block receives the final state.
enum BoundaryMode : int {
  BND_SAVE_X = 0,      // x = h (input block output); h is also s_0
  BND_ENTER_FIRST = 1, // h = N(s_0 + x) with s_0 = x held in h
  BND_ENTER_NEXT = 2,  // s = N(h); h = N(s + x)
  BND_EXIT = 3,        // h = N(h)  (final state s_k)
  BND_SAVE_ENTER = 4,  // x = h; h = N(x + x)  (BND_SAVE_X then BND_ENTER_FIRST)
};

// With y != null the row is first moved by the pending nGPT step of the last
// sublayer, h <- N(h + alpha * (N(y) - h)), y being that sublayer's
// projection output (n_parts partial sums part_stride apart).
// Per-sequence loop counts (kb != null, one row per sequence): at the
// boundary after loop `loop` a row whose count is `loop` saves its final
// state s into save (BND_ENTER_NEXT), and at the exit after the last loop a
// row whose count is below `loop` takes its saved state back (BND_EXIT), so
// the output block sees every row's s_(k_b).
__global__ void __launch_bounds__(kRowThreads) boundary_kernel(float* h32, __nv_bfloat16* hb,
                                                               float* x32, int d, int mode,
                                                               const float* y, int n_parts,
                                                               long long part_stride,
                                                               const float* alpha, const int* kb,
                                                               int loop, float* save) {
  __shared__ float red[4];
  pdl_wait();
  pdl_trigger();
  const long long row = blockIdx.x;
  const int nch = d / 8;
  float hv[kRowMaxChunks][8];
#pragma unroll
  for (int j = 0; j < kRowMaxChunks; ++j) {
    const int ch = threadIdx.x + j * kRowThreads;
    if (ch < nch) load8(h32 + row * d + ch * 8, hv[j]);
  }
  if (y != nullptr) {
    float yv[kRowMaxChunks][8];
    float sy = 0.f;
#pragma unroll
    for (int j = 0; j < kRowMaxChunks; ++j) {
      const int ch = threadIdx.x + j * kRowThreads;
      if (ch < nch) {
        load8(y + row * d + ch * 8, yv[j]);
        for (int p = 1; p < n_parts; ++p) {
          float t[8];
          load8(y + p * part_stride + row * d + ch * 8, t);
#pragma unroll
          for (int i = 0; i < 8; ++i) yv[j][i] += t[i];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) sy += yv[j][i] * yv[j][i];
      }
    }
    const float inv_y = 1.0f / sqrtf(fmaxf(block_sum128(sy, red), 1e-12f));
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kRowMaxChunks; ++j) {
      const int ch = threadIdx.x + j * kRowThreads;
      if (ch < nch) {
        float av[8];
        load8(alpha + ch * 8, av);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          hv[j][i] += av[i] * (yv[j][i] * inv_y - hv[j][i]);
          ss += hv[j][i] * hv[j][i];
        }
      }
    }
    const float inv = 1.0f / sqrtf(fmaxf(block_sum128(ss, red), 1e-12f));
#pragma unroll
    for (int j = 0; j < kRowMaxChunks; ++j)
#pragma unroll
      for (int i = 0; i < 8; ++i) hv[j][i] *= inv;
  }
  if (mode == BND_SAVE_X || mode == BND_SAVE_ENTER) {
#pragma unroll
    for (int j = 0; j < kRowMaxChunks; ++j) {
      const int ch = threadIdx.x + j * kRowThreads;
      if (ch < nch) store8(x32 + row * d + ch * 8, hv[j]);
    }
    if (mode == BND_SAVE_X) {
      if (y != nullptr) {
#pragma unroll
        for (int j = 0; j < kRowMaxChunks; ++j) {
          const int ch = threadIdx.x + j * kRowThreads;
          if (ch < nch) {
            store8(h32 + row * d + ch * 8, hv[j]);
            store8_bf16(hb + row * d + ch * 8, hv[j]);
          }
        }
      }
      return;
    }
  }
  if (mode == BND_ENTER_NEXT || mode == BND_EXIT) {
    float s2 = 0.f;
#pragma unroll
    for (int j = 0; j < kRowMaxChunks; ++j) {
      const int ch = threadIdx.x + j * kRowThreads;
      if (ch < nch) {
#pragma unroll
        for (int i = 0; i < 8; ++i) s2 += hv[j][i] * hv[j][i];
      }
    }
    const float inv = 1.0f / sqrtf(fmaxf(block_sum128(s2, red), 1e-12f));
#pragma unroll
    for (int j = 0; j < kRowMaxChunks; ++j)
#pragma unroll
      for (int i = 0; i < 8; ++i) hv[j][i] *= inv;
    if (kb) {
      const int krow = kb[row];
      const bool keep = mode == BND_ENTER_NEXT && krow == loop;
      const bool take = mode == BND_EXIT && krow != loop;
#pragma unroll
      for (int j = 0; j < kRowMaxChunks; ++j) {
        const int ch = threadIdx.x + j * kRowThreads;
        if (ch < nch) {
          if (keep) store8(save + row * d + ch * 8, hv[j]);
          if (take) load8(save + row * d + ch * 8, hv[j]);
        }
      }
    }
  }
  if (mode != BND_EXIT) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kRowMaxChunks; ++j) {
      const int ch = threadIdx.x + j * kRowThreads;
      if (ch < nch) {
        float xv[8];
        load8(x32 + row * d + ch * 8, xv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          hv[j][i] += xv[i];
          ss += hv[j][i] * hv[j][i];
        }
      }
    }
    const float inv = 1.0f / sqrtf(fmaxf(block_sum128(ss, red), 1e-12f));
#pragma unroll
    for (int j = 0; j < kRowMaxChunks; ++j)
#pragma unroll
      for (int i = 0; i < 8; ++i) hv[j][i] *= inv;
  }
#pragma unroll
  for (int j = 0; j < kRowMaxChunks; ++j) {
    const int ch = threadIdx.x + j * kRowThreads;
    if (ch < nch) {
      store8(h32 + row * d + ch * 8, hv[j]);
      store8_bf16(hb + row * d + ch * 8, hv[j]);
    }
  }
}

// KV-cache writer: positions P0 + t for t in [t_first, C) of every sequence
// go to ring slot (P0 + t) mod S of this layer/slice.  grid = (C - t_first, B),
// block covers n_kv * dh / 8 16-byte chunks (K and V).
__global__ void kv_write_kernel(const __nv_bfloat16* k_cur, const __nv_bfloat16* v_cur,
                                __nv_bfloat16* k_cache, __nv_bfloat16* v_cache, int C, int P0,
                                int S, int t_first, int n_kv, int dh) {
  pdl_wait();
  pdl_trigger();
  const int t = t_first + blockIdx.x, b = blockIdx.y;
  const int slot = (P0 + t) % S;
  const int cpr = dh / 8;
  for (int idx = threadIdx.x; idx < n_kv * cpr; idx += blockDim.x) {
    const int h = idx / cpr, c = idx % cpr;
    const long long src = (((long long)b * C + t) * n_kv + h) * dh + c * 8;
    const long long dst = (((long long)b * n_kv + h) * S + slot) * dh + c * 8;
    *reinterpret_cast<uint4*>(k_cache + dst) = *reinterpret_cast<const uint4*>(k_cur + src);
    *reinterpret_cast<uint4*>(v_cache + dst) = *reinterpret_cast<const uint4*>(v_cur + src);
  }
}

// RoPE tables for the positions of one call: tab_b[t][i] = (cos, sin) of
// (P0 + t) * base_b^(-2i/dh) for the two bases (b = 0: sliding-window
// layers, b = 1: full layers); the angle is formed and reduced mod 2 pi in
// fp64 so long contexts keep full fp32 accuracy.  tabt_b holds the same
// pairs transposed, two frequencies per 16 bytes: tabt_b[(i / 2) C + t]
// = pairs i & ~1 and i | 1 (coalesced reads across consecutive positions).
__global__ void rope_table_kernel(float2* tab0, float2* tab1, float2* tabt0, float2* tabt1, int C,
                                  int P0, int dh, double base0, double base1) {
  pdl_wait();
  pdl_trigger();
  const int half = dh / 2;
  const long long n = (long long)C * half;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < 2 * n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int which = idx >= n;
    const long long e = idx - which * n;
    const int t = (int)(e / half), i = (int)(e % half);
    const double inv_freq = pow(which ? base1 : base0, -2.0 * i / dh);
    double ang = (double)(P0 + t) * inv_freq;
    const double two_pi = 6.283185307179586476925286766559;
    ang -= floor(ang / two_pi) * two_pi;
    double s, c;
    sincos(ang, &s, &c);
    const float2 cs = make_float2((float)c, (float)s);
    (which ? tab1 : tab0)[e] = cs;
    (which ? tabt1 : tabt0)[((long long)(i >> 1) * C + t) * 2 + (i & 1)] = cs;
  }
}

// Ragged batches: the position of each sequence's new token (host values
// carried in the launch parameters).
constexpr int kRaggedMax = 128;
struct SeqPos {
  int p[kRaggedMax];       // positions
  int k[kRaggedMax];       // loop counts (per-sequence loop counts only)
};

// RoPE (cos, sin) rows of B sequences at their own positions (tab0: base0,
// tab1: base1, [B][dh / 2]; null tables when RoPE is off) and the positions
// themselves into pos_out [B] for the decode attention.
__global__ void rope_rows_kernel(float2* tab0, float2* tab1, const __grid_constant__ SeqPos sp,
                                 int B, int dh, double base0, double base1, int* pos_out,
                                 int* k_out) {
  pdl_wait();
  pdl_trigger();
  const int half = dh / 2;
  const long long n = (long long)B * half;
  if (blockIdx.x == 0)
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
      pos_out[b] = sp.p[b];
      if (k_out) k_out[b] = sp.k[b];
    }
  if (!tab0) return;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < 2 * n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int which = idx >= n;
    const long long e = idx - which * n;
    const int b = (int)(e / half), i = (int)(e % half);
    const double inv_freq = pow(which ? base1 : base0, -2.0 * i / dh);
    double ang = (double)sp.p[b] * inv_freq;
    const double two_pi = 6.283185307179586476925286766559;
    ang -= floor(ang / two_pi) * two_pi;
    double s, c;
    sincos(ang, &s, &c);
    (which ? tab1 : tab0)[e] = make_float2((float)c, (float)s);
  }
}

// Mixed steps: RoPE rows for Bd decode rows at sp.p[r] followed by C rows of
// one chunk at positions p_chunk + t, in both layouts of rope_table_kernel
// (the call's rows counted as M = Bd + C), and the decode rows' positions
// into pos_out.
__global__ void rope_mixed_kernel(float2* tab0, float2* tab1, float2* tabt0, float2* tabt1,
                                  const __grid_constant__ SeqPos sp, int Bd, int p_chunk, int C,
                                  int dh, double base0, double base1, int* pos_out) {
  pdl_wait();
  pdl_trigger();
  const int half = dh / 2, M = Bd + C;
  const long long n = (long long)M * half;
  if (blockIdx.x == 0)
    for (int b = threadIdx.x; b < Bd; b += blockDim.x) pos_out[b] = sp.p[b];
  if (!tab0) return;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < 2 * n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int which = idx >= n;
    const long long e = idx - which * n;
    const int r = (int)(e / half), i = (int)(e % half);
    const int pos = r < Bd ? sp.p[r] : p_chunk + (r - Bd);
    const double inv_freq = pow(which ? base1 : base0, -2.0 * i / dh);
    double ang = (double)pos * inv_freq;
    const double two_pi = 6.283185307179586476925286766559;
    ang -= floor(ang / two_pi) * two_pi;
    double s, c;
    sincos(ang, &s, &c);
    const float2 cs = make_float2((float)c, (float)s);
    (which ? tab1 : tab0)[e] = cs;
    (which ? tabt1 : tabt0)[((long long)(i >> 1) * M + r) * 2 + (i & 1)] = cs;
  }
}

// Greedy token per row: argmax of logits[row, 0..V), lowest index on ties.
__global__ void __launch_bounds__(1024) argmax_kernel(const float* logits, int V, int32_t* next) {
  __shared__ float bv[32];
  __shared__ int bi[32];
  pdl_wait();
  pdl_trigger();
  const long long row = blockIdx.x;
  const float* z = logits + row * V;
  float best = -INFINITY;
  int idx = 0x7fffffff;
  // 16-byte loads, four rows of them in flight per thread (V % 16 == 0);
  // within a thread indices grow, so "strictly greater" keeps the lowest
  const float4* z4 = reinterpret_cast<const float4*>(z);
  const int n4 = V / 4;
  for (int base = threadIdx.x; base < n4; base += 4 * blockDim.x) {
    float4 q[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i4 = base + u * blockDim.x;
      q[u] = i4 < n4 ? z4[i4] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = 4 * (base + u * blockDim.x);
      if (q[u].x > best) { best = q[u].x; idx = i; }
      if (q[u].y > best) { best = q[u].y; idx = i + 1; }
      if (q[u].z > best) { best = q[u].z; idx = i + 2; }
      if (q[u].w > best) { best = q[u].w; idx = i + 3; }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
    if (ov > best || (ov == best && oi < idx)) {
      best = ov;
      idx = oi;
    }
  }
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    bv[w] = best;
    bi[w] = idx;
  }
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x >> 5;
    best = threadIdx.x < nw ? bv[threadIdx.x] : -INFINITY;
    idx = threadIdx.x < nw ? bi[threadIdx.x] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
      if (ov > best || (ov == best && oi < idx)) {
        best = ov;
        idx = oi;
      }
    }
    if (threadIdx.x == 0) next[row] = idx == 0x7fffffff ? 0 : idx;
  }
}

// ------------------------------------------------------------------------
// Self-speculative decoding ("Dory1.0-4B: A Looped Normalized-GPT",
// Self-Speculative Decoding): drafts at a shallow loop count, one verifying
// forward pass at the deep one, greedy acceptance.

// One sliding-window cache block of the KV region: byte offsets of its K and
// V arrays ([max_batch][n_kv][slots][head_dim] bf16) and its ring size.
struct SpecRing {
  long long k_off, v_off;
  int slots, pad;
};

// Ring slots of positions L .. L + n_pos - 1 of every window block, for B
// sequences: dir 0 copies them from the KV region to `backup`, dir 1 back
// for the positions L + i with i >= *i0 (i0 null: all of them).  One
// 16-byte chunk per thread; rows are head_dim bf16.
__global__ void spec_ring_copy_kernel(uint8_t* kv, const SpecRing* blocks, int n_blocks, int B,
                                      int n_kv, int dh, int L, int n_pos, uint4* backup, int dir,
                                      const int* i0) {
  pdl_wait();
  pdl_trigger();
  const int cpr = dh / 8;                                        // 16-byte chunks per row
  const long long rows = (long long)n_blocks * 2 * B * n_kv * n_pos;
  const int first = i0 ? *i0 : 0;
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < rows * cpr;
       t += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(t % cpr);
    long long r = t / cpr;
    const int i = (int)(r % n_pos);
    r /= n_pos;
    const int kvh = (int)(r % n_kv);
    r /= n_kv;
    const int b = (int)(r % B);
    r /= B;
    const int which = (int)(r % 2);
    const int blk = (int)(r / 2);
    const SpecRing g = blocks[blk];
    uint4* row = reinterpret_cast<uint4*>(kv + (which ? g.v_off : g.k_off)) +
                 (((long long)b * n_kv + kvh) * g.slots + (L + i) % g.slots) * cpr + c;
    uint4* bk = backup + t;
    if (dir == 0)
      *bk = *row;
    else if (i >= first)
      *row = *bk;
  }
}

// The verifying pass's tokens: [B, gamma + 1] = the last emitted token, then
// the gamma drafts (drafts[j * B + b]).
__global__ void spec_gather_kernel(const int32_t* tokens, const int32_t* drafts, int B, int gamma,
                                   int32_t* vin) {
  pdl_wait();
  pdl_trigger();
  const int n = B * (gamma + 1);
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < n; t += gridDim.x * blockDim.x) {
    const int b = t / (gamma + 1), j = t % (gamma + 1);
    vin[t] = j == 0 ? tokens[b] : drafts[(j - 1) * B + b];
  }
}

// Greedy acceptance (one block): sequence b accepts a_b leading drafts, each
// equal to the verifier's greedy token at the position before it (g[b][j]:
// the verifier's token after position L + j).  The batch advances by
// n = min_b a_b + 1: out[b][j] = drafts[j][b] for j < n - 1, g[b][n - 1] at
// j = n - 1 (the verifier's token), -1 after; *n_out = n.
__global__ void spec_accept_kernel(const int32_t* drafts, const int32_t* g, int B, int gamma,
                                   int32_t* out, int* n_out) {
  __shared__ int s_min;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) s_min = gamma;
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    int a = 0;
    while (a < gamma && drafts[a * B + b] == g[b * (gamma + 1) + a]) ++a;
    atomicMin(&s_min, a);
  }
  __syncthreads();
  const int n = s_min + 1;
  for (int t = threadIdx.x; t < B * (gamma + 1); t += blockDim.x) {
    const int b = t / (gamma + 1), j = t % (gamma + 1);
    out[t] = j < n - 1 ? drafts[j * B + b] : (j == n - 1 ? g[t] : -1);
  }
  if (threadIdx.x == 0) *n_out = n;
}

// ------------------------------------------------------------------------
// Prefix caching: the cached keys and values of one sequence copied into
// other sequences of the same KV region.

constexpr int kKvCopyMaxBlocks = 1024;   // (layer, slice) pairs
constexpr int kKvCopyMaxDst = 256;

// Byte offset of each (layer, slice) K block ([max_batch][n_kv][slots][dh]
// bf16; the V block follows it), its ring size and the slots to copy.
struct KvCopyTable {
  int n_blocks, n_dst, src, max_batch;
  long long k_off[kKvCopyMaxBlocks];
  int slots[kKvCopyMaxBlocks];
  int rows[kKvCopyMaxBlocks];
  int dst[kKvCopyMaxDst];
};

// grid: x over (K/V, kv head, slot row, 16-byte chunk) of the largest block,
// y = block, z = destination.  Slots 0 .. rows-1 of the source sequence go to
// the same slots of the destination.
__global__ void kv_copy_kernel(uint8_t* kv, const __grid_constant__ KvCopyTable t, int n_kv,
                               int dh) {
  pdl_wait();
  pdl_trigger();
  const int blk = blockIdx.y, d = blockIdx.z;
  const int cpr = dh / 8;
  const int rows = t.rows[blk], slots = t.slots[blk];
  const long long total = 2ll * n_kv * rows * cpr;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int c = (int)(i % cpr);
  long long r = i / cpr;
  const int row = (int)(r % rows);
  r /= rows;
  const int kvh = (int)(r % n_kv);
  const int which = (int)(r / n_kv);
  const long long blk_bytes = (long long)t.max_batch * n_kv * slots * dh * 2;
  const uint4* base = reinterpret_cast<const uint4*>(kv + t.k_off[blk] + which * blk_bytes);
  uint4* dbase = reinterpret_cast<uint4*>(kv + t.k_off[blk] + which * blk_bytes);
  const long long src = (((long long)t.src * n_kv + kvh) * slots + row) * cpr + c;
  const long long dst = (((long long)t.dst[d] * n_kv + kvh) * slots + row) * cpr + c;
  dbase[dst] = base[src];
}

}  // namespace dory
