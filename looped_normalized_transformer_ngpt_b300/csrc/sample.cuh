// sample.cuh - temperature sampling and the rejection-sampling step of
// self-speculative decoding ("Dory1.0-4B: A Looped Normalized-GPT",
// Self-Speculative Decoding: drafts from a shallow loop count, one
// verifying pass at the full count, rejection sampling that keeps the
// verifier's distribution).
//
// Distributions are softmax(z / T) over the vocabulary.  A draw from
// non-negative weights w with uniform u is the smallest index x whose
// running sum w_0 + ... + w_x exceeds u * sum(w) (the last index with w > 0
// if rounding leaves none).  Draft x at a position is kept iff u * q(x) <
// p(x) (probability min(1, p / q)); the first rejected position is redrawn
// from max(0, p - q); if every draft is kept one more token is drawn from
// the verifier after the last draft; a batch advances by its smallest count
// of kept drafts plus one.  The uniforms are inputs.
//
// Running sums are formed in one fixed order (block_draw): warp w owns a
// contiguous range of the vocabulary, walked in steps of 32 elements (lane
// l holds element 32 s + l); a step's sum is the warp's butterfly sum and
// the warp's total the ordered sum of its steps, so the pass that locates
// the crossing step repeats the first pass's arithmetic exactly.
#pragma once
#include "ptx.cuh"

namespace dory {

constexpr int kSampleThreads = 1024;

__device__ __forceinline__ float block_reduce_max(float v, float* red) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) r = fmaxf(r, red[i]);
  return r;
}

__device__ __forceinline__ float block_reduce_sum(float v, float* red) {
  v = warp_sum(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) r += red[i];
  return r;
}

// The draw described above, by the whole block (1024 threads); w(x) >= 0.
template <class Wfn>
__device__ int block_draw(int V, float u, Wfn w) {
  __shared__ float s_tot[32];
  __shared__ float s_pre, s_target;
  __shared__ int s_warp, s_res;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = ((V + 31) / 32 + 31) / 32 * 32;          // elements per warp
  const int lo = warp * R, hi = min(V, lo + R);
  float run = 0.f;
  for (int base = lo; base < hi; base += 32) {
    const int x = base + lane;
    run += warp_sum(x < hi ? w(x) : 0.f);
  }
  if (lane == 0) s_tot[warp] = run;
  __syncthreads();
  if (threadIdx.x == 0) {
    float total = 0.f;
    for (int i = 0; i < 32; ++i) total += s_tot[i];
    const float target = u * total;
    float pre = 0.f;
    int W = -1;
    for (int i = 0; i < 32; ++i) {
      if (pre + s_tot[i] > target) {
        W = i;
        break;
      }
      pre += s_tot[i];
    }
    s_warp = W;
    s_pre = pre;
    s_target = target;
    s_res = -1;
  }
  __syncthreads();
  const int W = s_warp;
  if (W >= 0 && warp == W) {
    const float pre = s_pre, target = s_target;
    float r = 0.f;
    for (int base = lo; base < hi; base += 32) {
      const int x = base + lane;
      const float v = x < hi ? w(x) : 0.f;
      const float step = warp_sum(v);
      if (pre + (r + step) > target) {
        float incl = v;                                   // inclusive scan within the step
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, pre + (r + incl) > target);
        const unsigned pos = __ballot_sync(0xffffffffu, v > 0.f);
        if (lane == 0) s_res = base + (hit ? __ffs(hit) - 1 : 31 - __clz(pos));
        break;
      }
      r += step;
    }
  }
  __syncthreads();
  if (s_res < 0) {
    // rounding left no crossing: the last index with positive weight
    __shared__ int s_last;
    if (threadIdx.x == 0) s_last = -1;
    __syncthreads();
    int last = -1;
    for (int x = threadIdx.x; x < V; x += blockDim.x)
      if (w(x) > 0.f) last = x;
    if (last >= 0) atomicMax(&s_last, last);
    __syncthreads();
    if (threadIdx.x == 0) s_res = s_last < 0 ? 0 : s_last;
    __syncthreads();
  }
  return s_res;
}

// stats[row] = (max z, sum exp((z - max) / T)) of logits rows [rows][V].
__global__ void __launch_bounds__(kSampleThreads) row_stats_kernel(const float* logits, int V,
                                                                   float inv_t, float2* stats) {
  __shared__ float red[32];
  pdl_wait();
  pdl_trigger();
  const float* z = logits + (long long)blockIdx.x * V;
  float m = -INFINITY;
  for (int x = threadIdx.x; x < V; x += blockDim.x) m = fmaxf(m, z[x]);
  m = block_reduce_max(m, red);
  float s = 0.f;
  for (int x = threadIdx.x; x < V; x += blockDim.x) s += expf((z[x] - m) * inv_t);
  s = block_reduce_sum(s, red);
  if (threadIdx.x == 0) stats[blockIdx.x] = make_float2(m, s);
}

// One token per logits row [rows][V] drawn from softmax(z / T) with the
// uniform u[row * u_stride]; out[row].
__global__ void __launch_bounds__(kSampleThreads) sample_kernel(const float* logits, int V,
                                                                float inv_t, const float* u,
                                                                int u_stride, int32_t* out) {
  __shared__ float red[32];
  pdl_wait();
  pdl_trigger();
  const float* z = logits + (long long)blockIdx.x * V;
  float m = -INFINITY;
  for (int x = threadIdx.x; x < V; x += blockDim.x) m = fmaxf(m, z[x]);
  m = block_reduce_max(m, red);
  const float ub = u[(long long)blockIdx.x * u_stride];
  const int x = block_draw(V, ub, [&](int i) { return expf((z[i] - m) * inv_t); });
  if (threadIdx.x == 0) out[blockIdx.x] = x;
}

// Kept drafts per sequence (one block, a thread per sequence):
// verifier logits zp [B][gamma + 1][V] with stats sp, drafter logits zq
// [gamma][B][V] with stats sq, drafts [gamma][B], uniforms u [B][2 gamma + 1]
// (column gamma + i decides draft i).  kept[b] = leading kept drafts.
__global__ void spec_keep_kernel(const float* zp, const float2* sp, const float* zq,
                                 const float2* sq, const int32_t* drafts, const float* u, int B,
                                 int gamma, int V, float inv_t, int32_t* kept) {
  pdl_wait();
  pdl_trigger();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    int a = 0;
    while (a < gamma) {
      const int x = drafts[a * B + b];
      const long long rp = (long long)b * (gamma + 1) + a, rq = (long long)a * B + b;
      const float p = expf((zp[rp * V + x] - sp[rp].x) * inv_t) / sp[rp].y;
      const float q = expf((zq[rq * V + x] - sq[rq].x) * inv_t) / sq[rq].y;
      if (!(u[(long long)b * (2 * gamma + 1) + gamma + a] * q < p)) break;
      ++a;
    }
    kept[b] = a;
  }
}

// Emitted tokens (a block per sequence): n = min kept + 1; out[b][j] =
// drafts for j < n - 1; at j = n - 1 the kept draft, or a draw from
// max(0, p - q) at the first rejected position, or from the verifier after
// the last draft (uniform column 2 gamma); -1 after.  Block 0 writes n.
__global__ void __launch_bounds__(kSampleThreads) spec_emit_kernel(
    const float* zp, const float2* sp, const float* zq, const float2* sq, const int32_t* drafts,
    const float* u, const int32_t* kept, int B, int gamma, int V, float inv_t, int32_t* out,
    int* n_out) {
  __shared__ int s_n;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) {
    int mn = gamma;
    for (int b = 0; b < B; ++b) mn = min(mn, kept[b]);
    s_n = mn + 1;
  }
  __syncthreads();
  const int n = s_n, b = blockIdx.x, j = n - 1;
  int tok;
  if (kept[b] > j) {
    tok = drafts[j * B + b];
  } else {
    const float ub = u[(long long)b * (2 * gamma + 1) + 2 * gamma];
    const long long rp = (long long)b * (gamma + 1) + j;
    const float* p = zp + rp * V;
    const float mp = sp[rp].x, ip = 1.0f / sp[rp].y;
    if (j < gamma) {
      const long long rq = (long long)j * B + b;
      const float* q = zq + rq * V;
      const float mq = sq[rq].x, iq = 1.0f / sq[rq].y;
      tok = block_draw(V, ub, [&](int x) {
        return fmaxf(expf((p[x] - mp) * inv_t) * ip - expf((q[x] - mq) * inv_t) * iq, 0.f);
      });
    } else {
      tok = block_draw(V, ub, [&](int x) { return expf((p[x] - mp) * inv_t); });
    }
  }
  if (threadIdx.x == 0) {
    for (int t = 0; t <= gamma; ++t)
      out[(long long)b * (gamma + 1) + t] = t < j ? drafts[t * B + b] : (t == j ? tok : -1);
    if (b == 0) *n_out = n;
  }
}

}  // namespace dory
