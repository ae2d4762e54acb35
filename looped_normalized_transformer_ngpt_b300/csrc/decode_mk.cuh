// decode_mk.cuh - one decode step of the looped nGPT (a new token for each
// of B <= 16 sequences) as ONE persistent cooperative kernel.
//
// With few rows every projection streams its weights once and the attention
// reads a few MB of cache: each step of the layer is short and the cost of a
// decode step is the chain of dependent steps (about five per layer
// application: 240 at k = 4 for the small model).  Separate kernel launches
// pay a launch and a full-grid drain at every link of that chain; here one
// CTA per SM runs all of them, separated by grid barriers, and spends each
// barrier wait streaming the next step's weights:
//   * before a barrier every warp loads its first weight chunks of the next
//     projection into registers (weights never change during the step) and
//     thread 0 prefetches the CTA's later weight rows into L2 with bulk
//     prefetches, so the weight stream overlaps the barrier;
//   * the nGPT step owed by a projection is formed by every CTA from the
//     projection output in the next projection's prologue (or by the row
//     phase of a loop boundary), as in the multi-kernel path;
//   * attention work items (sequence, kv head, key split) end with an atomic
//     ticket; the last item of a (sequence, kv head) merges the splits with
//     the new token's own key / value and writes the gated output.
//
// Schedule ("Dory1.0-4B: A Looped Normalized-GPT", Training with Loops;
// Last-Loop KV Caching): embedding, input layers, for i = 1..k a boundary
// (save x and enter / re-inject) and the recurrent layers (cache slice i-1
// in per-loop mode, stored every loop; slice 0 stored at loop k only in
// last-loop mode), the exit boundary, output layers, the final nGPT step,
// the LM head and the greedy argmax.
//
// Grid barriers are a counter plus a generation word in the workspace; a
// wait gives up after kWaitLimitNs, sets the status word and an abort flag,
// and every CTA leaves at its next barrier (waiting first for its own copies
// in flight).  The launch is cooperative, so all CTAs are co-resident.
#pragma once
#include "attn.cuh"
#include "gemv.cuh"
#include "rowops.cuh"

namespace dory {

enum : int { DEV_MK_BARRIER = 0x31 };

constexpr int kMkThreads = 256, kMkWarps = 8;
constexpr int kMkTile = 128;          // keys per attention tile: 8 warps x 16
constexpr int kMkStages = 2;
constexpr int kMkMaxD = 2048;         // row phases: one 8-element chunk per thread
constexpr int kMkMaxSplits = 64;

// Per-layer device table (built at bind time in the workspace).
struct MkLayer {
  const __nv_bfloat16 *w_qkvg, *w_o, *w_upgate, *w_down;
  const float *alpha_attn, *alpha_mlp, *s_qk;
  __nv_bfloat16* kv;       // K block of slice 0; V block at kv + blk; slice s at kv + 2 s blk
  long long blk;           // elements of one K (or V) block
  int S, full;
};

struct MkArgs {
  const MkLayer* layers;
  int n_in, n_rec, n_out, d, n_q, n_kv, ffn, vocab, window;
  int B, P0, k, per_loop;
  float scale_log2;
  const int32_t* tokens;
  const __nv_bfloat16* embed_in;
  const __nv_bfloat16* embed_out;
  const float* s_z;
  float* logits;            // [B, vocab] or null (then no LM head / argmax)
  int32_t* next;            // [B] or null
  float* h0;                // hidden state, two buffers [B, d]; the step ends in h0
  float* h1;
  float* x32;               // loop injection x [B, d]
  __nv_bfloat16* hb;        // bf16 hidden rows for projections without a fused step
  float* y32;               // O / down projection output [B, d]
  float* gy;                // QKV + gate projection output [B, nqkvg]
  __nv_bfloat16* att;       // gated attention output [B, n_q dh]
  __nv_bfloat16* mo;        // SwiGLU output [B, ffn]
  const float2* rope_swa;   // [dh / 2] (cos, sin) of position P0, or null (no RoPE)
  const float2* rope_full;
  float* part_o;            // [B, n_q, kMkMaxSplits, dh]
  float* part_ml;           // [B, n_q, kMkMaxSplits, 2]
  int* counter;             // [B * n_kv] tickets, zero between uses
  unsigned* bar;            // [0] arrivals, [1] generation
  int* abort_flag;
  int* status;
};

// ------------------------------------------------------------------ helpers
__device__ __forceinline__ float mk_block_sum(float v, float* red) {
  v = warp_sum(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kMkWarps; ++i) s += red[i];
  return s;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned atom_add_acqrel_u32(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void st_relaxed_u32(unsigned* p, unsigned v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void l2_prefetch_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Grid barrier.  The CTA's writes are ordered before thread 0's arrival by
// the CTA barrier; the arrival is an acquire-release add, the last arriver
// resets the count and publishes the new generation with a release store,
// the others poll it with acquire loads.  Returns false when the step is
// being abandoned (a wait expired here or elsewhere).
__device__ __forceinline__ bool mk_sync(const MkArgs& a, unsigned& gen) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned target = gen + 1;
    int ok = 1;
    if (atom_add_acqrel_u32(&a.bar[0], 1u) == gridDim.x - 1) {
      st_relaxed_u32(&a.bar[0], 0u);
      st_release_u32(&a.bar[1], target);
    } else {
      const unsigned long long t0 = globaltimer();
      uint32_t n = 0;
      while (ld_acquire_u32(&a.bar[1]) != target) {
        if ((++n & 255u) == 0) {
          if (*reinterpret_cast<volatile int*>(a.abort_flag) ||
              globaltimer() - t0 > kWaitLimitNs) {
            atomicCAS(a.status, 0, DEV_MK_BARRIER);
            atomicExch(a.abort_flag, 1);
            ok = 0;
            break;
          }
        }
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  gen += 1;
  return s_ok != 0;
}

// ------------------------------------------------------------ row phases
// CTA b < B works on row b; thread t owns elements 8t .. 8t+7 (t < d / 8).

// v = N(h + alpha * (N(y) - h)) for this thread's chunk (y = null: v = h).
__device__ __forceinline__ void mk_row_step(const float* h, const float* y, const float* alpha,
                                            int d, float* v, float* red) {
  const int ch = threadIdx.x;
  const bool own = ch < d / 8;
  if (own) ld8f(h + ch * 8, v);
  if (y == nullptr) return;
  float yv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float sy = 0.f;
  if (own) {
    ld8f(y + ch * 8, yv);
#pragma unroll
    for (int i = 0; i < 8; ++i) sy += yv[i] * yv[i];
  }
  const float inv_y = 1.0f / sqrtf(fmaxf(mk_block_sum(sy, red), 1e-12f));
  float su = 0.f;
  if (own) {
    float al[8];
    ld8f(alpha + ch * 8, al);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[i] += al[i] * (yv[i] * inv_y - v[i]);
      su += v[i] * v[i];
    }
  }
  const float inv = 1.0f / sqrtf(fmaxf(mk_block_sum(su, red), 1e-12f));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] *= inv;
}

__device__ __forceinline__ void mk_row_normalize(float* v, int d, float* red) {
  float s = 0.f;
  if (threadIdx.x < d / 8) {
#pragma unroll
    for (int i = 0; i < 8; ++i) s += v[i] * v[i];
  }
  const float inv = 1.0f / sqrtf(fmaxf(mk_block_sum(s, red), 1e-12f));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] *= inv;
}

__device__ __forceinline__ void mk_row_store(float* h, __nv_bfloat16* hb, int d, const float* v) {
  const int ch = threadIdx.x;
  if (ch < d / 8) {
    store8(h + ch * 8, v);
    store8_bf16(hb + ch * 8, v);
  }
}

// ------------------------------------------------------------ projections
struct MkGemv {
  const __nv_bfloat16* W;
  int N, K, S, J, fpi, n_iters, pair_off;
};

__device__ __forceinline__ MkGemv mk_gemv_cfg(const __nv_bfloat16* W, int N, int K, bool swiglu) {
  MkGemv g;
  g.W = W;
  g.N = N;
  g.K = K;
  g.pair_off = swiglu ? N : 0;
  const int jmax = swiglu ? 4 : 8;
  const int kc = (K + 255) / 256;
  int S = 1;
  while ((kc + S - 1) / S > jmax && S < kMkWarps) S *= 2;
  g.S = S;
  g.J = (kc + S - 1) / S;
  g.fpi = kMkWarps / S;
  g.n_iters = (N + g.fpi - 1) / g.fpi;
  return g;
}

// This warp's weight chunks of CTA iteration `it` (zeros when out of range):
// w[j] (j < J <= 8), or for SwiGLU W_up chunks in w[0..3] and W_sl chunks in
// w[4..7] (J <= 4).
template <bool SW>
__device__ __forceinline__ void mk_gemv_load(const MkGemv& g, int it, uint4 (&w)[8]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = it * g.fpi + warp / g.S;
  const int kbase = (warp % g.S) * (g.J * 256) + lane * 8;
  const bool valid = it < g.n_iters && n < g.N;
  constexpr int JM = SW ? 4 : 8;
#pragma unroll
  for (int r = 0; r < (SW ? 2 : 1); ++r) {
    const __nv_bfloat16* wr = g.W + (long long)(valid ? n + r * g.pair_off : 0) * g.K;
#pragma unroll
    for (int j = 0; j < JM; ++j) {
      const int k = kbase + j * 256;
      w[r * JM + j] =
          (valid && j < g.J && k < g.K) ? ld_stream16(wr + k) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// Register prefetch before a barrier: this CTA's first iteration into w and,
// when a non-SwiGLU row fits in four chunks, its second into w2; bulk L2
// prefetch of the next few iterations.
template <bool SW>
__device__ __forceinline__ void mk_gemv_prefetch(const MkGemv& g, uint4 (&w)[8], uint4 (&w2)[4],
                                                 int n_l2) {
  mk_gemv_load<SW>(g, blockIdx.x, w);
  int skip = 0;
  if (!SW && g.J <= 4) {
    uint4 t[8];
    mk_gemv_load<false>(g, blockIdx.x + gridDim.x, t);
#pragma unroll
    for (int j = 0; j < 4; ++j) w2[j] = t[j];
    skip = 1;
  }
  if (threadIdx.x == 0) {
    for (int i = 1 + skip; i <= n_l2 + skip; ++i) {
      const int it = blockIdx.x + i * gridDim.x;
      if (it >= g.n_iters) break;
      const int n0 = it * g.fpi;
      const int rows = min(g.fpi, g.N - n0);
#pragma unroll
      for (int r = 0; r < (SW ? 2 : 1); ++r)
        l2_prefetch_bulk(g.W + (long long)(n0 + r * g.pair_off) * g.K, (uint32_t)rows * g.K * 2);
    }
  }
}

// Y[m, n] (or m_out for SwiGLU) for all CTA iterations of this CTA; the first
// iteration's weights are already in w.  X: M rows of K bf16 (smem or
// global, 16-byte aligned rows, ldx elements apart).
template <int MM, bool SW>
__device__ void mk_gemv_run(const MkGemv& g, uint4 (&w)[8], const uint4 (&w2)[4],
                            const __nv_bfloat16* X, int ldx, int M, float* Y, int ldy,
                            const float* col_scale, __nv_bfloat16* m_out, int ldm,
                            float* red /* [8][2][MM] */) {
  constexpr int R = SW ? 2 : 1, JM = SW ? 4 : 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kbase = (warp % g.S) * (g.J * 256) + lane * 8;
  for (int it = blockIdx.x; it < g.n_iters; it += gridDim.x) {
    if (it != blockIdx.x) {
      if (!SW && g.J <= 4 && it == blockIdx.x + gridDim.x) {
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = w2[j];      // second iteration: prefetched too
      } else {
        mk_gemv_load<SW>(g, it, w);
      }
    }
    const int n = it * g.fpi + warp / g.S;
    const bool valid = n < g.N;
    float acc[R][MM];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MM; ++m) acc[r][m] = 0.f;
#pragma unroll
    for (int j = 0; j < JM; ++j) {
      const int k = kbase + j * 256;
      if (valid && j < g.J && k < g.K) {
        float fw[R][8];
#pragma unroll
        for (int r = 0; r < R; ++r) bf16x8_to_f32(w[r * JM + j], fw[r]);
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
        if (lane == 0) red[(warp * 2 + r) * MM + m] = v;
      }
    __syncthreads();
    const int t = threadIdx.x;
    if (t < g.fpi * MM) {
      const int rl = t / MM, m = t % MM;
      const int nn = it * g.fpi + rl;
      if (nn < g.N && m < M) {
        float s0 = 0.f, s1 = 0.f;
        for (int sg = 0; sg < g.S; ++sg) {
          s0 += red[((rl * g.S + sg) * 2) * MM + m];
          if (SW) s1 += red[((rl * g.S + sg) * 2 + 1) * MM + m];
        }
        if (SW)
          m_out[(long long)m * ldm + nn] = __float2bfloat16_rn(s0 * (s1 / (1.0f + __expf(-s1))));
        else
          Y[(long long)m * ldy + nn] = s0 * (col_scale ? col_scale[nn] : 1.f);
      }
    }
    __syncthreads();
  }
}

// Activation rows formed in shared memory by the owed nGPT step: warp w
// forms rows w, w + 8, ...; CTA 0 also stores them as the next hidden state.
__device__ void mk_pre_rows(const float* h_in, const float* y, const float* alpha, int d, int M,
                            __nv_bfloat16* xs, float* h_out) {
  constexpr int MAXC = kMkMaxD / 256;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nch = d / 8;
  for (int m = warp; m < M; m += kMkWarps) {
    float u[MAXC][8];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < MAXC; ++j) {
      const int ch = lane + 32 * j;
      if (ch < nch) {
        ld8f(y + (long long)m * d + ch * 8, u[j]);
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
        ld8f(h_in + (long long)m * d + ch * 8, h);
        ld8f(alpha + ch * 8, al);
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
        store8_bf16(xs + (long long)m * d + ch * 8, u[j]);
        if (blockIdx.x == 0) store8(h_out + (long long)m * d + ch * 8, u[j]);
      }
    }
  }
}

// ------------------------------------------------------------ attention
template <int DH>
struct MkAttnCfg {
  static constexpr int QB = 16 * DH * 2;
  static constexpr int KVB = kMkTile * DH * 2;
  static constexpr int STAGE = 2 * KVB;
  static constexpr int MERGE = kMkWarps * 16 * DH * 4;
  static constexpr int RING = kMkStages * STAGE > MERGE ? kMkStages * STAGE : MERGE;
  static constexpr int SMEM = QB + RING + 2 * DH * 4 + 2 * kMkWarps * 16 * 4 + 64;
};

// Number of key splits of one (sequence, kv head) for a layer (same on
// every CTA): enough items for the grid, at least two tiles per split.
__device__ __forceinline__ void mk_splits(const MkArgs& a, int n_cache, int& n_splits,
                                          int& chunk) {
  int sp = (int)((gridDim.x + a.B * a.n_kv - 1) / (a.B * a.n_kv));
  if (sp > kMkMaxSplits) sp = kMkMaxSplits;
  if (sp < 1) sp = 1;
  chunk = (n_cache + sp - 1) / sp;
  chunk = (chunk + kMkTile - 1) / kMkTile * kMkTile;
  if (chunk < 2 * kMkTile) chunk = 2 * kMkTile;
  n_splits = n_cache > 0 ? (n_cache + chunk - 1) / chunk : 1;
}

template <int DH>
__device__ void mk_attention(const MkArgs& a, const MkLayer& L, int slice, int store,
                             uint8_t* smem) {
  using Cf = MkAttnCfg<DH>;
  constexpr int CH = DH / 8, HALF = DH / 2, NE = (HALF + 31) / 32;
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem);
  uint8_t* ring = smem + Cf::QB;
  float* sKc = reinterpret_cast<float*>(ring + Cf::RING);
  float* sVc = sKc + DH;
  float* sM = sVc + DH;                          // [8][16]
  float* sL = sM + kMkWarps * 16;                // [8][16]
  int* sFlag = reinterpret_cast<int*>(sL + kMkWarps * 16);
  float* sCur = reinterpret_cast<float*>(sFlag + 1);   // [8]
  const uint32_t sQa = smem_u32(sQ), ringa = smem_u32(ring);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.n_q / a.n_kv;
  const int P0 = a.P0;
  const int window = L.full ? 0 : a.window;
  const int lo = window > 0 ? max(0, P0 - window + 1) : 0;
  int NS, chunk;
  mk_splits(a, P0 - lo, NS, chunk);
  const int nqkvg = (2 * a.n_q + 2 * a.n_kv) * DH;
  const __nv_bfloat16* kc = L.kv + 2 * (long long)slice * L.blk;
  const __nv_bfloat16* vc = kc + L.blk;
  const float2* rope = L.full ? a.rope_full : a.rope_swa;
  const int n_items = a.B * a.n_kv * NS;

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int split = item % NS, kvh = (item / NS) % a.n_kv, b = item / (NS * a.n_kv);
    const int k0 = lo + split * chunk;
    const int k1 = min(k0 + chunk, P0);
    const int ntiles = k1 > k0 ? (k1 - k0 + kMkTile - 1) / kMkTile : 0;
    auto load_tile = [&](int t, int buf) {
      const int j0 = k0 + t * kMkTile;
      const uint32_t kb = ringa + (uint32_t)(buf * Cf::STAGE), vb = kb + Cf::KVB;
      for (int idx = tid; idx < kMkTile * CH; idx += kMkThreads) {
        const int r = idx / CH, c = idx % CH;
        const int j = j0 + r;
        const bool ok = j < k1;
        const long long off = ok ? (((long long)b * a.n_kv + kvh) * L.S + (j % L.S)) * DH + c * 8 : 0;
        cp_async16(kb + swz_off<DH>(r, c), kc + off, ok);
        cp_async16(vb + swz_off<DH>(r, c), vc + off, ok);
      }
    };
    __syncthreads();                               // smem free (previous item)
    if (ntiles > 0) load_tile(0, 0);
    cp_async_commit();

    // prologue: q^ rows of sQ, current k^ / v
    for (int idx = tid; idx < 16 * CH; idx += kMkThreads) {
      const int r = idx / CH, c = idx % CH;
      if (r >= G) *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(sQ) + swz_off<DH>(r, c)) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    for (int hh = warp; hh < G + 2; hh += kMkWarps) {
      const int col0 = hh < G ? (kvh * G + hh) * DH
                              : (hh == G ? (a.n_q + kvh) * DH : (a.n_q + a.n_kv + kvh) * DH);
      const float* yr = a.gy + (long long)b * nqkvg + col0;
      float x1[NE], x2[NE];
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < NE; ++e) {
        const int i = lane + 32 * e;
        x1[e] = i < HALF ? yr[i] : 0.f;
        x2[e] = i < HALF ? yr[i + HALF] : 0.f;
        ss += x1[e] * x1[e] + x2[e] * x2[e];
      }
      if (hh <= G) {
        const float inv = 1.0f / sqrtf(fmaxf(warp_sum(ss), 1e-12f));
#pragma unroll
        for (int e = 0; e < NE; ++e) {
          const int i = lane + 32 * e;
          if (i < HALF) {
            float c1 = x1[e], c2 = x2[e];
            if (rope) {
              const float2 cs = rope[i];
              c1 = x1[e] * cs.x - x2[e] * cs.y;
              c2 = x2[e] * cs.x + x1[e] * cs.y;
            }
            x1[e] = c1 * inv * L.s_qk[i];
            x2[e] = c2 * inv * L.s_qk[i + HALF];
          }
        }
      }
#pragma unroll
      for (int e = 0; e < NE; ++e) {
        const int i = lane + 32 * e;
        if (i >= HALF) continue;
        const __nv_bfloat16 b1 = __float2bfloat16_rn(x1[e]), b2 = __float2bfloat16_rn(x2[e]);
        if (hh < G) {
          sQ[(swz_off<DH>(hh, i / 8) >> 1) + (i & 7)] = b1;
          sQ[(swz_off<DH>(hh, (i + HALF) / 8) >> 1) + (i & 7)] = b2;
        } else {
          float* dst = hh == G ? sKc : sVc;
          dst[i] = __bfloat162float(b1);
          dst[i + HALF] = __bfloat162float(b2);
          if (store && split == 0) {
            __nv_bfloat16* cache = const_cast<__nv_bfloat16*>(hh == G ? kc : vc);
            const long long off = (((long long)b * a.n_kv + kvh) * L.S + (P0 % L.S)) * DH;
            cache[off + i] = b1;
            cache[off + i + HALF] = b2;
          }
        }
      }
    }
    __syncthreads();

    const int g = lane >> 2, t4 = lane & 3;
    uint32_t qf[DH / 16][4];
#pragma unroll
    for (int kk = 0; kk < DH / 16; ++kk) {
      const int r = lane & 15;
      const int c = 2 * kk + (lane >> 4);
      ldsm_x4(sQa + swz_off<DH>(r, c), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
    }
    float o[DH / 8][4];
#pragma unroll
    for (int i = 0; i < DH / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

    for (int t = 0; t < ntiles; ++t) {
      if (t + 1 < ntiles) load_tile(t + 1, (t + 1) & 1);
      cp_async_commit();
      cp_async_wait<1>();
      __syncthreads();
      const uint32_t kbase = ringa + (uint32_t)((t & 1) * Cf::STAGE);
      const uint32_t vbase = kbase + Cf::KVB;
      float s[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        const int key = 16 * warp + (lane & 7) + ((lane >> 4) & 1) * 8;
        const int c = 2 * kk + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + swz_off<DH>(key, c), b0, b1, b2, b3);
        mma_bf16_16816(s[0], qf[kk], b0, b1);
        mma_bf16_16816(s[1], qf[kk], b2, b3);
      }
      const int j0 = k0 + t * kMkTile + 16 * warp;
      float corr[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int j = j0 + 8 * nt + 2 * t4 + e;
            float v = s[nt][2 * h + e] * a.scale_log2;
            v = j < k1 ? v : -INFINITY;
            s[nt][2 * h + e] = v;
            mx = fmaxf(mx, v);
          }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run[h], mx);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        corr[h] = exp2f(m_run[h] - m_use);
        m_run[h] = m_new;
        float ls = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float p = exp2f(s[nt][2 * h + e] - m_use);
            s[nt][2 * h + e] = p;
            ls += p;
          }
        l_run[h] = l_run[h] * corr[h] + ls;
      }
#pragma unroll
      for (int i = 0; i < DH / 8; ++i) {
        o[i][0] *= corr[0];
        o[i][1] *= corr[0];
        o[i][2] *= corr[1];
        o[i][3] *= corr[1];
      }
      uint32_t pa[4];
      pa[0] = pack_bf16x2(s[0][0], s[0][1]);
      pa[1] = pack_bf16x2(s[0][2], s[0][3]);
      pa[2] = pack_bf16x2(s[1][0], s[1][1]);
      pa[3] = pack_bf16x2(s[1][2], s[1][3]);
#pragma unroll
      for (int dp = 0; dp < DH / 16; ++dp) {
        const int key = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = 2 * dp + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vbase + swz_off<DH>(key, c), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * dp], pa, b0, b1);
        mma_bf16_16816(o[2 * dp + 1], pa, b2, b3);
      }
      __syncthreads();                             // buffer t & 1 is refilled next
    }
    cp_async_wait<0>();
    __syncthreads();

    // merge the 8 warps and store this split's partial
    float* sO = reinterpret_cast<float*>(ring);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float l = l_run[h];
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      const int r = g + 8 * h;
      if (t4 == 0) {
        sM[warp * 16 + r] = m_run[h];
        sL[warp * 16 + r] = l;
      }
#pragma unroll
      for (int nt = 0; nt < DH / 8; ++nt) {
        const int dim = 8 * nt + 2 * t4;
        *reinterpret_cast<float2*>(sO + (warp * 16 + r) * DH + dim) =
            make_float2(o[nt][2 * h], o[nt][2 * h + 1]);
      }
    }
    __syncthreads();
    for (int idx = tid; idx < G * DH; idx += kMkThreads) {
      const int r = idx / DH, dd = idx % DH;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kMkWarps; ++w) M = fmaxf(M, sM[w * 16 + r]);
      float Ls = 0.f, acc = 0.f;
#pragma unroll
      for (int w = 0; w < kMkWarps; ++w) {
        const float wt = sM[w * 16 + r] == -INFINITY ? 0.f : exp2f(sM[w * 16 + r] - M);
        Ls += sL[w * 16 + r] * wt;
        acc += sO[(w * 16 + r) * DH + dd] * wt;
      }
      const long long base = ((long long)b * a.n_q + kvh * G + r) * kMkMaxSplits + split;
      a.part_o[base * DH + dd] = acc;
      if (dd == 0) {
        a.part_ml[base * 2] = M;
        a.part_ml[base * 2 + 1] = Ls;
      }
    }

    // ticket: the last split of (b, kvh) merges all of them + the new token
    __threadfence();
    __syncthreads();
    if (tid == 0) *sFlag = atomicAdd(&a.counter[b * a.n_kv + kvh], 1) == NS - 1;
    __syncthreads();
    if (!*sFlag) continue;
    __threadfence();
    for (int r = warp; r < G; r += kMkWarps) {
      float acc = 0.f;
      for (int i = lane; i < DH; i += 32)
        acc += __bfloat162float(sQ[(swz_off<DH>(r, i / 8) >> 1) + (i & 7)]) * sKc[i];
      acc = warp_sum(acc);
      if (lane == 0) sCur[r] = acc * a.scale_log2;
    }
    __syncthreads();
    float* sW = reinterpret_cast<float*>(ring);    // [G][NS + 1]
    for (int r = warp; r < G; r += kMkWarps) {
      const long long bh = (long long)b * a.n_q + kvh * G + r;
      float mx = sCur[r];
      for (int sp = lane; sp < NS; sp += 32)
        mx = fmaxf(mx, __ldcg(a.part_ml + (bh * kMkMaxSplits + sp) * 2));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      float Ls = 0.f;
      for (int sp = lane; sp < NS; sp += 32) {
        const float ms = __ldcg(a.part_ml + (bh * kMkMaxSplits + sp) * 2);
        const float wt = ms == -INFINITY ? 0.f : exp2f(ms - mx);
        sW[r * (NS + 1) + sp] = wt;
        Ls += __ldcg(a.part_ml + (bh * kMkMaxSplits + sp) * 2 + 1) * wt;
      }
      Ls = warp_sum(Ls);
      if (lane == 0) {
        const float wc = exp2f(sCur[r] - mx);
        sW[r * (NS + 1) + NS] = wc;
        sM[r] = 1.0f / (Ls + wc);
      }
    }
    __syncthreads();
    for (int idx = tid; idx < G * DH; idx += kMkThreads) {
      const int r = idx / DH, dd = idx % DH;
      const long long bh = (long long)b * a.n_q + kvh * G + r;
      const float* wr = sW + r * (NS + 1);
      const float* po = a.part_o + bh * kMkMaxSplits * DH + dd;
      float acc = wr[NS] * sVc[dd];
      int sp = 0;
      for (; sp + 4 <= NS; sp += 4) {
        const float o0 = __ldcg(po + (sp + 0) * DH), o1 = __ldcg(po + (sp + 1) * DH);
        const float o2 = __ldcg(po + (sp + 2) * DH), o3 = __ldcg(po + (sp + 3) * DH);
        acc += wr[sp] * o0 + wr[sp + 1] * o1 + wr[sp + 2] * o2 + wr[sp + 3] * o3;
      }
      for (; sp < NS; ++sp) acc += wr[sp] * __ldcg(po + sp * DH);
      const float gr = a.gy[(long long)b * nqkvg + (long long)(a.n_q + 2 * a.n_kv) * DH +
                            (kvh * G + r) * DH + dd];
      const float gt = 1.0f / (1.0f + __expf(-gr));
      a.att[bh * DH + dd] = __float2bfloat16_rn(acc * sM[r] * gt);
    }
    if (tid == 0) a.counter[b * a.n_kv + kvh] = 0;
  }
  cp_async_wait<0>();
}

// ------------------------------------------------------------ the kernel
template <int MM, int DH>
__global__ void __launch_bounds__(kMkThreads, 1) decode_step_kernel(const MkArgs a) {
  extern __shared__ __align__(128) uint8_t mk_smem[];
  __shared__ float red[kMkWarps * 2 * MM];
  __shared__ float rsum[kMkWarps];
  unsigned gen = ld_acquire_u32(&a.bar[1]);
  const int d = a.d, B = a.B;
  const int hq = a.n_q * DH, nqkvg = (2 * a.n_q + 2 * a.n_kv) * DH;
  const int n_apps = a.n_in + a.k * a.n_rec + a.n_out;
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(mk_smem);
  uint4 w[8], w2[4];

  // the layer application `ap`: layer, cache slice, store flag and the
  // boundary transform that precedes it (-1: none)
  auto app = [&](int ap, int& l, int& slice, int& store, int& bnd) {
    bnd = -1;
    slice = 0;
    store = 1;
    if (ap < a.n_in) {
      l = ap;
    } else if (ap < a.n_in + a.k * a.n_rec) {
      const int r = ap - a.n_in, i = r / a.n_rec + 1;
      l = a.n_in + r % a.n_rec;
      slice = a.per_loop ? i - 1 : 0;
      store = a.per_loop || i == a.k;
      if (r % a.n_rec == 0) bnd = i == 1 ? BND_SAVE_ENTER : BND_ENTER_NEXT;
    } else {
      l = ap - a.k * a.n_rec + a.n_rec;
      if (ap == a.n_in + a.k * a.n_rec && a.n_rec > 0) bnd = BND_EXIT;
    }
  };

  // ---- embedding (row phase)
  if ((int)blockIdx.x < B) {
    const int b = blockIdx.x;
    int tok = a.tokens[b];
    if (tok < 0 || tok >= a.vocab) {
      if (threadIdx.x == 0) atomicCAS(a.status, 0, DEV_BAD_TOKEN);
      tok = 0;
    }
    float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if ((int)threadIdx.x < d / 8) load8_bf16(a.embed_in + (long long)tok * d + threadIdx.x * 8, v);
    mk_row_normalize(v, d, rsum);
    mk_row_store(a.h0 + (long long)b * d, a.hb + (long long)b * d, d, v);
  }
  int hsel = 0;
  const float* pend = nullptr;              // owed nGPT step (rate vector) on y32
  {
    int l, sl, st, bnd;
    app(0, l, sl, st, bnd);
    if (n_apps > 0 && bnd < 0) {
      const MkGemv g = mk_gemv_cfg(a.layers[l].w_qkvg, nqkvg, d, false);
      mk_gemv_prefetch<false>(g, w, w2, 3);
    }
  }
  if (!mk_sync(a, gen)) return;

  for (int ap = 0; ap < n_apps; ++ap) {
    int l, slice, store, bnd;
    app(ap, l, slice, store, bnd);
    const MkLayer& L = a.layers[l];
    float* hcur = hsel ? a.h1 : a.h0;
    if (bnd >= 0) {
      // loop boundary on rows (owed step first)
      if ((int)blockIdx.x < B) {
        const int b = blockIdx.x;
        float v[8];
        mk_row_step(hcur + (long long)b * d, pend ? a.y32 + (long long)b * d : nullptr, pend, d, v,
                    rsum);
        float* xr = a.x32 + (long long)b * d;
        const bool own = (int)threadIdx.x < d / 8;
        if (bnd == BND_SAVE_ENTER) {
          if (own) store8(xr + threadIdx.x * 8, v);
        } else {
          mk_row_normalize(v, d, rsum);      // s = N(h)
        }
        if (bnd != BND_EXIT) {
          float xv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          if (own) ld8f(xr + threadIdx.x * 8, xv);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] += xv[i];
          mk_row_normalize(v, d, rsum);
        }
        mk_row_store(hcur + (long long)b * d, a.hb + (long long)b * d, d, v);
      }
      pend = nullptr;
      {
        const MkGemv g = mk_gemv_cfg(L.w_qkvg, nqkvg, d, false);
        mk_gemv_prefetch<false>(g, w, w2, 3);
      }
      if (!mk_sync(a, gen)) return;
    }

    // ---- QKV + gate projection
    {
      const MkGemv g = mk_gemv_cfg(L.w_qkvg, nqkvg, d, false);
      const __nv_bfloat16* X = a.hb;
      if (pend) {
        mk_pre_rows(hcur, a.y32, pend, d, B, xs, hsel ? a.h0 : a.h1);
        __syncthreads();
        X = xs;
        hsel ^= 1;
        hcur = hsel ? a.h1 : a.h0;
        pend = nullptr;
      }
      mk_gemv_run<MM, false>(g, w, w2, X, d, B, a.gy, nqkvg, nullptr, nullptr, 0, red);
    }
    if (!mk_sync(a, gen)) return;

    // ---- attention (+ KV write), then prefetch the output projection
    mk_attention<DH>(a, L, slice, store, mk_smem);
    {
      const MkGemv g = mk_gemv_cfg(L.w_o, d, hq, false);
      mk_gemv_prefetch<false>(g, w, w2, 3);
    }
    if (!mk_sync(a, gen)) return;

    // ---- output projection (its nGPT step is owed)
    {
      const MkGemv g = mk_gemv_cfg(L.w_o, d, hq, false);
      mk_gemv_run<MM, false>(g, w, w2, a.att, hq, B, a.y32, d, nullptr, nullptr, 0, red);
      const MkGemv gu = mk_gemv_cfg(L.w_upgate, a.ffn, d, true);
      mk_gemv_prefetch<true>(gu, w, w2, 3);
    }
    pend = L.alpha_attn;
    if (!mk_sync(a, gen)) return;

    // ---- up + gate projection with SwiGLU (attention step fused)
    {
      const MkGemv g = mk_gemv_cfg(L.w_upgate, a.ffn, d, true);
      mk_pre_rows(hcur, a.y32, pend, d, B, xs, hsel ? a.h0 : a.h1);
      __syncthreads();
      hsel ^= 1;
      hcur = hsel ? a.h1 : a.h0;
      pend = nullptr;
      mk_gemv_run<MM, true>(g, w, w2, xs, d, B, nullptr, 0, nullptr, a.mo, a.ffn, red);
      const MkGemv gd = mk_gemv_cfg(L.w_down, d, a.ffn, false);
      mk_gemv_prefetch<false>(gd, w, w2, 3);
    }
    if (!mk_sync(a, gen)) return;

    // ---- down projection (its nGPT step is owed)
    {
      const MkGemv g = mk_gemv_cfg(L.w_down, d, a.ffn, false);
      mk_gemv_run<MM, false>(g, w, w2, a.mo, a.ffn, B, a.y32, d, nullptr, nullptr, 0, red);
      if (ap + 1 < n_apps) {
        int l2, s2, st2, b2;
        app(ap + 1, l2, s2, st2, b2);
        const MkGemv gq = mk_gemv_cfg(a.layers[l2].w_qkvg, nqkvg, d, false);
        mk_gemv_prefetch<false>(gq, w, w2, 3);
      }
    }
    pend = L.alpha_mlp;
    if (!mk_sync(a, gen)) return;
  }

  // ---- the last owed step (and the exit boundary when no output layer ran)
  const bool exit_pending = a.n_rec > 0 && a.n_out == 0;
  if ((int)blockIdx.x < B) {
    const int b = blockIdx.x;
    float* hcur = hsel ? a.h1 : a.h0;
    float v[8];
    mk_row_step(hcur + (long long)b * d, pend ? a.y32 + (long long)b * d : nullptr, pend, d, v,
                rsum);
    if (exit_pending) mk_row_normalize(v, d, rsum);
    mk_row_store(a.h0 + (long long)b * d, a.hb + (long long)b * d, d, v);
  }
  if (a.logits == nullptr) return;
  const MkGemv g = mk_gemv_cfg(a.embed_out, a.vocab, d, false);
  mk_gemv_prefetch<false>(g, w, w2, 4);
  if (!mk_sync(a, gen)) return;
  mk_gemv_run<MM, false>(g, w, w2, a.hb, d, B, a.logits, a.vocab, a.s_z, nullptr, 0, red);
  if (a.next == nullptr) return;
  if (!mk_sync(a, gen)) return;

  // ---- greedy token (row phase): lowest index among equal maxima
  if ((int)blockIdx.x < B) {
    __shared__ float bv[kMkWarps];
    __shared__ int bi[kMkWarps];
    const int b = blockIdx.x;
    const float* z = a.logits + (long long)b * a.vocab;
    float best = -INFINITY;
    int idx = 0x7fffffff;
    for (int i = threadIdx.x; i < a.vocab; i += kMkThreads) {
      const float v = z[i];
      if (v > best) {
        best = v;
        idx = i;
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
    if ((threadIdx.x & 31) == 0) {
      bv[threadIdx.x >> 5] = best;
      bi[threadIdx.x >> 5] = idx;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float bb = bv[0];
      int ii = bi[0];
      for (int w2 = 1; w2 < kMkWarps; ++w2)
        if (bv[w2] > bb || (bv[w2] == bb && bi[w2] < ii)) {
          bb = bv[w2];
          ii = bi[w2];
        }
      a.next[b] = ii == 0x7fffffff ? 0 : ii;
    }
  }
}

}  // namespace dory
