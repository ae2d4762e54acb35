// attn.cuh - masked grouped-query attention over cached and current keys.
//
// "Dory1.0-4B: A Looped Normalized-GPT", Architecture: grouped-query
// attention (G = n_q / n_kv query heads share one kv head), 3:1 interleave
// of sliding-window and full causal layers, input-dependent sigmoid gate on
// the attention output.  Last-Loop KV Caching: keys of earlier positions come
// from the cache slice (final-loop entries, or loop-i entries in per-loop
// mode), keys of the positions processed by this call come from this loop's
// own projections.
//
//   o_h(t) = sum_j softmax_j(scale * q_h(t) . k_{h/G}(j)) v_{h/G}(j),
//   j visible from t iff j <= t and (full layer or t - j < W);
//   out_h(t) = o_h(t) * sigmoid(g_h(t))            (bf16)
//
// q and k arrive already RoPE-rotated, L2-normalised and s_qk-scaled.  The
// normalisation of the concatenated gated output before the output
// projection is not applied here: the projection is linear and the nGPT step
// normalises its result, so a positive per-row scale of the projection input
// cancels exactly.
//
// One CTA = (sequence b, kv head, block of 64/G query positions); its 64
// rows are (position, head-in-group) pairs so every K/V tile staged in shared
// memory serves all G heads.  With few such CTAs (a short chunk over a long
// cache: the speculative verifier's gamma + 1 tokens) the key blocks are
// split over n_split CTAs whose partial results a second kernel merges.  4 warps x 16 rows, mma.sync m16n8k16 bf16 with
// fp32 accumulation, online softmax in fp32 (exp2), K/V tiles of 64 keys
// double-buffered with cp.async, XOR-swizzled 16-byte chunks for ldmatrix.
#pragma once
#include "ptx.cuh"

namespace dory {

struct AttnArgs {
  const __nv_bfloat16* q;        // [B*C, n_q, dh]
  const __nv_bfloat16* k_cur;    // [B*C, n_kv, dh]
  const __nv_bfloat16* v_cur;
  const __nv_bfloat16* k_cache;  // [max_batch, n_kv, S, dh] (this layer/slice)
  const __nv_bfloat16* v_cache;
  const __nv_bfloat16* gate;     // [B*C, n_q*dh], sigmoid(g)
  __nv_bfloat16* out;            // [B*C, n_q*dh]
  int C, P0, S;                  // tokens per sequence in the call, first position, ring slots
  int n_q, n_kv;
  int window;                    // 0 = full causal
  float scale_log2;              // softmax scale * log2(e)
  // key-range splits (n_split > 1): each CTA covers one split of its key
  // blocks and writes un-normalised partials; attn_split_combine_kernel
  // merges them, normalises and applies the gate
  int n_split;
  float* part_o;                 // [B*C, n_q, n_split, dh]
  float* part_ml;                // [B*C, n_q, n_split, 2]: running max (log2 units), sum
  int part_cap;                  // launcher input: most splits the partial buffers hold
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float* c, const uint32_t* a, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int DH>
struct AttnCfg {
  static constexpr int BR = 64, BKEY = 64;
  static constexpr int CH = DH / 8;                 // 16-byte chunks per row
  static constexpr int SWZ = CH < 8 ? CH - 1 : 7;   // XOR mask on the chunk index
  static constexpr size_t SMEM = (size_t)(BR * DH + 4 * BKEY * DH) * 2;
};

template <int DH>
__device__ __forceinline__ uint32_t swz_off(int row, int chunk) {
  using Cf = AttnCfg<DH>;
  return (uint32_t)(row * DH + ((chunk ^ (row & Cf::SWZ)) << 3)) * 2u;   // bytes
}

template <int DH>
__global__ void __launch_bounds__(128) attn_prefill_kernel(const AttnArgs a) {
  using Cf = AttnCfg<DH>;
  constexpr int BR = Cf::BR, BKEY = Cf::BKEY, CH = Cf::CH;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  __nv_bfloat16* sK = sQ + BR * DH;             // [2][BKEY*DH]
  __nv_bfloat16* sV = sK + 2 * BKEY * DH;       // [2][BKEY*DH]
  const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV);
  pdl_wait();
  pdl_trigger();

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.n_q / a.n_kv, BQ = BR / G;
  const int qb = gridDim.x - 1 - blockIdx.x;    // longest rows first
  const int n_split = a.n_split > 1 ? a.n_split : 1;
  const int kvh = blockIdx.y, b = blockIdx.z / n_split, split = blockIdx.z % n_split;
  const int q0 = qb * BQ;
  const int nqv = min(BQ, a.C - q0);
  const int p_lo = a.P0 + q0, p_hi = a.P0 + q0 + nqv - 1;
  const int k_lo = a.window > 0 ? max(0, p_lo - a.window + 1) : 0;
  const int k_hi = p_hi;
  const int nblk_all = (k_hi - k_lo) / BKEY + 1;
  const int blk0 = (int)((long long)split * nblk_all / n_split);
  const int blk1 = (int)((long long)(split + 1) * nblk_all / n_split);

  // ---- Q tile: row r = (position i = r / G, head hg = r % G)
  for (int idx = tid; idx < BR * CH; idx += 128) {
    const int r = idx / CH, c = idx % CH;
    const int i = r / G, hg = r % G;
    const bool ok = i < nqv;
    const __nv_bfloat16* src =
        ok ? a.q + (((long long)b * a.C + q0 + i) * a.n_q + kvh * G + hg) * DH + c * 8 : a.q;
    cp_async16(sQa + swz_off<DH>(r, c), src, ok);
  }
  auto load_kv = [&](int blk, int buf) {
    const int kb0 = k_lo + blk * BKEY;
    for (int idx = tid; idx < BKEY * CH; idx += 128) {
      const int r = idx / CH, c = idx % CH;
      const int j = kb0 + r;
      const bool ok = j <= k_hi;
      const __nv_bfloat16 *ks = a.k_cur, *vs = a.v_cur;
      if (ok) {
        long long off;
        if (j < a.P0) {
          off = (((long long)b * a.n_kv + kvh) * a.S + (j % a.S)) * DH + c * 8;
          ks = a.k_cache + off;
          vs = a.v_cache + off;
        } else {
          off = (((long long)b * a.C + (j - a.P0)) * a.n_kv + kvh) * DH + c * 8;
          ks = a.k_cur + off;
          vs = a.v_cur + off;
        }
      }
      const uint32_t o = swz_off<DH>(r, c) + (uint32_t)(buf * BKEY * DH * 2);
      cp_async16(sKa + o, ks, ok);
      cp_async16(sVa + o, vs, ok);
    }
  };
  if (blk0 < blk1) load_kv(blk0, 0);
  cp_async_commit();

  const int g = lane >> 2, t4 = lane & 3;
  uint32_t qf[DH / 16][4];
  float o[DH / 8][4];
#pragma unroll
  for (int i = 0; i < DH / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  // query position of this thread's two rows (row = 16 warp + g + 8 half)
  int qpos[2];
  bool qok[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = warp * 16 + g + 8 * h;
    const int i = r / G;
    qok[h] = i < nqv;
    qpos[h] = a.P0 + q0 + i;
  }

  for (int blk = blk0; blk < blk1; ++blk) {
    const int buf = (blk - blk0) & 1;
    if (blk + 1 < blk1) {
      load_kv(blk + 1, buf ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (blk == blk0) {
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        const int r = warp * 16 + (lane & 15);
        const int c = 2 * kk + (lane >> 4);
        ldsm_x4(sQa + swz_off<DH>(r, c), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }
    const uint32_t kbase = sKa + (uint32_t)(buf * BKEY * DH * 2);
    const uint32_t vbase = sVa + (uint32_t)(buf * BKEY * DH * 2);

    // ---- S = Q K^T  (16 x 64 per warp)
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int np = 0; np < 4; ++np) {
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        const int key = 16 * np + (lane & 7) + ((lane >> 4) & 1) * 8;
        const int c = 2 * kk + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + swz_off<DH>(key, c), b0, b1, b2, b3);
        mma_bf16_16816(s[2 * np], qf[kk], b0, b1);
        mma_bf16_16816(s[2 * np + 1], qf[kk], b2, b3);
      }
    }
    // ---- mask, online softmax
    const int kb0 = k_lo + blk * BKEY;
    float corr[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = kb0 + 8 * nt + 2 * t4 + e;
          const int rel = qpos[h] - j;
          const bool vis = qok[h] && j <= k_hi && rel >= 0 && (a.window <= 0 || rel < a.window);
          float v = s[nt][2 * h + e] * a.scale_log2;
          v = vis ? v : -INFINITY;
          s[nt][2 * h + e] = v;
          mx = fmaxf(mx, v);
        }
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run[h], mx);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      corr[h] = exp2f(m_run[h] - m_use);
      m_run[h] = m_new;
      float ls = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float p = exp2f(s[nt][2 * h + e] - m_use);
          s[nt][2 * h + e] = p;
          ls += p;
        }
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
    // ---- O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < DH / 16; ++dp) {
        const int key = 16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = 2 * dp + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vbase + swz_off<DH>(key, c), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * dp], pa, b0, b1);
        mma_bf16_16816(o[2 * dp + 1], pa, b2, b3);
      }
    }
    __syncthreads();
  }

  cp_async_wait<0>();
  if (n_split > 1) {
    // ---- un-normalised partials of this split (an empty split: m = -inf, l = 0)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float l = l_run[h];
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      if (!qok[h]) continue;
      const int r = warp * 16 + g + 8 * h;
      const int i = r / G, hg = r % G;
      const long long slot =
          (((long long)b * a.C + q0 + i) * a.n_q + kvh * G + hg) * n_split + split;
      float* po = a.part_o + slot * DH;
#pragma unroll
      for (int nt = 0; nt < DH / 8; ++nt)
        *reinterpret_cast<float2*>(po + 8 * nt + 2 * t4) = make_float2(o[nt][2 * h], o[nt][2 * h + 1]);
      if (t4 == 0) *reinterpret_cast<float2*>(a.part_ml + slot * 2) = make_float2(m_run[h], l);
    }
    return;
  }
  // ---- normalise, gate, store
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float l = l_run[h];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    if (!qok[h]) continue;
    const float inv = l > 0.f ? 1.0f / l : 0.f;
    const int r = warp * 16 + g + 8 * h;
    const int i = r / G, hg = r % G;
    const long long row = (long long)b * a.C + q0 + i;
    const long long base = row * a.n_q * DH + (long long)(kvh * G + hg) * DH;
#pragma unroll
    for (int nt = 0; nt < DH / 8; ++nt) {
      const int dim = 8 * nt + 2 * t4;
      const __nv_bfloat162 gt = *reinterpret_cast<const __nv_bfloat162*>(a.gate + base + dim);
      const float2 gf = __bfloat1622float2(gt);
      const uint32_t pk = pack_bf16x2(o[nt][2 * h] * inv * gf.x, o[nt][2 * h + 1] * inv * gf.y);
      *reinterpret_cast<uint32_t*>(a.out + base + dim) = pk;
    }
  }
}

// Merge of the key-range splits: one CTA of DH threads per (row, head);
// out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s, times the gate.
template <int DH>
__global__ void __launch_bounds__(DH) attn_split_combine_kernel(const AttnArgs a, int rows) {
  pdl_wait();
  pdl_trigger();
  const long long rh = blockIdx.x;                     // row * n_q + head
  const int n_split = a.n_split;
  const float* ml = a.part_ml + rh * n_split * 2;
  float M = -INFINITY;
  for (int s = 0; s < n_split; ++s) M = fmaxf(M, ml[2 * s]);
  float acc = 0.f, l = 0.f;
  for (int s = 0; s < n_split; ++s) {
    const float w = ml[2 * s] == -INFINITY ? 0.f : exp2f(ml[2 * s] - M);
    acc += w * a.part_o[(rh * n_split + s) * DH + threadIdx.x];
    l += w * ml[2 * s + 1];
  }
  const long long idx = rh * DH + threadIdx.x;
  const float gt = __bfloat162float(a.gate[idx]);
  const float inv = l > 0.f ? 1.0f / l : 0.f;         // as the one-pass epilogue
  a.out[idx] = __float2bfloat16_rn(acc * inv * gt);
}

}  // namespace dory

namespace dory {

// ---------------------------------------------------------------------------
// Decode attention (one new token per sequence), split over the keys.
//
// The new token at position P0 sees its own current-loop key/value and the
// cached keys of earlier positions (final-loop or loop-i entries; "Dory1.0-4B:
// A Looped Normalized-GPT", Last-Loop KV Caching).  The visible keys are cut
// into splits of `chunk` keys; one CTA = (split, kv head, sequence) serves
// all G query heads of that kv head from one shared-memory copy of each K/V
// tile and writes an un-normalised partial (o, running max m, sum l) per
// head.  The combine kernel merges the splits, normalises, applies the gate.
// Memory-bound: each K/V byte is read once per loop, with 16-byte loads.
// ---------------------------------------------------------------------------
constexpr int kDecMaxSplits = 128;
constexpr int kDecTile = 64;
constexpr int kDecMaxG = 8;

struct DecodeArgs {
  const __nv_bfloat16* q;        // [B, n_q, dh]
  const __nv_bfloat16* k_cur;    // [B, n_kv, dh]
  const __nv_bfloat16* v_cur;
  const __nv_bfloat16* k_cache;  // [max_batch, n_kv, S, dh]
  const __nv_bfloat16* v_cache;
  int P0, S, n_q, n_kv, window;
  float scale_log2;
  int chunk, n_splits;
  float* part_o;                 // [B, n_q, kDecMaxSplits, dh]
  float* part_ml;                // [B, n_q, kDecMaxSplits, 2]
};

template <int DH>
__global__ void __launch_bounds__(128) attn_decode_split_kernel(const DecodeArgs a) {
  constexpr int KP = DH + 8;                            // padded bf16 row (conflict-free)
  __shared__ __align__(16) __nv_bfloat16 ks[kDecTile * KP];
  __shared__ __align__(16) __nv_bfloat16 vs[kDecTile * DH];
  __shared__ float qs[kDecMaxG * DH];
  __shared__ float ps[kDecMaxG * kDecTile];
  __shared__ float m_s[kDecMaxG], l_s[kDecMaxG], c_s[kDecMaxG];
  pdl_wait();
  pdl_trigger();
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.n_q / a.n_kv;
  const int p = a.P0;
  const int lo = a.window > 0 ? max(0, p - a.window + 1) : 0;
  const int k0 = lo + split * a.chunk;
  const int k1 = min(k0 + a.chunk, p + 1);
  for (int i = tid; i < G * DH; i += 128) {
    const int g = i / DH, d = i % DH;
    qs[i] = __bfloat162float(a.q[((long long)b * a.n_q + kvh * G + g) * DH + d]);
  }
  if (tid < G) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
  }
  constexpr int ITEMS = kDecMaxG * DH / 128;
  float o[ITEMS];
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) o[i] = 0.f;
  constexpr int CPR = DH / 8;                           // 16-byte chunks per row
  for (int t0 = k0; t0 < k1; t0 += kDecTile) {
    const int n = min(kDecTile, k1 - t0);
    __syncthreads();
    for (int i = tid; i < kDecTile * CPR; i += 128) {
      const int r = i / CPR, c = i % CPR;
      uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
      if (r < n) {
        const int j = t0 + r;
        long long off;
        const __nv_bfloat16 *kb, *vb;
        if (j < a.P0) {
          off = (((long long)b * a.n_kv + kvh) * a.S + (j % a.S)) * DH + c * 8;
          kb = a.k_cache;
          vb = a.v_cache;
        } else {
          off = ((long long)b * a.n_kv + kvh) * DH + c * 8;
          kb = a.k_cur;
          vb = a.v_cur;
        }
        kv = *reinterpret_cast<const uint4*>(kb + off);
        vv = *reinterpret_cast<const uint4*>(vb + off);
      }
      *reinterpret_cast<uint4*>(ks + r * KP + c * 8) = kv;
      *reinterpret_cast<uint4*>(vs + r * DH + c * 8) = vv;
    }
    __syncthreads();
    // scores for (head g, key r)
    for (int i = tid; i < G * kDecTile; i += 128) {
      const int g = i / kDecTile, r = i % kDecTile;
      float s = -INFINITY;
      if (r < n) {
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < CPR; ++c) {
          float kf[8];
          const uint4 u = *reinterpret_cast<const uint4*>(ks + r * KP + c * 8);
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h2[e]);
            kf[2 * e] = f.x;
            kf[2 * e + 1] = f.y;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) acc = fmaf(qs[g * DH + c * 8 + e], kf[e], acc);
        }
        s = acc * a.scale_log2;
      }
      ps[g * kDecTile + r] = s;
    }
    __syncthreads();
    // online softmax per head (warp w handles heads w, w + 4, ...)
    for (int g = warp; g < G; g += 4) {
      const float s0 = ps[g * kDecTile + lane], s1 = ps[g * kDecTile + lane + 32];
      float mx = fmaxf(s0, s1);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_old = m_s[g];
      const float m_new = fmaxf(m_old, mx);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float p0 = exp2f(s0 - m_use), p1 = exp2f(s1 - m_use);
      ps[g * kDecTile + lane] = p0;
      ps[g * kDecTile + lane + 32] = p1;
      const float sum = warp_sum(p0 + p1);
      if (lane == 0) {
        const float corr = exp2f(m_old - m_use);
        c_s[g] = corr;
        l_s[g] = l_s[g] * corr + sum;
        m_s[g] = m_new;
      }
    }
    __syncthreads();
    // o[g][d] = corr * o + sum_r p[g][r] v[r][d]
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const int i = tid + it * 128;
      const int g = i / DH, d = i % DH;
      if (g < G) {
        float acc = o[it] * c_s[g];
        for (int r = 0; r < n; ++r)
          acc = fmaf(ps[g * kDecTile + r], __bfloat162float(vs[r * DH + d]), acc);
        o[it] = acc;
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int it = 0; it < ITEMS; ++it) {
    const int i = tid + it * 128;
    const int g = i / DH, d = i % DH;
    if (g < G) {
      const long long base = (((long long)b * a.n_q + kvh * G + g) * kDecMaxSplits + split);
      a.part_o[base * DH + d] = o[it];
      if (d == 0) {
        a.part_ml[base * 2] = m_s[g];
        a.part_ml[base * 2 + 1] = l_s[g];
      }
    }
  }
}

// Merges the splits of every (sequence, head): out = gate * sum_s o_s 2^(m_s - M)
// / sum_s l_s 2^(m_s - M).  grid = B * n_q, block = dh.
__global__ void attn_decode_combine_kernel(const float* part_o, const float* part_ml, int n_splits,
                                           int n_q, int dh, const __nv_bfloat16* gate,
                                           __nv_bfloat16* out) {
  pdl_wait();
  pdl_trigger();
  const long long bh = blockIdx.x;
  const int d = threadIdx.x;
  const float* ml = part_ml + bh * kDecMaxSplits * 2;
  float M = -INFINITY;
  for (int s = 0; s < n_splits; ++s) M = fmaxf(M, ml[2 * s]);
  float L = 0.f, acc = 0.f;
  for (int s = 0; s < n_splits; ++s) {
    const float w = ml[2 * s] == -INFINITY ? 0.f : exp2f(ml[2 * s] - M);
    L += ml[2 * s + 1] * w;
    acc += part_o[(bh * kDecMaxSplits + s) * dh + d] * w;
  }
  const long long b = bh / n_q, h = bh % n_q;
  const long long idx = (b * n_q + h) * dh + d;
  const float gt = __bfloat162float(gate[idx]);
  out[idx] = __float2bfloat16_rn(L > 0.f ? acc * (1.0f / L) * gt : 0.f);
}

}  // namespace dory

namespace dory {

// ---------------------------------------------------------------------------
// Decode attention of the forward pass: one new token per sequence at
// position P0, split over the cached keys, with the split merge, the output
// gate and the KV-cache write fused in ("Dory1.0-4B: A Looped
// Normalized-GPT", Architecture; Last-Loop KV Caching).
//
// Grid (split, kv head, sequence), 128 threads.  The CTA's 16 mma rows are the
// G query heads of its kv head (rows >= G are zero).  Cached keys of the
// split stream through a 2-stage cp.async ring of 64-key K/V tiles (XOR
// swizzled 16-byte chunks, ldmatrix-friendly); warp w takes keys 16w..16w+15
// of every tile with mma.sync m16n8k16 (bf16 in, fp32 accumulate) and keeps
// its own online-softmax state; the 4 warps merge through shared memory and
// the CTA writes an unnormalised partial (o, max, sum) per head.
//
// The new token sees its own current-loop key and value, never the cache:
// every CTA forms q^, k^ and v of the token in its prologue, split 0 of each
// (sequence, kv head) writes k^ / v into ring slot P0 mod S when `store` is
// set (no CTA of the launch reads that slot: it holds no visible position),
// and the last CTA of the group to finish (atomic ticket, no waiting) merges
// all partials with the new token's own term, applies sigmoid(g) and writes
// the gated output.  The ticket counter returns to zero for the next launch.
//
// RAW inputs are the fp32 rows of the QKV + gate projection (columns
// [q heads | k heads | v heads | gate], n_parts partial sums part_stride
// apart); the prologue applies RoPE, the per-head L2 norm and s_qk to q and k
// and rounds k^ / v to bf16 (the cache precision).  Otherwise the inputs are
// ready bf16 q^, k^, v and sigmoid(g).
// ---------------------------------------------------------------------------
constexpr int kDecStages = 2;
constexpr int kDecMinTiles = 2;

struct DecAttnArgs {
  const float* y;                 // RAW: [B, ldy] fp32 projection rows
  int ldy, n_parts;
  long long part_stride;
  const float* s_qk;              // RAW: [dh]
  const float2* rope;             // RAW: [dh / 2] (cos, sin) of position P0 ([B][dh / 2] of
                                  // each sequence's position when p0s is set), or null
  const __nv_bfloat16* q;         // READY: [B, n_q, dh]
  const __nv_bfloat16* k_cur;     // READY: [B, n_kv, dh]
  const __nv_bfloat16* v_cur;
  const __nv_bfloat16* gate;      // READY: [B, n_q * dh], sigmoid applied
  __nv_bfloat16* k_cache;         // [., n_kv, S, dh] of this layer / slice
  __nv_bfloat16* v_cache;
  int store;
  int P0, S, n_q, n_kv, window;   // P0: the position of every sequence's new token, or
                                  // (ragged batches) the largest one
  const int* p0s;                 // ragged batches: [B] each sequence's position (device), or null
  const int* kstore;              // per-sequence loop counts: [B]; sequence b also stores
  int loop;                       //   its key and value when kstore[b] == loop
  float scale_log2;
  int chunk, n_splits;
  int tpg;                        // TMA kernel: 64-key tiles per (sequence, kv head) group
  float* part_o;                  // [B, n_q, n_splits, dh]
  float* part_ml;                 // [B, n_q, n_splits, 2]
  int* counter;                   // [B * n_kv], zero between launches
  __nv_bfloat16* out;             // [B, n_q * dh]
  int B;                          // sequences
  long long cache_rows;           // rows of the cache block ([batch][n_kv][S]); 0 = unknown
  int* status;                    // device status word (bounded waits), or null
};

template <int DH>
struct DecCfg {
  static constexpr int QB = 16 * DH * 2;                    // Q tile bytes
  static constexpr int KVB = kDecTile * DH * 2;             // one K or V tile
  static constexpr int STAGE = 2 * KVB;
  static constexpr int MERGE = 4 * 16 * DH * 4;             // per-warp o for the merge
  static constexpr int RING = kDecStages * STAGE > MERGE ? kDecStages * STAGE : MERGE;
  static constexpr size_t SMEM = QB + RING + 2 * DH * 4 + 4 * 16 * 2 * 4 + 64 + kDecMaxG * DH * 4;
};

template <int DH, bool RAW>
__global__ void __launch_bounds__(128) attn_decode_kernel(const DecAttnArgs a) {
  using Cf = DecCfg<DH>;
  constexpr int CH = DH / 8, HALF = DH / 2;
  extern __shared__ __align__(128) uint8_t dsm[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(dsm);
  uint8_t* ring = dsm + Cf::QB;
  float* sKc = reinterpret_cast<float*>(ring + Cf::RING);     // current k^ (bf16-rounded)
  float* sVc = sKc + DH;                                      // current v (bf16-rounded)
  float* sM = sVc + DH;                                       // [4][16]
  float* sL = sM + 64;                                        // [4][16]
  int* sFlag = reinterpret_cast<int*>(sL + 64);
  float* sCur = reinterpret_cast<float*>(sFlag + 1);          // [8] new-token score per head
  float* sGate = sCur + 8;                                    // [G][DH] sigmoid(g)
  const uint32_t sQa = smem_u32(sQ), ringa = smem_u32(ring);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.n_q / a.n_kv;
  const int NS = a.n_splits;
  const int n_items = NS * a.n_kv * a.B;

  // ragged batches: the positions were written by an earlier kernel of the
  // step, so wait for the previous kernel before the first tile loads
  if (a.p0s) pdl_wait();
  // Work items (split, kv head, sequence) of equal size; the CTAs of the grid
  // (no more than are resident) stride over them.
  bool first = true;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int split = item % NS, kvh = (item / NS) % a.n_kv, b = item / (NS * a.n_kv);
    // this sequence's position (ragged batches: its own; trailing splits of
    // shorter sequences are empty)
    const int P0 = a.p0s ? a.p0s[b] : a.P0;
    const int lo = a.window > 0 ? max(0, P0 - a.window + 1) : 0;
    const int k0 = lo + split * a.chunk;
    const int k1 = min(k0 + a.chunk, P0);                    // cached keys only
    const int ntiles = k1 > k0 ? (k1 - k0 + kDecTile - 1) / kDecTile : 0;

    // cached K / V tile t into ring buffer `buf` (zero-filled beyond k1).
    // The cache was written by earlier launches, so the first item's loads
    // may start before the wait on the previous kernel.
    auto load_tile = [&](int t, int buf) {
      const int j0 = k0 + t * kDecTile;
      const uint32_t kb = ringa + (uint32_t)(buf * Cf::STAGE), vb = kb + Cf::KVB;
      for (int idx = tid; idx < kDecTile * CH; idx += 128) {
        const int r = idx / CH, c = idx % CH;
        const int j = j0 + r;
        const bool ok = j < k1;
        const long long off =
            ok ? (((long long)b * a.n_kv + kvh) * a.S + (j % a.S)) * DH + c * 8 : 0;
        cp_async16(kb + swz_off<DH>(r, c), a.k_cache + off, ok);
        cp_async16(vb + swz_off<DH>(r, c), a.v_cache + off, ok);
      }
    };
    if (!first) __syncthreads();                           // smem of the previous item free
#pragma unroll
    for (int st = 0; st < kDecStages; ++st) {              // fill the whole ring
      if (st < ntiles) load_tile(st, st);
      cp_async_commit();
    }
    if (first) {
      pdl_wait();
      pdl_trigger();
      first = false;
    }

    // ---- prologue: q^ (rows of sQ), current k^ and v
    for (int idx = tid; idx < 16 * CH; idx += 128) {       // zero rows >= G
      const int r = idx / CH, c = idx % CH;
      if (r >= G) *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(sQ) + swz_off<DH>(r, c)) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    // gate of the G heads (needed only by the item that merges, but its
    // load overlaps the rest of the prologue here instead of lengthening the
    // merge at the end)
    for (int idx = tid; idx < G * DH; idx += 128) {
      const int r = idx / DH, dd = idx % DH;
      float gt;
      if (RAW) {
        float gr = 0.f;
        const float* yg = a.y + (long long)b * a.ldy + (long long)(a.n_q + 2 * a.n_kv) * DH +
                          (kvh * G + r) * DH + dd;
        for (int p = 0; p < a.n_parts; ++p) gr += yg[p * a.part_stride];
        gt = 1.0f / (1.0f + __expf(-gr));
      } else {
        gt = __bfloat162float(a.gate[((long long)b * a.n_q + kvh * G + r) * DH + dd]);
      }
      sGate[idx] = gt;
    }
    for (int hh = warp; hh < G + 2; hh += 4) {
      // hh < G: query head kvh * G + hh; hh == G: key; hh == G + 1: value
      if (RAW) {
        const int col0 = hh < G ? (kvh * G + hh) * DH
                                : (hh == G ? (a.n_q + kvh) * DH : (a.n_q + a.n_kv + kvh) * DH);
        const float* yr = a.y + (long long)b * a.ldy + col0;
        float x1[(HALF + 31) / 32], x2[(HALF + 31) / 32];
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < (HALF + 31) / 32; ++e) {
          const int i = lane + 32 * e;
          x1[e] = x2[e] = 0.f;
          if (i < HALF) {
            for (int p = 0; p < a.n_parts; ++p) {
              x1[e] += yr[p * a.part_stride + i];
              x2[e] += yr[p * a.part_stride + i + HALF];
            }
          }
          ss += x1[e] * x1[e] + x2[e] * x2[e];
        }
        if (hh <= G) {
          const float inv = 1.0f / sqrtf(fmaxf(warp_sum(ss), 1e-12f));
#pragma unroll
          for (int e = 0; e < (HALF + 31) / 32; ++e) {
            const int i = lane + 32 * e;
            if (i < HALF) {
              float c1 = x1[e], c2 = x2[e];
              if (a.rope) {
                const float2 cs = a.rope[(a.p0s ? b * HALF : 0) + i];
                c1 = x1[e] * cs.x - x2[e] * cs.y;
                c2 = x2[e] * cs.x + x1[e] * cs.y;
              }
              x1[e] = c1 * inv * a.s_qk[i];
              x2[e] = c2 * inv * a.s_qk[i + HALF];
            }
          }
        }
#pragma unroll
        for (int e = 0; e < (HALF + 31) / 32; ++e) {
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
            if ((a.store || (a.kstore && a.kstore[b] == a.loop)) && split == 0) {
              __nv_bfloat16* cache = hh == G ? a.k_cache : a.v_cache;
              const long long off = (((long long)b * a.n_kv + kvh) * a.S + (P0 % a.S)) * DH;
              cache[off + i] = b1;
              cache[off + i + HALF] = b2;
            }
          }
        }
      } else {
        for (int i = lane; i < DH; i += 32) {
          if (hh < G) {
            sQ[(swz_off<DH>(hh, i / 8) >> 1) + (i & 7)] =
                a.q[((long long)b * a.n_q + kvh * G + hh) * DH + i];
          } else {
            const __nv_bfloat16* src = hh == G ? a.k_cur : a.v_cur;
            const __nv_bfloat16 v = src[((long long)b * a.n_kv + kvh) * DH + i];
            (hh == G ? sKc : sVc)[i] = __bfloat162float(v);
            if ((a.store || (a.kstore && a.kstore[b] == a.loop)) && split == 0) {
              __nv_bfloat16* cache = hh == G ? a.k_cache : a.v_cache;
              cache[(((long long)b * a.n_kv + kvh) * a.S + (P0 % a.S)) * DH + i] = v;
            }
          }
        }
      }
    }
    __syncthreads();

    // ---- cached keys: S = Q K^T, online softmax, O += P V (warp: 16 keys / tile)
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
    float m_run = -INFINITY, l_run = 0.f;

    for (int t = 0; t < ntiles; ++t) {
      // tile t landed (tile t + 1 may still be in flight)
      if (t + 1 < ntiles) cp_async_wait<1>(); else cp_async_wait<0>();
      __syncthreads();
      const uint32_t kbase = ringa + (uint32_t)((t % kDecStages) * Cf::STAGE);
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
      // Only mma rows g < 8 can hold a head (G <= 8): the second row half
      // (g + 8) gets P = 0 and no softmax work.  The running max is raised
      // only when it grows by more than 2^8 (exact: the same stale max scales
      // P and the row sum), so the accumulators are rarely rescaled.
      const int j0 = k0 + t * kDecTile + 16 * warp;
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = j0 + 8 * nt + 2 * t4 + e;
          float v = s[nt][e] * a.scale_log2;
          v = j < k1 ? v : -INFINITY;
          s[nt][e] = v;
          mx = fmaxf(mx, v);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      if (mx > m_run + 8.0f) {
        const float corr = m_run == -INFINITY ? 0.f : exp2f(m_run - mx);
        m_run = mx;
        l_run *= corr;
#pragma unroll
        for (int i = 0; i < DH / 8; ++i) {
          o[i][0] *= corr;
          o[i][1] *= corr;
        }
      }
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      float ls = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float p = exp2f(s[nt][e] - m_use);
          s[nt][e] = p;
          ls += p;
        }
      l_run += ls;
      uint32_t pa[4];
      pa[0] = pack_bf16x2(s[0][0], s[0][1]);
      pa[1] = 0u;
      pa[2] = pack_bf16x2(s[1][0], s[1][1]);
      pa[3] = 0u;
#pragma unroll
      for (int dp = 0; dp < DH / 16; ++dp) {
        const int key = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c = 2 * dp + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vbase + swz_off<DH>(key, c), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * dp], pa, b0, b1);
        mma_bf16_16816(o[2 * dp + 1], pa, b2, b3);
      }
      __syncthreads();                                     // buffer t % 2 free
      if (t + kDecStages < ntiles) load_tile(t + kDecStages, t % kDecStages);
      cp_async_commit();
    }
    cp_async_wait<0>();
    __syncthreads();                                       // ring free: reuse for the merge

    // ---- merge the 4 warps: row r = head, per warp (m, l, o[r][:])
    float* sO = reinterpret_cast<float*>(ring);             // [4][16][DH]
    {
      float l = l_run;
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      if (t4 == 0) {
        sM[warp * 16 + g] = m_run;
        sL[warp * 16 + g] = l;
      }
#pragma unroll
      for (int nt = 0; nt < DH / 8; ++nt) {
        const int dim = 8 * nt + 2 * t4;
        *reinterpret_cast<float2*>(sO + (warp * 16 + g) * DH + dim) =
            make_float2(o[nt][0], o[nt][1]);
      }
    }
    __syncthreads();
    for (int idx = tid; idx < G * DH; idx += 128) {
      const int r = idx / DH, dd = idx % DH;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; ++w) M = fmaxf(M, sM[w * 16 + r]);
      float L = 0.f, acc = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float wt = sM[w * 16 + r] == -INFINITY ? 0.f : exp2f(sM[w * 16 + r] - M);
        L += sL[w * 16 + r] * wt;
        acc += sO[(w * 16 + r) * DH + dd] * wt;
      }
      const long long base = ((long long)b * a.n_q + kvh * G + r) * a.n_splits + split;
      a.part_o[base * DH + dd] = acc;
      if (dd == 0) {
        a.part_ml[base * 2] = M;
        a.part_ml[base * 2 + 1] = L;
      }
    }

    // ---- ticket: the last CTA of (b, kvh) merges all splits + the new token
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const int prev = atomicAdd(&a.counter[b * a.n_kv + kvh], 1);
      *sFlag = prev == a.n_splits - 1;
    }
    __syncthreads();
    if (!*sFlag) continue;
    __threadfence();
    // new token's own score per head: q^ . k^_cur (bf16 operands, fp32 sum)
    for (int r = warp; r < G; r += 4) {
      float acc = 0.f;
      for (int i = lane; i < DH; i += 32)
        acc += __bfloat162float(sQ[(swz_off<DH>(r, i / 8) >> 1) + (i & 7)]) * sKc[i];
      acc = warp_sum(acc);
      if (lane == 0) sCur[r] = acc * a.scale_log2;
    }
    __syncthreads();
    // per head: global max and split weights, one lane per split (warp = head)
    float* sW = reinterpret_cast<float*>(ring);                // [G][NS + 1]
    for (int r = warp; r < G; r += 4) {
      const long long bh = (long long)b * a.n_q + kvh * G + r;
      float mx = sCur[r];
      for (int sp = lane; sp < NS; sp += 32) mx = fmaxf(mx, __ldcg(a.part_ml + (bh * NS + sp) * 2));
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
      float L = 0.f;
      for (int sp = lane; sp < NS; sp += 32) {
        const float ms = __ldcg(a.part_ml + (bh * NS + sp) * 2);
        const float wt = ms == -INFINITY ? 0.f : exp2f(ms - mx);
        sW[r * (NS + 1) + sp] = wt;
        L += __ldcg(a.part_ml + (bh * NS + sp) * 2 + 1) * wt;
      }
      L = warp_sum(L);
      if (lane == 0) {
        const float wc = exp2f(sCur[r] - mx);
        sW[r * (NS + 1) + NS] = wc;                              // new token's weight
        sM[r] = 1.0f / (L + wc);
      }
    }
    __syncthreads();
    for (int idx = tid; idx < G * DH; idx += 128) {
      const int r = idx / DH, dd = idx % DH;
      const long long bh = (long long)b * a.n_q + kvh * G + r;
      const float* wr = sW + r * (NS + 1);
      float acc = wr[NS] * sVc[dd];
      const float* po = a.part_o + bh * NS * DH + dd;
      int sp = 0;
      for (; sp + 4 <= NS; sp += 4) {
        const float o0 = __ldcg(po + (sp + 0) * DH), o1 = __ldcg(po + (sp + 1) * DH);
        const float o2 = __ldcg(po + (sp + 2) * DH), o3 = __ldcg(po + (sp + 3) * DH);
        acc += wr[sp] * o0 + wr[sp + 1] * o1 + wr[sp + 2] * o2 + wr[sp + 3] * o3;
      }
      for (; sp < NS; ++sp) acc += wr[sp] * __ldcg(po + sp * DH);
      a.out[bh * DH + dd] = __float2bfloat16_rn(acc * sM[r] * sGate[idx]);
    }
    if (tid == 0) a.counter[b * a.n_kv + kvh] = 0;
  }
  if (first) {                                                // no item: still order the grid
    pdl_wait();
    pdl_trigger();
  }
}

}  // namespace dory
