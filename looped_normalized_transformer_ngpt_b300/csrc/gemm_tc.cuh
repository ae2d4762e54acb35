// gemm_tc.cuh - tcgen05 / TMEM BF16 GEMM for the dense projections of the
// looped nGPT layer (QKV+gate, output, up+gate, down, LM head), with the
// per-projection epilogues fused.
//
//   C[m, n] = sum_k A[m, k] * B[n, k]      A: activations [M, K] bf16
//                                          B: weights     [N, K] bf16
//
// Persistent, warp-specialised, one CTA per SM (320 threads):
//   warp 0      TMA producer: A tile 128 x 64 and B tile BN x 64 per stage,
//               128-byte swizzle, STAGES-deep ring of shared-memory buffers;
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma 128 x BN x 16 into
//               one of two TMEM accumulators (2 x BN fp32 columns);
//   warps 2..9  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//               lanes 32 (w % 4) .. +31, i.e. tile rows; warps 2..5 take the
//               first half of the tile's columns, warps 6..9 the second),
//               fused math, stores.
// The epilogue of tile i overlaps the MMAs of tile i + 1.
//
// Epilogues (projection names from "Dory1.0-4B: A Looped Normalized-GPT",
// Architecture):
//   EPI_F32     fp32 store, optional per-column scale (LM head: s_z).
//   EPI_QKVG    columns are [q heads | k heads | v heads | gate]; q and k heads
//               get RoPE (rotate-half, table lookup), L2 normalisation over the
//               head and the s_qk scale; the gate gets a sigmoid; all stored
//               as bf16 in head-major rows.
//   EPI_SWIGLU  B tile = 64/128 rows of W_up and the same rows of W_sl; the
//               epilogue forms m = u * SiLU(v) and stores m as bf16.
// With BN = 256 these three stage their output in shared memory in the
// 128-byte swizzled layout and one thread of each 4-warp half writes it with
// TMA tensor stores (whole 128-byte rows; a thread-per-row store pattern
// touches 32 rows per instruction).
//   EPI_NGPT    output / down projection with the nGPT step fused: the CTAs
//               of a thread-block cluster hold the d / 256 column tiles of
//               the same 128 rows; y = the accumulator, and per row
//               h <- N(h + alpha (N(y) - h)) with both row norms summed over
//               the cluster through distributed shared memory; h is written
//               back as fp32 and as the bf16 copy the next GEMM reads.
//   EPI_PARTS   swapped operands for few activation rows (decode batches):
//               A = 128 weight rows, B = BN activation rows, and K split into
//               k_splits ranges so that even a 2048-wide projection spreads
//               over the SMs; each (weight tile, split) stores its fp32
//               partial sum transposed, out[split][m][n] (row = activation);
//               the consumers add the partials.
#pragma once
#include "ptx.cuh"
#include "quant.cuh"

namespace dory {

enum EpiKind { EPI_F32 = 0, EPI_QKVG = 1, EPI_SWIGLU = 2, EPI_PARTS = 3, EPI_NGPT = 4,
               EPI_QPARTS = 5 };

struct GemmArgs {
  int M, N, K;          // N: output columns of the GEMM (for SWIGLU: 2 * ffn)
  int tiles_m, tiles_n;
  int b_second;         // SWIGLU: row offset of W_sl inside B (= ffn)
  int* status;
  // EPI_F32
  float* out;
  long long ldo;
  const float* col_scale;   // may be null
  // EPI_QKVG
  __nv_bfloat16 *q, *k, *v, *g;
  int n_q, n_kv, head_dim;
  const float* s_qk;
  const float2* rope;       // [rows_per_seq][head_dim / 2] (cos, sin), or null
  // the same table transposed for the staged head_dim-128 epilogue, two
  // frequencies per entry: rope_t[j * rows_per_seq + t] =
  // (cos, sin of frequency 2j, cos, sin of frequency 2j + 1), or null
  const float4* rope_t;
  int rows_per_seq;
  // EPI_SWIGLU
  __nv_bfloat16* m_out;
  int ldm;
  // EPI_PARTS: M = weight rows (N of the projection), N = activation rows,
  // out[split * part_stride + n * ldo + m]
  int k_splits;
  long long part_stride;
  // EPI_F32 / EPI_SWIGLU with BN = 256: 1 if EpiMaps::out describes the
  // output (then it is written through shared memory), else direct stores
  int staged;
  // EPI_NGPT: h fp32 [M, N] (read, then rewritten through EpiMaps::out; the
  // bf16 copy through EpiMaps::hb) and alpha [N]; the cluster size is
  // tiles_n (N / 256 <= 8)
  const float* h32;
  const float* alpha;
  // EPI_QPARTS (EPI_PARTS with weight-only quantised weights): tmA maps the
  // packed codes (uint8 [M][K or K / 2]) and EpiMaps::q the block scales
  // (uint8 [M][K / 32 or K / 16], {16, 128} boxes); qfmt 1 MXFP8, 2 NVFP4;
  // qrow: NVFP4 row scales [M]
  int qfmt;
  const uint8_t* qscales;
  const float* qrow;
  // 1: the weight operand (A for EPI_PARTS, else B) never changes during the
  // forward pass, so the producer issues the weight loads of the first ring
  // stages before waiting on the previous kernel (programmatic launch); the
  // activation loads follow the wait.  0: every load after the wait.
  int w_pre;
};

template <int BN, int EPI = 0>
struct GemmCfg {
  static constexpr int BM = 128, BK = 64;
  // Staged epilogues keep their output tile in shared memory for TMA stores:
  // QKV+gate 2 halves x 128 x 128 bf16 (64 KB), fp32 2 halves x 2 buffers x
  // {32 x 128} fp32 (64 KB), SwiGLU 2 halves x {64 x 128} bf16 (32 KB).
  // The first two cost a stage of the operand ring.
  static constexpr bool PARTS = EPI == 3 || EPI == 5;
  static constexpr bool QA = EPI == 5;          // A: packed codes expanded in shared memory
  static constexpr bool STAGED = BN == 256 && !PARTS;
  static constexpr bool NGPT = EPI == 4;
  static constexpr uint32_t OUT_BYTES = !STAGED ? 0 : (EPI == 2 ? 2 * 16384 : 4 * 16384);
  static constexpr int STAGES = STAGED ? (EPI == 2 ? 4 : 3) : (BN == 256 || QA ? 4 : 6);
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  static constexpr uint32_t B_BYTES = BN * BK * 2;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static constexpr uint32_t BAR_BYTES = QA ? 512 : 256;
  // EPI_QPARTS: a ring of raw stages, deeper than the operand ring, each
  // holding a tile's codes for one k block (128 rows x 64 bytes for MXFP8,
  // 32 for NVFP4, with the 64- / 32-byte swizzle) and a 16-byte group of
  // each row's block scales (the k block's scales among them); warp 14
  // loads them, a converter warpgroup (warps 10..13) expands them into the
  // operand ring's bf16 A stages
  static constexpr int RAW_STAGES = QA ? 10 : 0;
  static constexpr uint32_t RAW_SCALES = BM * 16;
  static constexpr uint32_t RAW_STAGE = QA ? BM * BK + RAW_SCALES : 0;
  static constexpr int THREADS = QA ? 480 : 320;
  static constexpr uint32_t SQK_BYTES = EPI == 1 ? 512 : 0;   // s_qk of a 128-wide head
  // EPI_NGPT: alpha slice [256], half partial sums for y and u [2][128] each,
  // the cluster's per-row sums for y and u [8][128] each, two mbarriers
  static constexpr uint32_t NGPT_BYTES = NGPT ? (256 + 2 * 256 + 2 * 8 * 128) * 4 + 16 : 0;
  static constexpr uint32_t BASE_BYTES =
      STAGES * STAGE_BYTES + OUT_BYTES + BAR_BYTES + SQK_BYTES + NGPT_BYTES;
  static constexpr uint32_t RAW_OFF = (BASE_BYTES + 1023) / 1024 * 1024;   // swizzle-aligned
  static constexpr size_t SMEM = (QA ? RAW_OFF + RAW_STAGES * RAW_STAGE : BASE_BYTES) + 1024;
  // full, empty [STAGES]; tfull, tempty [2]; drain; TMEM slot + abort flag;
  // EPI_QPARTS: raw_full, raw_empty [RAW_STAGES], conv [STAGES]
  static_assert((2 * STAGES + 6 + 2 * RAW_STAGES + (QA ? STAGES : 0)) * 8 <= BAR_BYTES,
                "barrier area");
  static_assert(RAW_STAGE % 1024 == 0, "raw stages keep the swizzle alignment");
};

// Destination maps of the staged epilogues, all with the 128-byte swizzle:
//   QKV+gate  q, k, v, g: bf16 [M, heads x 128], {64 columns, 128 rows} boxes;
//   fp32      out: fp32 [M, N], {32 columns, 128 rows} boxes;
//   SwiGLU    out: bf16 [M, ffn], {64 columns, 128 rows} boxes;
//   nGPT      out: h fp32 [M, d], {32 columns, 128 rows} boxes; hb: h bf16
//             [M, d], {64 columns, 128 rows} boxes.
struct EpiMaps {
  CUtensorMap q, k, v, g, out, hb;
};

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + __expf(-x)); }
// epilogue form: reciprocal instead of a division
__device__ __forceinline__ float sigmoid_fast(float x) { return __frcp_rn(1.0f + __expf(-x)); }

// 16-byte chunk `chunk` (0..7) of row `r` of a 128-byte swizzled box
__device__ __forceinline__ uint4* sw128_chunk(uint8_t* box, int r, int chunk) {
  return reinterpret_cast<uint4*>(box + r * 128 + ((chunk ^ (r & 7)) << 4));
}

__device__ __forceinline__ void store_bf16x16(__nv_bfloat16* dst, const float* v) {
  uint4 a, b;
  a.x = pack_bf16x2(v[0], v[1]);   a.y = pack_bf16x2(v[2], v[3]);
  a.z = pack_bf16x2(v[4], v[5]);   a.w = pack_bf16x2(v[6], v[7]);
  b.x = pack_bf16x2(v[8], v[9]);   b.y = pack_bf16x2(v[10], v[11]);
  b.z = pack_bf16x2(v[12], v[13]); b.w = pack_bf16x2(v[14], v[15]);
  reinterpret_cast<uint4*>(dst)[0] = a;
  reinterpret_cast<uint4*>(dst)[1] = b;
}

// 16 fp32 values given as their bit patterns -> 16 bf16.
__device__ __forceinline__ void store_bf16x16_bits(__nv_bfloat16* dst, const uint32_t* r) {
  float v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
  store_bf16x16(dst, v);
}

// ------------------------------------------------------------- epilogues
template <int BN>
__device__ __forceinline__ void epi_f32(const GemmArgs& a, uint32_t tacc, int row, int n0,
                                        int c_lo, int c_hi) {
  const bool row_ok = row < a.M;
#pragma unroll 1
  for (int c = c_lo; c < c_hi; c += 16) {
    if (n0 + c >= a.N) break;                       // uniform across the warp
    float v[16];
    tmem_ld16(tacc + c, v);
    if (!row_ok) continue;
    float* dst = a.out + (long long)row * a.ldo + n0 + c;
    const int nvalid = min(16, a.N - n0 - c);
    if (a.col_scale) {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (i < nvalid) v[i] *= a.col_scale[n0 + c + i];
    }
    if (nvalid == 16 && (a.ldo & 3) == 0) {
#pragma unroll
      for (int i = 0; i < 16; i += 4)
        *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    } else {
      for (int i = 0; i < nvalid; ++i) dst[i] = v[i];
    }
  }
}

template <int BN>
__device__ __forceinline__ void epi_swiglu(const GemmArgs& a, uint32_t tacc, int row, int tn,
                                           int c_lo, int c_hi) {
  constexpr int H = BN / 2;
  const int col0 = tn * H;                          // column of m
#pragma unroll 1
  for (int c = c_lo; c < c_hi; c += 16) {
    float u[16], s[16];
    tmem_ld16(tacc + c, u);
    tmem_ld16(tacc + H + c, s);
    if (row < a.M) {
#pragma unroll
      for (int i = 0; i < 16; ++i) u[i] = u[i] * (s[i] * sigmoidf_(s[i]));
      store_bf16x16(a.m_out + (long long)row * a.ldm + col0 + c, u);
    }
  }
}

template <int BN>
__device__ __forceinline__ void epi_qkvg(const GemmArgs& a, uint32_t tacc, int row, int n0,
                                         int c_lo, int c_hi) {
  const int dh = a.head_dim, half = dh >> 1;
  const int nq = a.n_q, nkv = a.n_kv;
  const bool row_ok = row < a.M;
  const int t = row_ok ? row % a.rows_per_seq : 0;
#pragma unroll 1
  for (int hc = c_lo; hc < c_hi; hc += dh) {
    const int gcol = n0 + hc;
    if (gcol >= a.N) break;
    const int head = gcol / dh;
    if (head < nq + nkv) {
      // q or k head: RoPE, per-head L2 norm, s_qk (head_dim 128 takes the
      // staged epilogue instead)
      const bool is_q = head < nq;
      __nv_bfloat16* dst = is_q ? a.q + ((long long)row * nq + head) * dh
                                : a.k + ((long long)row * nkv + (head - nq)) * dh;
      float ss = 0.f;
#pragma unroll 1
      for (int c = 0; c < dh; c += 16) {
        float v[16];
        tmem_ld16(tacc + hc + c, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) ss += v[i] * v[i];
      }
      const float inv = 1.0f / sqrtf(fmaxf(ss, 1e-12f));
#pragma unroll 1
      for (int c = 0; c < half; c += 16) {
        float x1[16], x2[16];
        tmem_ld16(tacc + hc + c, x1);
        tmem_ld16(tacc + hc + half + c, x2);
        if (!row_ok) continue;
        if (a.rope) {
          const float2* cs = a.rope + (long long)t * half + c;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 r = cs[i];
            const float y1 = x1[i] * r.x - x2[i] * r.y;
            const float y2 = x2[i] * r.x + x1[i] * r.y;
            x1[i] = y1;
            x2[i] = y2;
          }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          x1[i] *= inv * a.s_qk[c + i];
          x2[i] *= inv * a.s_qk[half + c + i];
        }
        store_bf16x16(dst + c, x1);
        store_bf16x16(dst + half + c, x2);
      }
    } else if (head < nq + 2 * nkv) {
      __nv_bfloat16* dst = a.v + ((long long)row * nkv + (head - nq - nkv)) * dh;
#pragma unroll 1
      for (int c = 0; c < dh; c += 16) {
        float v[16];
        tmem_ld16(tacc + hc + c, v);
        if (row_ok) store_bf16x16(dst + c, v);
      }
    } else {
      __nv_bfloat16* dst = a.g + ((long long)row * nq + (head - nq - 2 * nkv)) * dh;
#pragma unroll 1
      for (int c = 0; c < dh; c += 16) {
        float v[16];
        tmem_ld16(tacc + hc + c, v);
        if (!row_ok) continue;
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = sigmoidf_(v[i]);
        store_bf16x16(dst + c, v);
      }
    }
  }
}

// Transposed partial store: this thread holds weight row `row` (projection
// feature) and BN activation rows (TMEM columns).
template <int BN>
__device__ __forceinline__ void epi_parts(const GemmArgs& a, uint32_t tacc, int row, int n0,
                                          int split, int c_lo, int c_hi) {
  float* dst = a.out + (long long)split * a.part_stride + row;
#pragma unroll 1
  for (int c = c_lo; c < c_hi; c += 16) {
    if (n0 + c >= a.N) break;                       // uniform across the warp
    float v[16];
    tmem_ld16(tacc + c, v);
    if (row >= a.M) continue;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (n0 + c + i < a.N) dst[(long long)(n0 + c + i) * a.ldo] = v[i];
  }
}

// QKV+gate epilogue for head_dim 128 through shared memory: this thread's
// row of the head block (RoPE / q-k norm / s_qk, copy, or sigmoid applied)
// goes into the 128 x 128 staging tile in the 128-byte swizzled layout; one
// thread of the 4-warp half then writes the tile with two TMA stores.
//
// RoPE (cos, sin) pairs come from the transposed table, so the 32 lanes of
// a warp (32 consecutive rows, i.e. positions) read 512 contiguous bytes per
// load.  The rotation runs in four passes of 16 pairs; the first pass's
// pairs are fetched before the accumulator wait, each later pass's during
// the pass before it.  s_qk is read from shared memory.
__device__ __forceinline__ bool qkvg_rope_head(const GemmArgs& a, int gcol) {
  return a.rope_t != nullptr && gcol / 128 < a.n_q + a.n_kv && gcol < a.N;
}

// (cos, sin) of frequencies [16 part, 16 part + 16) at this row's position
__device__ __forceinline__ void qkvg_rope_load(const GemmArgs& a, int row, bool use, int part,
                                               float4 (&cs)[8]) {
  const float4* p = a.rope_t + (use ? row % a.rows_per_seq : 0);
  const long long stride = a.rows_per_seq;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    cs[j] = use ? __ldg(p + (8 * part + j) * stride) : make_float4(1.f, 0.f, 1.f, 0.f);
}

__device__ __forceinline__ void epi_qkvg_staged(const GemmArgs& a, const EpiMaps& maps,
                                                const float* sqk, uint32_t tacc, int row,
                                                int rloc, int n0, int hc, uint8_t* stage, int half,
                                                bool leader, float4 (&cs)[8]) {
  if (n0 + hc >= a.N) return;                          // uniform for the half
  const int head = (n0 + hc) / 128;
  const int nq = a.n_q, nkv = a.n_kv;
  // staging tile free (its previous TMA store has read it)
  if (leader) bulk_wait_read0();
  named_bar(1 + half, 128);
  auto put16 = [&](int col, const uint32_t* bits) {   // 16 values at tile column col
#pragma unroll
    for (int h8 = 0; h8 < 2; ++h8) {
      const int c = col + 8 * h8;                      // 8-element chunk start
      uint4 u;
      u.x = pack_bf16x2(__uint_as_float(bits[8 * h8 + 0]), __uint_as_float(bits[8 * h8 + 1]));
      u.y = pack_bf16x2(__uint_as_float(bits[8 * h8 + 2]), __uint_as_float(bits[8 * h8 + 3]));
      u.z = pack_bf16x2(__uint_as_float(bits[8 * h8 + 4]), __uint_as_float(bits[8 * h8 + 5]));
      u.w = pack_bf16x2(__uint_as_float(bits[8 * h8 + 6]), __uint_as_float(bits[8 * h8 + 7]));
      *sw128_chunk(stage + (c >> 6) * 16384, rloc, (c & 63) >> 3) = u;
    }
  };
  const CUtensorMap* map;
  int x0;
  if (head < nq + nkv) {
    map = head < nq ? &maps.q : &maps.k;
    x0 = (head < nq ? head : head - nq) * 128;
    const bool use = qkvg_rope_head(a, n0 + hc) && row < a.M;
    float ss = 0.f;
#pragma unroll 1
    for (int c = 0; c < 128; c += 64) {
      uint32_t r0[32], r1[32];
      tmem_ld32_nowait(tacc + hc + c, r0);
      tmem_ld32_nowait(tacc + hc + c + 32, r1);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float u0 = __uint_as_float(r0[i]), u1 = __uint_as_float(r1[i]);
        ss = fmaf(u0, u0, ss);
        ss = fmaf(u1, u1, ss);
      }
    }
    const float inv = 1.0f / sqrtf(fmaxf(ss, 1e-12f));
    const float4* sq4 = reinterpret_cast<const float4*>(sqk);
#pragma unroll 1
    for (int qp = 0; qp < 4; ++qp) {                   // pairs (i, i + 64), i in [16 qp, 16 qp + 16)
      uint32_t r1[16], r2[16];
      tmem_ld16_nowait(tacc + hc + 16 * qp, r1);
      tmem_ld16_nowait(tacc + hc + 64 + 16 * qp, r2);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 4; ++j) {                    // 4 pairs per step
        const float4 s1 = sq4[4 * qp + j], s2 = sq4[16 + 4 * qp + j];
        const float sa[4] = {s1.x, s1.y, s1.z, s1.w}, sb[4] = {s2.x, s2.y, s2.z, s2.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = 4 * j + e;
          const float4 c4 = cs[i >> 1];
          const float co = (i & 1) ? c4.z : c4.x, si = (i & 1) ? c4.w : c4.y;
          const float u1 = __uint_as_float(r1[i]), u2 = __uint_as_float(r2[i]);
          const float y1 = u1 * co - u2 * si;
          const float y2 = u2 * co + u1 * si;
          r1[i] = __float_as_uint(y1 * (inv * sa[e]));
          r2[i] = __float_as_uint(y2 * (inv * sb[e]));
        }
      }
      if (qp < 3) qkvg_rope_load(a, row, use, qp + 1, cs);   // next pass's pairs
      put16(16 * qp, r1);
      put16(64 + 16 * qp, r2);
    }
  } else {
    const bool is_v = head < nq + 2 * nkv;
    map = is_v ? &maps.v : &maps.g;
    x0 = (is_v ? head - nq - nkv : head - nq - 2 * nkv) * 128;
#pragma unroll 1
    for (int c = 0; c < 128; c += 64) {
      uint32_t r0[32], r1[32];
      tmem_ld32_nowait(tacc + hc + c, r0);
      tmem_ld32_nowait(tacc + hc + c + 32, r1);
      tmem_wait_ld();
      if (!is_v) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          r0[i] = __float_as_uint(sigmoid_fast(__uint_as_float(r0[i])));
          r1[i] = __float_as_uint(sigmoid_fast(__uint_as_float(r1[i])));
        }
      }
      put16(c, r0);
      put16(c + 16, r0 + 16);
      put16(c + 32, r1);
      put16(c + 48, r1 + 16);
    }
  }
  fence_proxy_async_smem();
  named_bar(1 + half, 128);
  if (leader) {
    const int m0 = row - rloc;                         // first row of the tile
    tma_store_2d(map, stage, x0, m0);
    tma_store_2d(map, stage + 16384, x0 + 64, m0);
    bulk_commit();
  }
}

// fp32 epilogue through shared memory, 32 columns at a time: each thread's
// 32 values (one 128-byte row of a {32 x 128} fp32 box) go into one of the
// half's two 16 KB buffers and the half's leader stores the box with TMA.
// The buffers alternate (counter nst, kept across tiles); before the
// barrier that publishes chunk j the leader waits until the store of chunk
// j - 1 has read its buffer, which is the one chunk j + 1 writes.
__device__ __forceinline__ void epi_f32_staged(const GemmArgs& a, const CUtensorMap* map,
                                               uint32_t tacc, int rloc, int m0, int n0, int c_lo,
                                               int c_hi, uint8_t* stage, int half, bool leader,
                                               uint32_t& nst) {
#pragma unroll 1
  for (int c = c_lo; c < c_hi; c += 32) {
    if (n0 + c >= a.N) break;                          // uniform for the half
    uint32_t r[32];
    tmem_ld32_nowait(tacc + c, r);
    tmem_wait_ld();
    if (a.col_scale) {
      const int nvalid = min(32, a.N - n0 - c);
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < nvalid) r[i] = __float_as_uint(__uint_as_float(r[i]) * a.col_scale[n0 + c + i]);
    }
    uint8_t* buf = stage + (nst & 1) * 16384;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *sw128_chunk(buf, rloc, j) = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
    fence_proxy_async_smem();
    if (leader) bulk_wait_read0();
    named_bar(1 + half, 128);
    if (leader) {
      tma_store_2d(map, buf, n0 + c, m0);
      bulk_commit();
    }
    ++nst;
  }
}

// SwiGLU epilogue through shared memory: the half's 64 columns of m
// (bf16, one 128-byte row per thread) go into its {64 x 128} box buffer,
// stored by the half's leader with TMA.
template <int BN>
__device__ __forceinline__ void epi_swiglu_staged(const GemmArgs& a, const CUtensorMap* map,
                                                  uint32_t tacc, int rloc, int m0, int tn,
                                                  int c_lo, uint8_t* stage, int half,
                                                  bool leader) {
  constexpr int H = BN / 2;
  const int col = tn * H + c_lo;                       // first column of m
  if (col >= a.N / 2) return;                          // uniform for the half
  if (leader) bulk_wait_read0();
  named_bar(1 + half, 128);
#pragma unroll 1
  for (int c = 0; c < H / 2; c += 32) {
    uint32_t u[32], v[32];
    tmem_ld32_nowait(tacc + c_lo + c, u);
    tmem_ld32_nowait(tacc + H + c_lo + c, v);
    tmem_wait_ld();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float m[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float x = __uint_as_float(u[8 * q + i]), g = __uint_as_float(v[8 * q + i]);
        m[i] = x * (g * sigmoid_fast(g));
      }
      *sw128_chunk(stage, rloc, (c >> 3) + q) =
          make_uint4(pack_bf16x2(m[0], m[1]), pack_bf16x2(m[2], m[3]), pack_bf16x2(m[4], m[5]),
                     pack_bf16x2(m[6], m[7]));
    }
  }
  fence_proxy_async_smem();
  named_bar(1 + half, 128);
  if (leader) {
    tma_store_2d(map, stage, col, m0);
    bulk_commit();
  }
}

// Shared state of the fused nGPT epilogue (EPI_NGPT) in this CTA's shared
// memory; xy / xu [rank][row] receive every cluster CTA's per-row partial
// sums by st.async, each completing bytes on bar_y / bar_u.
struct NgptSmem {
  float* alpha;     // [256]   alpha of this CTA's columns
  float* part_y;    // [2][128] per-half sums of y^2
  float* part_u;    // [2][128] per-half sums of u^2
  float* xy;        // [8][128]
  float* xu;        // [8][128]
  uint64_t* bar_y;
  uint64_t* bar_u;
};

// Sends this row's CTA-level partial sum to slot [rank][rloc] of every CTA
// of the cluster (including this one).
__device__ __forceinline__ void ngpt_broadcast(float* x, uint64_t* bar, int cn, int rank, int rloc,
                                               float v) {
  const uint32_t la = smem_u32(x + rank * 128 + rloc), lb = smem_u32(bar);
  for (int p = 0; p < cn; ++p) st_async_f32(mapa_shared(la, p), v, mapa_shared(lb, p));
}

// One 128 x 128 half tile of the fused nGPT step; this thread owns row rloc
// and the half's 128 columns.  Phases of bar_y / bar_u: one per tile (ph).
// Returns false (uniformly for the 8 epilogue warps) when an exchange wait
// expired.
__device__ __forceinline__ bool epi_ngpt(const GemmArgs& a, const EpiMaps& maps,
                                         const NgptSmem& ns, uint32_t tacc, int rloc, int m0,
                                         int n0, int c_lo, uint8_t* stage, int half, bool leader,
                                         uint32_t& nst, uint32_t ph, int cn, int rank) {
  const int row = m0 + rloc;
  const bool row_ok = row < a.M;
  const float* hrow = a.h32 + (long long)(row_ok ? row : 0) * a.N + n0 + c_lo;
  const bool sender = half == 0;
  const bool exch_leader = threadIdx.x == 64;          // first epilogue thread
  // -- 1. sum of y^2 over the row (this half, then the CTA, then the cluster)
  float ss = 0.f;
#pragma unroll 1
  for (int c = 0; c < 128; c += 64) {
    uint32_t r0[32], r1[32];
    tmem_ld32_nowait(tacc + c_lo + c, r0);
    tmem_ld32_nowait(tacc + c_lo + c + 32, r1);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float u0 = __uint_as_float(r0[i]), u1 = __uint_as_float(r1[i]);
      ss = fmaf(u0, u0, ss);
      ss = fmaf(u1, u1, ss);
    }
  }
  ns.part_y[half * 128 + rloc] = ss;
  named_bar(3, 256);
  if (sender) ngpt_broadcast(ns.xy, ns.bar_y, cn, rank, rloc, ns.part_y[rloc] + ns.part_y[128 + rloc]);
  // h of this row's first 32 columns, loaded while the sums travel
  float4 hv[8];
#pragma unroll
  for (int j = 0; j < 8; ++j)
    hv[j] = row_ok ? __ldg(reinterpret_cast<const float4*>(hrow) + j) : make_float4(0.f, 0.f, 0.f, 0.f);
  bool ok = mbar_wait_bounded(ns.bar_y, ph, a.status, DEV_GEMM_NGPT);
  if (!named_bar_and(3, 256, ok)) return false;
  if (exch_leader) mbar_arrive_expect_tx(ns.bar_y, cn * 128 * 4);   // next tile's phase
  float sy = 0.f;
  for (int p = 0; p < cn; ++p) sy += ns.xy[p * 128 + rloc];
  const float inv_y = 1.0f / sqrtf(fmaxf(sy, 1e-12f));
  // -- 2. u = h + alpha (y / |y| - h), kept in TMEM; sum of u^2
  float su = 0.f;
#pragma unroll 1
  for (int c = 0; c < 128; c += 32) {
    uint32_t yv[32];
    tmem_ld32_nowait(tacc + c_lo + c, yv);
    tmem_wait_ld();
    const float4* al = reinterpret_cast<const float4*>(ns.alpha + c_lo + c);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 a4 = al[j];
      const float hh[4] = {hv[j].x, hv[j].y, hv[j].z, hv[j].w};
      const float aa[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float u = fmaf(aa[e], fmaf(__uint_as_float(yv[4 * j + e]), inv_y, -hh[e]), hh[e]);
        yv[4 * j + e] = __float_as_uint(u);
        su = fmaf(u, u, su);
      }
    }
    if (c + 32 < 128) {                                  // next 32 columns of h
#pragma unroll
      for (int j = 0; j < 8; ++j)
        hv[j] = row_ok ? __ldg(reinterpret_cast<const float4*>(hrow + c + 32) + j)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    tmem_st32(tacc + c_lo + c, yv);
  }
  tmem_wait_st();
  ns.part_u[half * 128 + rloc] = su;
  named_bar(3, 256);
  if (sender) ngpt_broadcast(ns.xu, ns.bar_u, cn, rank, rloc, ns.part_u[rloc] + ns.part_u[128 + rloc]);
  ok = mbar_wait_bounded(ns.bar_u, ph, a.status, DEV_GEMM_NGPT);
  if (!named_bar_and(3, 256, ok)) return false;
  if (exch_leader) mbar_arrive_expect_tx(ns.bar_u, cn * 128 * 4);
  float su_all = 0.f;
  for (int p = 0; p < cn; ++p) su_all += ns.xu[p * 128 + rloc];
  const float inv_u = 1.0f / sqrtf(fmaxf(su_all, 1e-12f));
  // -- 3. h = u / |u| as fp32 (two {32 x 128} boxes) and bf16 (one {64 x 128}
  // box) per 64 columns, through the half's two alternating 16 KB buffers
  auto publish = [&](const CUtensorMap* map, int x) {
    fence_proxy_async_smem();
    if (leader) bulk_wait_read0();
    named_bar(1 + half, 128);
    if (leader) {
      tma_store_2d(map, stage + (nst & 1) * 16384, x, m0);
      bulk_commit();
    }
    ++nst;
  };
#pragma unroll 1
  for (int c = 0; c < 128; c += 64) {
    uint32_t u[64];
    tmem_ld32_nowait(tacc + c_lo + c, u);
    tmem_ld32_nowait(tacc + c_lo + c + 32, u + 32);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 64; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * inv_u);
#pragma unroll
    for (int b = 0; b < 2; ++b) {                        // fp32 boxes
      uint8_t* buf = stage + (nst & 1) * 16384;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *sw128_chunk(buf, rloc, j) =
            make_uint4(u[32 * b + 4 * j], u[32 * b + 4 * j + 1], u[32 * b + 4 * j + 2],
                       u[32 * b + 4 * j + 3]);
      publish(&maps.out, n0 + c_lo + c + 32 * b);
    }
    {                                                    // bf16 box
      uint8_t* buf = stage + (nst & 1) * 16384;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *sw128_chunk(buf, rloc, j) = make_uint4(
            pack_bf16x2(__uint_as_float(u[8 * j]), __uint_as_float(u[8 * j + 1])),
            pack_bf16x2(__uint_as_float(u[8 * j + 2]), __uint_as_float(u[8 * j + 3])),
            pack_bf16x2(__uint_as_float(u[8 * j + 4]), __uint_as_float(u[8 * j + 5])),
            pack_bf16x2(__uint_as_float(u[8 * j + 6]), __uint_as_float(u[8 * j + 7])));
      publish(&maps.hb, n0 + c_lo + c);
    }
  }
  return true;
}

// ------------------------------------------------------------- the kernel
constexpr int kGemmThreads = 320;   // producer, MMA, 8 epilogue warps

template <int BN, int EPI>
__global__ void __launch_bounds__(GemmCfg<BN, EPI>::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmArgs args, const __grid_constant__ EpiMaps maps) {
  using C = GemmCfg<BN, EPI>;
  constexpr int BM = C::BM, BK = C::BK, STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* out_stage = smem + STAGES * C::STAGE_BYTES;          // STAGED: OUT_BYTES
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES + C::OUT_BYTES);
  float* sqk = reinterpret_cast<float*>(smem + STAGES * C::STAGE_BYTES + C::OUT_BYTES +
                                        C::BAR_BYTES);               // EPI_QKVG: s_qk[128]
  NgptSmem ns{};
  if (C::NGPT) {
    float* f = reinterpret_cast<float*>(smem + STAGES * C::STAGE_BYTES + C::OUT_BYTES +
                                        C::BAR_BYTES + C::SQK_BYTES);
    ns.alpha = f;
    ns.part_y = f + 256;
    ns.part_u = f + 512;
    ns.xy = f + 768;
    ns.xu = f + 768 + 1024;
    ns.bar_y = reinterpret_cast<uint64_t*>(f + 768 + 2048);
    ns.bar_u = ns.bar_y + 1;
  }
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* tfull_bar = empty_bar + STAGES;   // [2]
  uint64_t* tempty_bar = tfull_bar + 2;       // [2]
  uint64_t* drain_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* raw_full = drain_bar + 2;                 // EPI_QPARTS: [RAW_STAGES]
  uint64_t* raw_empty = raw_full + C::RAW_STAGES;     // EPI_QPARTS: [RAW_STAGES]
  uint64_t* conv_bar = raw_empty + C::RAW_STAGES;     // EPI_QPARTS: [STAGES]
  uint8_t* raw_base = smem + C::RAW_OFF;
  const int raw_row = C::QA ? (args.qfmt == 2 ? BK / 2 : BK) : 0;   // code bytes per row
  const uint32_t raw_bytes = (uint32_t)(BM * raw_row);
  const int sc_kb = args.qfmt == 2 ? 4 : 2;           // scale bytes per row and k block
  // codes and the 16-byte scale group of k block kb into raw stage s
  auto raw_load = [&](int s, int kb, int m0) {
    uint8_t* dst = raw_base + s * C::RAW_STAGE;
    mbar_arrive_expect_tx(&raw_full[s], raw_bytes + C::RAW_SCALES);
    tma_load_2d(dst, &tmA, &raw_full[s], kb * raw_row, m0);
    tma_load_2d(dst + raw_bytes, &maps.q, &raw_full[s], (kb * sc_kb) & ~15, m0);
  };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int splits = C::PARTS ? args.k_splits : 1;
  const int num_tiles = args.tiles_m * args.tiles_n * splits;
  const int KB = (args.K + BK - 1) / BK;
  // K blocks [kb_lo, kb_hi) of work unit `tile` (split = tile / (tiles_m tiles_n))
  auto kb_range = [&](int tile, int& lo, int& hi) {
    const int sp = tile / (args.tiles_m * args.tiles_n);
    lo = (int)((long long)sp * KB / splits);
    hi = (int)((long long)(sp + 1) * KB / splits);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 256);
    }
    mbar_init(drain_bar, 1);
    if (C::QA) {
      for (int s = 0; s < C::RAW_STAGES; ++s) {
        mbar_init(&raw_full[s], 1);
        mbar_init(&raw_empty[s], 4);                // one arrival per converter warp
      }
      for (int s = 0; s < STAGES; ++s) mbar_init(&conv_bar[s], 4);
    }
    if (C::NGPT) {
      mbar_init(ns.bar_y, 1);
      mbar_init(ns.bar_u, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
    if (C::NGPT) {                                  // phase 0: every cluster CTA's row sums
      mbar_arrive_expect_tx(ns.bar_y, args.tiles_n * 128 * 4);
      mbar_arrive_expect_tx(ns.bar_u, args.tiles_n * 128 * 4);
    }
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (C::QA) tma_prefetch_desc(&maps.q);
  }
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  // the exchange barriers of every CTA of the cluster exist before any
  // st.async reaches them
  if (C::NGPT) cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // (tile, k block) -> operand coordinates, in the producer's order
  auto coords = [&](int tile, int& m0, int& nb0, int& nb1) {
    const int tt = tile % (args.tiles_m * args.tiles_n);
    // EPI_NGPT: the cluster's CTAs take the tiles_n column tiles of a row block
    const int tm = C::NGPT ? tt / args.tiles_n : tt % args.tiles_m;
    const int tn = C::NGPT ? tt % args.tiles_n : tt / args.tiles_m;
    m0 = tm * BM;
    if (EPI == EPI_SWIGLU) {
      nb0 = tn * (BN / 2);
      nb1 = args.b_second + tn * (BN / 2);
    } else {
      nb0 = tn * BN;
      nb1 = tn * BN + BN / 2;
    }
  };
  // weights of the first ring stages, before the wait on the previous kernel
  // (each stage's barrier expects the whole stage; the activations complete it)
  int n_pre = 0;
  if (args.w_pre && !C::QA && warp == 0 && lane == 0) {
    for (int tile = blockIdx.x; tile < num_tiles && n_pre < STAGES; tile += gridDim.x) {
      int m0, nb0, nb1, kb_lo, kb_hi;
      coords(tile, m0, nb0, nb1);
      kb_range(tile, kb_lo, kb_hi);
      for (int kb = kb_lo; kb < kb_hi && n_pre < STAGES; ++kb, ++n_pre) {
        uint8_t* a_dst = smem + n_pre * C::STAGE_BYTES;
        uint8_t* b_dst = a_dst + C::A_BYTES;
        mbar_arrive_expect_tx(&full_bar[n_pre], C::STAGE_BYTES);
        if (EPI == EPI_PARTS) {
          tma_load_2d(a_dst, &tmA, &full_bar[n_pre], kb * BK, m0);
        } else {
          tma_load_2d(b_dst, &tmB, &full_bar[n_pre], kb * BK, nb0);
          tma_load_2d(b_dst + C::B_BYTES / 2, &tmB, &full_bar[n_pre], kb * BK, nb1);
        }
      }
    }
  }
  // set-up above overlaps the previous kernel; global memory it may have
  // written only from here (the code loads and their expansion read weights
  // only and start at once)
  if (!(C::QA && warp >= 10)) {
    pdl_wait();
    pdl_trigger();
  }

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int g = 0;                                    // k blocks issued so far
      for (int tile = blockIdx.x; tile < num_tiles && !*abort_flag; tile += gridDim.x) {
        int m0, nb0, nb1, kb_lo, kb_hi;
        coords(tile, m0, nb0, nb1);
        kb_range(tile, kb_lo, kb_hi);
        for (int kb = kb_lo; kb < kb_hi; ++kb, ++g) {
          if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1, args.status, DEV_GEMM_PRODUCER)) {
            *abort_flag = 1;
            break;
          }
          uint8_t* a_dst = smem + stage * C::STAGE_BYTES;
          uint8_t* b_dst = a_dst + C::A_BYTES;
          if (C::QA) {                              // activations; warp 14 loads the codes
            mbar_arrive_expect_tx(&full_bar[stage], C::B_BYTES);
            tma_load_2d(b_dst, &tmB, &full_bar[stage], kb * BK, nb0);
            tma_load_2d(b_dst + C::B_BYTES / 2, &tmB, &full_bar[stage], kb * BK, nb1);
          } else if (g < n_pre) {                   // weights already on their way
            if (EPI == EPI_PARTS) {
              tma_load_2d(b_dst, &tmB, &full_bar[stage], kb * BK, nb0);
              tma_load_2d(b_dst + C::B_BYTES / 2, &tmB, &full_bar[stage], kb * BK, nb1);
            } else {
              tma_load_2d(a_dst, &tmA, &full_bar[stage], kb * BK, m0);
            }
          } else {
            mbar_arrive_expect_tx(&full_bar[stage], C::STAGE_BYTES);
            tma_load_2d(a_dst, &tmA, &full_bar[stage], kb * BK, m0);
            tma_load_2d(b_dst, &tmB, &full_bar[stage], kb * BK, nb0);
            tma_load_2d(b_dst + C::B_BYTES / 2, &tmB, &full_bar[stage], kb * BK, nb1);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc_idesc_bf16(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int tile = blockIdx.x; tile < num_tiles && !*abort_flag; tile += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!mbar_wait_bounded(&tempty_bar[acc], aph ^ 1, args.status, DEV_GEMM_MMA_TMEM)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        bool ok = true;
        int kb_lo, kb_hi;
        kb_range(tile, kb_lo, kb_hi);
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (!mbar_wait_bounded(&full_bar[stage], phase, args.status, DEV_GEMM_MMA_FULL) ||
              (C::QA &&
               !mbar_wait_bounded(&conv_bar[stage], phase, args.status, DEV_GEMM_MMA_FULL))) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + stage * C::STAGE_BYTES);
          const uint64_t adesc = tc_sdesc_sw128(a_addr);
          const uint64_t bdesc = tc_sdesc_sw128(a_addr + C::A_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            // +32 bytes per 16-element K step inside the swizzled 128-byte row
            tc_mma_bf16(d_tmem, adesc + 2 * k, bdesc + 2 * k, idesc, (kb - kb_lo) | k);
          }
          tc_commit(&empty_bar[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(&tfull_bar[acc]);
      }
      // no MMA may be in flight when TMEM is released
      tc_commit(drain_bar);
      mbar_wait_bounded(drain_bar, 0, args.status, DEV_GEMM_DRAIN);
    }
    __syncwarp();
  } else if (C::QA && warp == 14) {
    // ------------------------------------------------ code loads (warp 14)
    if (lane == 0) {
      int rs = 0;
      uint32_t rph = 0;
      for (int tile = blockIdx.x; tile < num_tiles && !*abort_flag; tile += gridDim.x) {
        int m0, nb0, nb1, kb_lo, kb_hi;
        coords(tile, m0, nb0, nb1);
        kb_range(tile, kb_lo, kb_hi);
        bool ok = true;
        for (int kb = kb_lo; kb < kb_hi; ++kb) {
          if (!mbar_wait_bounded(&raw_empty[rs], rph ^ 1, args.status, DEV_GEMM_PRODUCER)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          raw_load(rs, kb, m0);
          if (++rs == C::RAW_STAGES) {
            rs = 0;
            rph ^= 1;
          }
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (C::QA && warp >= 10) {
    // ------------------------------------------------ code expansion (warps 10..13)
    // thread r expands row r of each tile's k block into the bf16 A stage
    // (128-byte swizzle, as TMA would have written it) with the block scale
    // (and the NVFP4 row scale): the values of the dequantised bf16 matrix
    const int r = threadIdx.x - 320;
    const bool fp4 = args.qfmt == 2;
    // the raw rows carry the 64-byte (MXFP8) / 32-byte (NVFP4) swizzle:
    // 16-byte chunk q of row r sits at chunk q ^ sw of the row
    const int sw = fp4 ? (r >> 2) & 1 : (r >> 1) & 3;
    int stage = 0, rst = 0;
    uint32_t phase = 0, rph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles && ok && !*abort_flag; tile += gridDim.x) {
      int m0, nb0, nb1, kb_lo, kb_hi;
      coords(tile, m0, nb0, nb1);
      kb_range(tile, kb_lo, kb_hi);
      const int row = m0 + r;
      const bool rv = row < args.M;
      const float rs = (fp4 && rv && args.qrow) ? args.qrow[row] : 1.0f;
      for (int kb = kb_lo; kb < kb_hi; ++kb) {
        const bool w_ok =
            !*abort_flag &&
            mbar_wait_bounded(&empty_bar[stage], phase ^ 1, args.status, DEV_GEMM_CONV) &&
            mbar_wait_bounded(&raw_full[rst], rph, args.status, DEV_GEMM_CONV);
        if (!__all_sync(0xffffffffu, w_ok)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        uint8_t* a_st = smem + stage * C::STAGE_BYTES;
        const uint4* raw = reinterpret_cast<const uint4*>(raw_base + rst * C::RAW_STAGE +
                                                          r * raw_row);
        // this k block's scales: bytes (kb sc_kb) mod 16 .. of the row's group
        const uint32_t sword = *reinterpret_cast<const uint32_t*>(
            raw_base + rst * C::RAW_STAGE + raw_bytes + r * 16 + ((kb * sc_kb) & 12));
        uint32_t pk[32];
        if (!rv) {
#pragma unroll
          for (int i = 0; i < 32; ++i) pk[i] = 0u;
        } else if (!fp4) {
          const uint32_t sh = 8 * ((kb * 2) & 3);
          const float s0 = e8m0_to_f32((sword >> sh) & 0xFFu),
                      s1 = e8m0_to_f32((sword >> (sh + 8)) & 0xFFu);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 v = raw[q ^ sw];
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
            const float s = q < 2 ? s0 : s1;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              float f[4];
              e4m3x4_to_f32(w4[t], f);
              pk[q * 8 + 2 * t] = pack_bf16x2(f[0] * s, f[1] * s);
              pk[q * 8 + 2 * t + 1] = pack_bf16x2(f[2] * s, f[3] * s);
            }
          }
        } else {
          const uint32_t s4 = sword;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const uint4 v = raw[q ^ sw];
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {                  // 8 codes of block 2q + t / 2
              const float s = e4m3_to_f32((s4 >> (8 * (2 * q + t / 2))) & 0xFFu);
              float f[8];
              e2m1x8_to_f32(w4[t], f);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                pk[q * 16 + 4 * t + i] =
                    pack_bf16x2(__fmul_rn(f[2 * i] * s, rs), __fmul_rn(f[2 * i + 1] * s, rs));
            }
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *sw128_chunk(a_st, r, j) = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2],
                                                pk[4 * j + 3]);
        fence_proxy_async_smem();                   // visible to the tensor cores
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&conv_bar[stage]);
          mbar_arrive(&raw_empty[rst]);              // this warp's reads of the raw stage are done
        }
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
        if (++rst == C::RAW_STAGES) {
          rst = 0;
          rph ^= 1;
        }
      }
    }
  } else {
    // ------------------------------------------------ epilogue warps 2..9
    const int quarter = warp & 3;
    const int chalf = (warp - 2) >> 2;            // which half of the columns
    const bool leader = (warp & 3) == 2 && lane == 0;   // one thread per half
    constexpr int OUT_HALF = C::OUT_BYTES / 2;
    uint8_t* my_stage = out_stage + chalf * OUT_HALF;
    const bool staged =
        C::STAGED && (EPI == EPI_QKVG ? args.head_dim == 128 : (C::NGPT || args.staged != 0));
    uint32_t nst = 0;                             // fp32: boxes this half has staged
    if (EPI == EPI_QKVG && C::STAGED) {
      const int e = threadIdx.x - 64;
      if (e < 128) sqk[e] = args.s_qk && e < args.head_dim ? args.s_qk[e] : 1.0f;
      named_bar(3, 256);
    }
    const int ng_rank = C::NGPT ? (int)(blockIdx.x % args.tiles_n) : 0;   // = cluster rank
    if (C::NGPT) {                                  // alpha of this CTA's 256 columns
      const int e = threadIdx.x - 64;
      const int col = ng_rank * BN + e;
      ns.alpha[e] = col < args.N ? args.alpha[col] : 0.f;
      named_bar(3, 256);
    }
    int it = 0;
    // tcgen05.ld is warp-collective and the staged epilogue synchronises its
    // 4-warp half on a hardware barrier, so the go / stop decision for a tile
    // is made uniform across the warp (across the half when staged)
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      const int tt = tile % (args.tiles_m * args.tiles_n);
      const int tm = C::NGPT ? tt / args.tiles_n : tt % args.tiles_m;
      const int tn = C::NGPT ? tt % args.tiles_n : tt / args.tiles_m;
      const int row = tm * BM + quarter * 32 + lane;
      constexpr int CW = (EPI == EPI_SWIGLU ? BN / 2 : BN) / 2;   // columns per half
      const int c_lo = chalf * CW, c_hi = c_lo + CW;
      // RoPE pairs of this row are fetched while the accumulator is computed
      float4 cs[8];
      if (EPI == EPI_QKVG && C::STAGED && staged)
        qkvg_rope_load(args, row, qkvg_rope_head(args, tn * BN + c_lo) && row < args.M, 0, cs);
      bool ready = !*abort_flag &&
                   mbar_wait_bounded(&tfull_bar[acc], aph, args.status, DEV_GEMM_EPI);
      // (EPI_NGPT: uniform over all 8 epilogue warps, which meet at one barrier)
      ready = C::NGPT      ? named_bar_and(3, 256, ready)
              : C::STAGED ? named_bar_and(1 + chalf, 128, ready)
                          : __all_sync(0xffffffffu, ready);
      if (!ready) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tacc = tmem_base + acc * BN + ((uint32_t)(quarter * 32) << 16);
      const int rloc = quarter * 32 + lane, m0 = tm * BM;
      if (EPI == EPI_F32) {
        if (C::STAGED && staged)
          epi_f32_staged(args, &maps.out, tacc, rloc, m0, tn * BN, c_lo, c_hi, my_stage, chalf,
                         leader, nst);
        else
          epi_f32<BN>(args, tacc, row, tn * BN, c_lo, c_hi);
      }
      if (EPI == EPI_QKVG) {
        if (C::STAGED && staged)
          epi_qkvg_staged(args, maps, sqk, tacc, row, rloc, tn * BN, c_lo, my_stage, chalf,
                          leader, cs);
        else
          epi_qkvg<BN>(args, tacc, row, tn * BN, c_lo, c_hi);
      }
      if (EPI == EPI_SWIGLU) {
        if (C::STAGED && staged)
          epi_swiglu_staged<BN>(args, &maps.out, tacc, rloc, m0, tn, c_lo, my_stage, chalf,
                                leader);
        else
          epi_swiglu<BN>(args, tacc, row, tn, c_lo, c_hi);
      }
      if (C::PARTS)
        epi_parts<BN>(args, tacc, row, tn * BN, tile / (args.tiles_m * args.tiles_n), c_lo, c_hi);
      if (C::NGPT) {
        if (!epi_ngpt(args, maps, ns, tacc, rloc, m0, tn * BN, c_lo, my_stage, chalf, leader, nst,
                      (uint32_t)(it & 1), args.tiles_n, ng_rank)) {
          *abort_flag = 1;
          break;
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty_bar[acc]);
    }
    // staged stores must have completed before the CTA (and its shared
    // memory) goes away
    if (C::STAGED && leader) bulk_wait0();
  }

  if (*abort_flag) {
    // error path: give in-flight bulk copies time to land before the CTA's
    // shared memory is released
    for (int i = 0; i < 64; ++i) __nanosleep(1000);
  }
  // no CTA of the cluster leaves while another may still write its shared
  // memory (every exchange wait above is bounded, so all threads get here)
  if (C::NGPT) cluster_sync();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace dory
