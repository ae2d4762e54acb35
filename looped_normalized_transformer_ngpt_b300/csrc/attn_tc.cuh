// attn_tc.cuh - prefill attention on the 5th-generation tensor cores
// (tcgen05, operands fed by TMA, accumulators in TMEM), head_dim 128.
//
// Same operation as attn_prefill_kernel ("Dory1.0-4B: A Looped
// Normalized-GPT", Architecture; Last-Loop KV Caching): for every query
// position t of the call and query head h,
//   o_h(t) = sum_j softmax_j(scale * q_h(t) . k_{h/G}(j)) v_{h/G}(j),
//   j visible iff j <= t and (full layer or t - j < W),
// keys of positions < P0 from the cache slice, the others from this call's
// projections; out = o * sigmoid(g) (bf16).
//
// One CTA = (block of 128 / G query positions, kv head, sequence): its 128
// rows are (position, head-in-group) pairs, so one K/V tile serves all G
// heads.  96 KB of shared memory and 256 TMEM columns, so two CTAs share an
// SM and the tensor core works for one while the other runs its softmax.
// Warp roles (224 threads):
//   warp 0    TMA producer of Q and K: the Q tile once per item (3-D box: 64
//             dims x G heads x 128/G positions, two boxes for the 128 dims),
//             then 64-key K tiles into a 2-stage ring (128-byte swizzle); a K
//             stage is released when its S MMA completes, so K runs up to two
//             tiles ahead of the softmax;
//   warp 6    TMA producer of V: 64-key V tiles into their own 2-stage ring,
//             a stage released when its PV MMA completes;
//   warp 1    TMEM owner and MMA issuer: S_j = Q K_j^T (M = 128, N = 64,
//             K = 128) into TMEM S buffer j % 2, and O += P_j V_j into the TMEM
//             O accumulator with P_j read from TMEM (A operand) and V as an
//             MN-major shared-memory operand;
//   warps 2-5 softmax, one row per thread: S row from TMEM, mask (only on
//             tiles that need one, decided once per tile), running max,
//             P = exp2(S - max) packed to bf16 pairs and written back over the
//             first 32 columns of the same S buffer (so P is double-buffered
//             with S and the exponentials of tile j overlap the PV MMA of
//             tile j - 1); O is rescaled in TMEM only when the running max
//             rises by more than 8 (log2 units) - otherwise the stale max
//             stays exact, since the same max scales P and the row sum; final
//             O / sum * gate from TMEM to global.
// One thread issues every MMA and the MMAs of one thread run in order, so
// S_{j+2} (issued after PV_j) never overwrites P_j before PV_j has read it.
// Key tiles are aligned to 64 positions and never mix cached and current
// keys (the launcher requires P0 % 64 == 0 and 64-aligned ring sizes).
// Every wait is bounded (status word + orderly exit).
#pragma once
#include "ptx.cuh"

namespace dory {

struct AttnTcArgs {
  int C, P0, S;               // tokens per sequence in the call, first position, cache slots
  int n_kv, G;                // kv heads, query heads per kv head
  int window;                 // 0 = full causal
  float scale_log2;
  const __nv_bfloat16* gate;  // [B*C, n_q*128] sigmoid(g)
  __nv_bfloat16* out;         // [B*C, n_q*128]
  int n_q;
  int B;                      // sequences
  int* status;
};

struct AttnTcCfg {
  static constexpr int BK = 64;                  // keys per tile
  static constexpr int QHALF = 128 * 128;        // Q: one 64-dim half of the 128 rows (bytes)
  static constexpr int KVHALF = BK * 128;        // K or V: one 64-dim half of the BK rows
  static constexpr int KVTILE = 2 * KVHALF;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = 2 * QHALF;          // 2 stages
  static constexpr int V_OFF = K_OFF + 2 * KVTILE; // 2 stages
  static constexpr int BAR_OFF = V_OFF + 2 * KVTILE;
  static constexpr size_t SMEM = BAR_OFF + 256;    // two CTAs fit on one SM
  // S0 | S1 (64 fp32 columns each; P_j as 32 columns of bf16 pairs over S_j)
  // | O (128)
  static constexpr uint32_t TMEM_COLS = 256;
};

// tensor maps: q (3-D: dim, head, token), k/v current (3-D: dim, kv head,
// token), k/v cache (2-D: dim, slot row).  One 64-key K or V tile (both
// 64-dim halves) starting at key position j0: from the cache slice below P0,
// else from this call's projections.
__device__ __forceinline__ void attn_tc_load_tile(uint8_t* dst, const CUtensorMap* t_cache,
                                                  const CUtensorMap* t_cur, uint64_t* bar, int j0,
                                                  int b, int kvh, const AttnTcArgs& a) {
  if (j0 < a.P0) {
    const int row = (b * a.n_kv + kvh) * a.S + (j0 % a.S);
    tma_load_2d(dst, t_cache, bar, 0, row);
    tma_load_2d(dst + AttnTcCfg::KVHALF, t_cache, bar, 64, row);
  } else {
    const int tok = b * a.C + (j0 - a.P0);
    tma_load_3d(dst, t_cur, bar, 0, kvh, tok);
    tma_load_3d(dst + AttnTcCfg::KVHALF, t_cur, bar, 64, kvh, tok);
  }
}

// Geometry of one work item (query block qb of one (kv head, sequence)).
struct AttnTcItem {
  int kvh, b, q0, nqv, p_lo, p_hi, t_first, ntiles;
};

__device__ __forceinline__ AttnTcItem attn_tc_item(const AttnTcArgs& a, int item) {
  AttnTcItem it;
  const int QP = 128 / a.G;
  const int nqb = (a.C + QP - 1) / QP;
  const int per_q = a.n_kv * a.B;
  const int qb = nqb - 1 - item / per_q;                 // longest query blocks first
  const int rem = item % per_q;
  it.kvh = rem % a.n_kv;
  it.b = rem / a.n_kv;
  it.q0 = qb * QP;
  it.nqv = min(QP, a.C - it.q0);
  it.p_lo = a.P0 + it.q0;
  it.p_hi = a.P0 + it.q0 + it.nqv - 1;
  const int k_lo = a.window > 0 ? max(0, it.p_lo - a.window + 1) : 0;
  it.t_first = k_lo / AttnTcCfg::BK;
  it.ntiles = it.p_hi / AttnTcCfg::BK - it.t_first + 1;
  return it;
}

constexpr int kAttnTcThreads = 224;

__global__ void __launch_bounds__(kAttnTcThreads, 2)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_kc,
                   const __grid_constant__ CUtensorMap tm_vc, const AttnTcArgs a) {
  using Cf = AttnTcCfg;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  // the 128-byte swizzle atoms need 1024-byte alignment; the dynamic segment
  // of this kernel (no static shared memory) starts there
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0 && a.status) atomicCAS(a.status, 0, DEV_ATTN_ALIGN);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cf::BAR_OFF);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;     // [2]
  uint64_t* k_empty = bars + 4;    // [2]
  uint64_t* v_full = bars + 6;     // [2]
  uint64_t* v_empty = bars + 8;    // [2]
  uint64_t* s_full = bars + 10;    // [2]
  uint64_t* p_full = bars + 12;
  uint64_t* o_done = bars + 13;
  uint64_t* o_free = bars + 14;
  uint64_t* drain = bars + 15;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int QP = 128 / a.G;
  const int n_items = ((a.C + QP - 1) / QP) * a.n_kv * a.B;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
    }
    mbar_init(p_full, 128);
    mbar_init(o_done, 1);
    mbar_init(o_free, 128);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_kc);
    tma_prefetch_desc(&tm_vc);
  }
  if (warp == 1) tmem_alloc(tmem_slot, Cf::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;   // S0: cols 0..63, S1: 64..127, O: 128..255
  pdl_wait();
  pdl_trigger();

  // Work items are strided over the CTAs of the grid (no more than are
  // resident); barrier phases run on across items: g counts key tiles, n
  // counts this CTA's items.
  if (warp == 0) {
    // ------------------------------------------------ TMA producer: Q and K
    if (lane == 0) {
      int g = 0, n = 0;
      for (int item = blockIdx.x; item < n_items && !*abort_flag; item += gridDim.x, ++n) {
        const AttnTcItem it = attn_tc_item(a, item);
        if (n >= 1 && !mbar_wait_bounded(q_empty, (n - 1) & 1, a.status, DEV_ATTN_PRODUCER)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(q_full, 2 * Cf::QHALF);
        const int tok = it.b * a.C + it.q0;
        tma_load_3d(smem + Cf::Q_OFF, &tm_q, q_full, 0, it.kvh * a.G, tok);
        tma_load_3d(smem + Cf::Q_OFF + Cf::QHALF, &tm_q, q_full, 64, it.kvh * a.G, tok);
        for (int j = 0; j < it.ntiles; ++j, ++g) {
          const int st = g & 1;
          if (g >= 2 && !mbar_wait_bounded(&k_empty[st], ((g >> 1) - 1) & 1, a.status,
                                           DEV_ATTN_PRODUCER)) {
            *abort_flag = 1;
            break;
          }
          mbar_arrive_expect_tx(&k_full[st], Cf::KVTILE);
          attn_tc_load_tile(smem + Cf::K_OFF + st * Cf::KVTILE, &tm_kc, &tm_k, &k_full[st],
                            (it.t_first + j) * Cf::BK, it.b, it.kvh, a);
        }
        if (*abort_flag) break;
      }
    }
  } else if (warp == 6) {
    // ------------------------------------------------ TMA producer: V
    if (lane == 0) {
      int g = 0;
      for (int item = blockIdx.x; item < n_items && !*abort_flag; item += gridDim.x) {
        const AttnTcItem it = attn_tc_item(a, item);
        for (int j = 0; j < it.ntiles; ++j, ++g) {
          const int st = g & 1;
          if (g >= 2 && !mbar_wait_bounded(&v_empty[st], ((g >> 1) - 1) & 1, a.status,
                                           DEV_ATTN_PRODUCER)) {
            *abort_flag = 1;
            break;
          }
          mbar_arrive_expect_tx(&v_full[st], Cf::KVTILE);
          attn_tc_load_tile(smem + Cf::V_OFF + st * Cf::KVTILE, &tm_vc, &tm_v, &v_full[st],
                            (it.t_first + j) * Cf::BK, it.b, it.kvh, a);
        }
        if (*abort_flag) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc_idesc_bf16(128, Cf::BK);
      constexpr uint32_t idesc_o = tc_idesc_bf16(128, 128) | (1u << 16);   // B (V) MN-major
      const uint32_t q_addr = smem_u32(smem + Cf::Q_OFF);
      // S_g reuses the TMEM buffer of tile g - 2, whose softmax finished (its
      // p_full was waited for) and whose PV MMA was issued before this one
      auto issue_s = [&](int g) -> bool {
        const int st = g & 1;
        if (!mbar_wait_bounded(&k_full[st], (g >> 1) & 1, a.status, DEV_ATTN_MMA)) return false;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(smem + Cf::K_OFF + st * Cf::KVTILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t qo = (kk >> 2) * Cf::QHALF + (kk & 3) * 32;
          const uint32_t ko = (kk >> 2) * Cf::KVHALF + (kk & 3) * 32;
          tc_mma_bf16(tmem + st * Cf::BK, tc_sdesc_sw128(q_addr + qo), tc_sdesc_sw128(k_addr + ko),
                      idesc_s, kk);
        }
        tc_commit(&s_full[st]);
        tc_commit(&k_empty[st]);                  // K stage free once S_g is computed
        return true;
      };
      bool ok = true;
      int g = 0, n = 0;
      for (int item = blockIdx.x; ok && item < n_items && !*abort_flag; item += gridDim.x, ++n) {
        const AttnTcItem it = attn_tc_item(a, item);
        ok = mbar_wait_bounded(q_full, n & 1, a.status, DEV_ATTN_MMA) && issue_s(g);
        for (int j = 0; ok && j < it.ntiles && !*abort_flag; ++j) {
          const int gj = g + j;
          if (j + 1 < it.ntiles) {
            if (!issue_s(gj + 1)) {
              ok = false;
              break;
            }
          } else {
            tc_commit(q_empty);                   // Q free once this item's S MMAs are done
          }
          const int st = gj & 1;
          if (!mbar_wait_bounded(p_full, gj & 1, a.status, DEV_ATTN_MMA) ||
              !mbar_wait_bounded(&v_full[st], (gj >> 1) & 1, a.status, DEV_ATTN_MMA) ||
              (j == 0 && n >= 1 && !mbar_wait_bounded(o_free, (n - 1) & 1, a.status, DEV_ATTN_MMA))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t v_addr = smem_u32(smem + Cf::V_OFF + st * Cf::KVTILE);
#pragma unroll
          for (int kk = 0; kk < Cf::BK / 16; ++kk) {
            // A = P (128 rows x 16 keys: 8 TMEM columns of bf16 pairs), B = V
            // (16 keys x 128 dims, MN-major: the two 64-dim halves KVHALF
            // apart, 8-key groups 1024 B apart)
            tc_mma_bf16_ts(tmem + 2 * Cf::BK, tmem + st * Cf::BK + kk * 8,
                           tc_sdesc_sw128_mn(v_addr + kk * 2048, Cf::KVHALF, 1024), idesc_o,
                           (j | kk) != 0);
          }
          tc_commit(&v_empty[st]);
          tc_commit(o_done);
        }
        g += it.ntiles;
      }
      if (!ok) *abort_flag = 1;
      tc_commit(drain);
      mbar_wait_bounded(drain, 0, a.status, DEV_ATTN_DRAIN);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax warps 2..5
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                  // tile row = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    bool ok = true;
    int g = 0, n = 0;
    // tcgen05.ld / tcgen05.st are warp-collective: every decision that guards
    // them (abort, rescale) is made uniform across the warp.
    for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x, ++n) {
      const AttnTcItem it = attn_tc_item(a, item);
      const int i = r / a.G, hg = r % a.G;
      const bool row_ok = i < it.nqv;
      const int qpos = it.p_lo + i;
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < it.ntiles; ++j) {
        const int gj = g + j, st = gj & 1;
        bool w_ok = !*abort_flag &&
                    mbar_wait_bounded(&s_full[st], (gj >> 1) & 1, a.status, DEV_ATTN_SOFTMAX);
        if (!__all_sync(0xffffffffu, w_ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sv[Cf::BK];
#pragma unroll
        for (int c = 0; c < Cf::BK / 32; ++c)
          tmem_ld32_nowait(tmem + st * Cf::BK + lane_off + c * 32, sv + c * 32);
        tmem_wait_ld();
        // Mask (raw scores; scale > 0 keeps the order).  Whether the tile needs
        // a mask at all is uniform for the item (all keys visible to all of
        // its query positions, all 128 rows real), so the common case is a
        // plain maximum; otherwise key j0 + c is visible to this row iff
        // lo < c <= hi.
        const int j0 = (it.t_first + j) * Cf::BK;
        const bool plain = it.nqv * a.G == 128 && j0 + Cf::BK - 1 <= it.p_lo &&
                           (a.window <= 0 || it.p_hi - j0 < a.window);
        float mx;
        if (plain) {
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < Cf::BK; c += 8) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
              m4[u] = max3f(m4[u], __uint_as_float(sv[c + 2 * u]), __uint_as_float(sv[c + 2 * u + 1]));
          }
          mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        } else {
          const int hi = row_ok ? qpos - j0 : -1;
          const int lo = a.window > 0 ? qpos - j0 - a.window : -0x7fffffff;
          float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < Cf::BK; ++c) {
            const float v = (c <= hi && c > lo) ? __uint_as_float(sv[c]) : -INFINITY;
            sv[c] = __float_as_uint(v);
            m4[c & 3] = fmaxf(m4[c & 3], v);
          }
          mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        }
        mx *= a.scale_log2;
        float scale_o = 1.f;
        bool rescale = false;
        if (mx > m_run + 8.0f) {                     // stale max kept unless it grows by > 2^8
          scale_o = m_run == -INFINITY ? 0.f : ex2_ftz(m_run - mx);
          rescale = j > 0;
          l_run *= scale_o;
          m_run = mx;
        }
        const float m_use = m_run == -INFINITY ? 0.f : m_run;
        // P as bf16 pairs (key 2c in the low half of column c); the exponent
        // arguments and the row sum are formed two keys per instruction
        uint32_t pk[Cf::BK / 2];
        const unsigned long long sc2 = f32x2_pack(a.scale_log2, a.scale_log2);
        const unsigned long long nm2 = f32x2_pack(-m_use, -m_use);
        unsigned long long sum_a = f32x2_pack(0.f, 0.f), sum_b = sum_a;
#pragma unroll
        for (int c = 0; c < Cf::BK / 2; ++c) {
          float x0, x1;
          f32x2_unpack(f32x2_fma(f32x2_pack(__uint_as_float(sv[2 * c]),
                                            __uint_as_float(sv[2 * c + 1])),
                                 sc2, nm2),
                       x0, x1);
          const float p0 = ex2_ftz(x0), p1 = ex2_ftz(x1);
          if (c & 1)
            sum_b = f32x2_add(sum_b, f32x2_pack(p0, p1));
          else
            sum_a = f32x2_add(sum_a, f32x2_pack(p0, p1));
          pk[c] = pack_bf16x2(p0, p1);
        }
        float ls4[4];
        f32x2_unpack(sum_a, ls4[0], ls4[1]);
        f32x2_unpack(sum_b, ls4[2], ls4[3]);
        l_run += (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
        // O holds PV_{j-1} once o_done completed that phase (waited for every
        // tile, after the exponentials, so they overlap that MMA)
        w_ok = gj == 0 || mbar_wait_bounded(o_done, (gj - 1) & 1, a.status, DEV_ATTN_SOFTMAX);
        if (!__all_sync(0xffffffffu, w_ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, rescale)) {      // lanes without a rescale scale by 1
          if (!rescale) scale_o = 1.f;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t ov[32];
            tmem_ld32_nowait(tmem + 2 * Cf::BK + lane_off + c * 32, ov);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * scale_o);
            tmem_st32(tmem + 2 * Cf::BK + lane_off + c * 32, ov);
          }
        }
        tmem_st32(tmem + st * Cf::BK + lane_off, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_full);
      }
      if (!ok) break;
      // final: O / l * gate, then O is free for the next item.  The gate row
      // of this thread (256 bytes) is loaded before the wait for the last PV
      // MMA, so its latency overlaps that MMA instead of the output loop.
      const long long row = (long long)it.b * a.C + it.q0 + i;
      const long long base = row * a.n_q * 128 + (long long)(it.kvh * a.G + hg) * 128;
      uint4 gr[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        gr[e] = row_ok ? __ldg(reinterpret_cast<const uint4*>(a.gate + base) + e)
                       : make_uint4(0u, 0u, 0u, 0u);
      bool fin = !*abort_flag && mbar_wait_bounded(o_done, (g + it.ntiles - 1) & 1, a.status,
                                                   DEV_ATTN_SOFTMAX);
      if (!__all_sync(0xffffffffu, fin)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.0f / l_run : 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t ov[32];
        tmem_ld32_nowait(tmem + 2 * Cf::BK + lane_off + c * 32, ov);
        tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gr[4 * c + e]);
            uint4 o;
            uint32_t* op = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float2 gf = __bfloat1622float2(g2[u]);
              op[u] = pack_bf16x2(__uint_as_float(ov[8 * e + 2 * u]) * inv * gf.x,
                                  __uint_as_float(ov[8 * e + 2 * u + 1]) * inv * gf.y);
            }
            *reinterpret_cast<uint4*>(a.out + base + c * 32 + 8 * e) = o;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(o_free);
      g += it.ntiles;
    }
    if (!ok) *abort_flag = 1;
  }

  if (*abort_flag) {
    for (int k = 0; k < 64; ++k) __nanosleep(1000);   // let in-flight copies land
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cf::TMEM_COLS);
  }
}

}  // namespace dory
