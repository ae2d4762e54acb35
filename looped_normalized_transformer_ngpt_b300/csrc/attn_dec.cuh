// attn_dec.cuh - decode attention with TMA-fed key / value streaming,
// head_dim 128 ("Dory1.0-4B: A Looped Normalized-GPT", Architecture;
// Last-Loop KV Caching).
//
// Same operation as attn_decode_kernel (attn.cuh): one new token per
// sequence at position P0, its G query heads per kv head.  The work is
// scheduled stream-K style: the 64-key tiles of all (sequence, kv head)
// groups form one sequence of T = groups x tiles-per-group tiles, and CTA c
// of n takes tiles [c T / n, (c + 1) T / n), so every CTA streams the same
// number of bytes whatever the group count (no partly empty last round).  A
// CTA's range may cross group boundaries; each (CTA, group) piece is one
// split and writes an unnormalised partial (o, max, sum) per head.  The CTA
// holding tile x is ((x + 1) n - 1) / T, which gives each piece its split
// index and each group its number of splits.  The last CTA of the group
// (atomic ticket) merges the partials with the new token's own key / value,
// applies sigmoid(g) and writes the gated output; split 0 stores the new
// k^ / v into ring slot P0 mod S.
//
// What differs is the key / value path, which carries nearly all of the
// bytes of a long-context decode step:
//   warp 4    TMA producer: 64-key K and V tiles (two 64-dim boxes each,
//             128-byte swizzle) into a ring of kStages stages, running ahead
//             across the CTA's work items so the ring never drains between
//             them;
//   warps 0-3 consumers: warp w takes keys 16w..16w+15 of every tile with
//             mma.sync m16n8k16 (rows = the G heads) and releases the stage
//             through its mbarrier; no CTA-wide barrier per tile.
// Tiles start at multiples of 64 positions and the cache ring size S is a
// multiple of 64, so a tile never wraps around the ring and one box covers
// it; keys outside the split's range (or below the window) are masked.  The
// split ranges are 64-aligned as well, so no tile is read twice.
#pragma once
#include "attn.cuh"

namespace dory {

constexpr int kDecTmaStages = 4;
constexpr int kDecTmaThreads = 160;

struct DecTmaCfg {
  static constexpr int DH = 128;
  static constexpr int HALF = 64 * 128;                // one 64-key x 64-dim box (bytes)
  static constexpr int TILE = 2 * HALF;                // K or V tile
  static constexpr int STAGE = 2 * TILE;               // K then V
  static constexpr int RING = kDecTmaStages * STAGE;
  static constexpr int Q_OFF = RING;                   // 16 x 128 bf16 (swz_off layout)
  static constexpr int O_OFF = Q_OFF + 16 * DH * 2;    // [4 warps][kDecMaxG][DH] fp32
  static constexpr int W_OFF = O_OFF + 4 * kDecMaxG * DH * 4;   // [kDecMaxG][kDecMaxSplits + 1]
  static constexpr int GATE_OFF = W_OFF + kDecMaxG * (kDecMaxSplits + 1) * 4;
  static constexpr int KC_OFF = GATE_OFF + kDecMaxG * DH * 4;   // current k^, v (fp32)
  static constexpr int ML_OFF = KC_OFF + 2 * DH * 4;            // sM[64], sL[64], sCur[8], flag
  static constexpr int BAR_OFF = ML_OFF + (64 + 64 + 8 + 8) * 4;
  static constexpr size_t SMEM = BAR_OFF + 2 * kDecTmaStages * 8 + 1024;   // + alignment slack
};

// byte offset of 16-byte chunk `chunk` (0..15) of key row `row` in a tile
// stored as two 64-dim boxes with the 128-byte swizzle
__device__ __forceinline__ uint32_t sw128_tile_off(int row, int chunk) {
  return (uint32_t)((chunk >> 3) * DecTmaCfg::HALF + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

template <bool RAW>
__global__ void __launch_bounds__(kDecTmaThreads, 1)
    attn_decode_tma_kernel(const __grid_constant__ CUtensorMap tm_kc,
                           const __grid_constant__ CUtensorMap tm_vc, const DecAttnArgs a) {
  using Cf = DecTmaCfg;
  constexpr int DH = Cf::DH, CH = DH / 8, HALF = DH / 2;
  extern __shared__ uint8_t dsm_raw[];
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
  const uint32_t ringa = smem_u32(dsm);
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(dsm + Cf::Q_OFF);
  float* sO = reinterpret_cast<float*>(dsm + Cf::O_OFF);
  float* sW = reinterpret_cast<float*>(dsm + Cf::W_OFF);
  float* sGate = reinterpret_cast<float*>(dsm + Cf::GATE_OFF);
  float* sKc = reinterpret_cast<float*>(dsm + Cf::KC_OFF);
  float* sVc = sKc + DH;
  float* sM = reinterpret_cast<float*>(dsm + Cf::ML_OFF);
  float* sL = sM + 64;
  float* sCur = sL + 64;
  int* sFlag = reinterpret_cast<int*>(sCur + 8);
  volatile int* abort_flag = sFlag + 1;
  uint64_t* full = reinterpret_cast<uint64_t*>(dsm + Cf::BAR_OFF);
  uint64_t* empty = full + kDecTmaStages;
  const uint32_t sQa = smem_u32(sQ);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.n_q / a.n_kv;
  const int n_groups = a.n_kv * a.B;
  const long long tpg = a.tpg;
  const long long T = (long long)n_groups * tpg;
  const long long ncta = gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < kDecTmaStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_kc);
    tma_prefetch_desc(&tm_vc);
  }
  __syncthreads();
  // ragged batches: the positions were written by an earlier kernel of the
  // step, so every warp waits for the previous kernel before using them
  if (a.p0s) pdl_wait();

  // This CTA's pieces in order.  With cached keys: its tile range cut at
  // group boundaries; without (tpg == 0): groups blockIdx.x, + gridDim.x, ...
  // as single pieces with no tiles.  `cur` is the piece's first global tile
  // (or its group); returns false past the last piece.  Every group spans
  // tpg tiles of the schedule; in a ragged batch a shorter sequence's group
  // has fewer real tiles, and its pieces past them carry none.  P0 / lo:
  // the group's sequence position and first visible cached key.
  const long long x_end = tpg > 0 ? ((long long)blockIdx.x + 1) * T / ncta : n_groups;
  auto piece = [&](long long cur, int& grp, int& split, int& nseg, int& k0, int& k1,
                   int& ntiles, long long& next, int& P0, int& lo) -> bool {
    if (cur >= x_end) return false;
    grp = (int)(tpg == 0 ? cur : cur / tpg);
    P0 = a.p0s ? a.p0s[grp / a.n_kv] : a.P0;
    lo = a.window > 0 ? max(0, P0 - a.window + 1) : 0;
    const int lo_a = lo / kDecTile * kDecTile;
    if (tpg == 0) {
      split = 0;
      nseg = 1;
      k0 = k1 = lo_a;
      ntiles = 0;
      next = cur + ncta;
      return true;
    }
    const long long g0 = (long long)grp * tpg;
    const long long e = min(x_end, g0 + tpg);
    const long long c_first = ((g0 + 1) * ncta - 1) / T;
    const long long c_last = ((g0 + tpg) * ncta - 1) / T;
    split = (int)(blockIdx.x - c_first);
    nseg = (int)(c_last - c_first + 1);
    const long long real = P0 > lo_a ? (P0 - lo_a + kDecTile - 1) / kDecTile : 0;   // <= tpg
    k0 = lo_a + (int)(cur - g0) * kDecTile;            // 64-aligned
    k1 = min(lo_a + (int)(e - g0) * kDecTile, P0);      // cached keys only
    ntiles = (int)max(0ll, min(e, g0 + real) - cur);
    next = e;
    return true;
  };
  const long long x_begin = tpg > 0 ? (long long)blockIdx.x * T / ncta : blockIdx.x;

  if (warp == 4) {
    // ------------------------------------------------ TMA producer
    // The cache was written by earlier launches (this launch writes only
    // slot P0 mod S, which no item reads), so loads start before the wait
    // on the previous kernel (the consumers wait for it before reading the
    // projections).
    if (lane == 0) {
      int g = 0;
      int grp, split, nseg, k0, k1, ntiles, p0g, log;
      long long nx;
      for (long long cur = x_begin;
           !*abort_flag && piece(cur, grp, split, nseg, k0, k1, ntiles, nx, p0g, log); cur = nx) {
        const int row0 = grp * a.S;                    // group = b * n_kv + kv head
        for (int t = 0; t < ntiles; ++t, ++g) {
          const int st = g % kDecTmaStages;
          if (g >= kDecTmaStages &&
              !mbar_wait_bounded(&empty[st], ((g / kDecTmaStages) - 1) & 1, a.status,
                                 DEV_DEC_PRODUCER)) {
            *abort_flag = 1;
            break;
          }
          const int row = row0 + (k0 + t * kDecTile) % a.S;
          uint8_t* dst = dsm + st * Cf::STAGE;
          mbar_arrive_expect_tx(&full[st], Cf::STAGE);
          tma_load_2d(dst, &tm_kc, &full[st], 0, row);
          tma_load_2d(dst + Cf::HALF, &tm_kc, &full[st], 64, row);
          tma_load_2d(dst + Cf::TILE, &tm_vc, &full[st], 0, row);
          tma_load_2d(dst + Cf::TILE + Cf::HALF, &tm_vc, &full[st], 64, row);
        }
      }
    }
    return;
  }

  // ------------------------------------------------ consumers (warps 0-3)
  // RoPE (cos, sin) of position P0 and s_qk for this lane's columns: weights
  // and a table written before the previous kernel, so read before its wait
  float2 rcs[HALF / 32];
  float rsq[HALF / 32][2];
#pragma unroll
  for (int e = 0; e < HALF / 32; ++e) {
    const int i = lane + 32 * e;
    rcs[e] = RAW && a.rope ? a.rope[i] : make_float2(1.f, 0.f);
    rsq[e][0] = RAW ? a.s_qk[i] : 1.f;
    rsq[e][1] = RAW ? a.s_qk[i + HALF] : 1.f;
  }
  auto csync = [] { named_bar(1, 128); };
  bool first = true;
  int g = 0;
  int grp, split, nseg, k0, k1, ntiles, P0, lo;
  long long nx;
  for (long long cur = x_begin; piece(cur, grp, split, nseg, k0, k1, ntiles, nx, P0, lo);
       cur = nx) {
    const int kvh = grp % a.n_kv, b = grp / a.n_kv;
    const int NS = nseg;                                 // splits of this group
    const int kv_lo = max(k0, lo);                       // visible keys [kv_lo, k1)
    if (RAW && a.rope && a.p0s) {
      // ragged batches: RoPE of this sequence's own position
#pragma unroll
      for (int e = 0; e < HALF / 32; ++e) rcs[e] = a.rope[b * HALF + lane + 32 * e];
    }
    if (first) {
      pdl_wait();
      pdl_trigger();
      first = false;
    } else {
      csync();                                           // shared state of the last item free
    }

    // ---- prologue: q^ (rows of sQ), current k^ and v, gate.  Every global
    // load of the item is issued before any is used (one memory round trip);
    // warp w forms heads hh = w and w + 4 (hh < G: query head kvh G + hh,
    // hh == G: key, hh == G + 1: value), lane l columns l, l + 32 of each half.
    for (int idx = tid; idx < 16 * CH; idx += 128) {     // zero rows >= G
      const int r = idx / CH, c = idx % CH;
      if (r >= G) *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(sQ) + swz_off<DH>(r, c)) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    constexpr int GPT = kDecMaxG * DH / 128;             // gate values per thread (max)
    float gv[GPT];
#pragma unroll
    for (int e = 0; e < GPT; ++e) {
      const int idx = tid + 128 * e;
      gv[e] = 0.f;
      if (idx < G * DH) {
        const int r = idx / DH, dd = idx % DH;
        if (RAW) {
          const float* yg = a.y + (long long)b * a.ldy + (long long)(a.n_q + 2 * a.n_kv) * DH +
                            (kvh * G + r) * DH + dd;
          for (int p = 0; p < a.n_parts; ++p) gv[e] += yg[p * a.part_stride];
        } else {
          gv[e] = __bfloat162float(a.gate[((long long)b * a.n_q + kvh * G + r) * DH + dd]);
        }
      }
    }
    if (RAW) {
      float x1[2][HALF / 32], x2[2][HALF / 32];
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        const int hh = warp + 4 * s2;
#pragma unroll
        for (int e = 0; e < HALF / 32; ++e) x1[s2][e] = x2[s2][e] = 0.f;
        if (hh < G + 2) {
          const int col0 = hh < G ? (kvh * G + hh) * DH
                                  : (hh == G ? (a.n_q + kvh) * DH : (a.n_q + a.n_kv + kvh) * DH);
          const float* yr = a.y + (long long)b * a.ldy + col0;
          for (int p = 0; p < a.n_parts; ++p) {
#pragma unroll
            for (int e = 0; e < HALF / 32; ++e) {
              const int i = lane + 32 * e;
              x1[s2][e] += yr[p * a.part_stride + i];
              x2[s2][e] += yr[p * a.part_stride + i + HALF];
            }
          }
        }
      }
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        const int hh = warp + 4 * s2;
        if (hh >= G + 2) continue;                         // uniform for the warp
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < HALF / 32; ++e) ss += x1[s2][e] * x1[s2][e] + x2[s2][e] * x2[s2][e];
        if (hh <= G) {
          const float inv = 1.0f / sqrtf(fmaxf(warp_sum(ss), 1e-12f));
#pragma unroll
          for (int e = 0; e < HALF / 32; ++e) {
            const float c1 = x1[s2][e] * rcs[e].x - x2[s2][e] * rcs[e].y;
            const float c2 = x2[s2][e] * rcs[e].x + x1[s2][e] * rcs[e].y;
            x1[s2][e] = c1 * inv * rsq[e][0];
            x2[s2][e] = c2 * inv * rsq[e][1];
          }
        }
#pragma unroll
        for (int e = 0; e < HALF / 32; ++e) {
          const int i = lane + 32 * e;
          const __nv_bfloat16 b1 = __float2bfloat16_rn(x1[s2][e]), b2 = __float2bfloat16_rn(x2[s2][e]);
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
      }
    } else {
      for (int hh = warp; hh < G + 2; hh += 4) {
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
#pragma unroll
    for (int e = 0; e < GPT; ++e) {
      const int idx = tid + 128 * e;
      if (idx < G * DH) sGate[idx] = RAW ? 1.0f / (1.0f + __expf(-gv[e])) : gv[e];
    }
    csync();

    // ---- cached keys: S = Q K^T, online softmax, O += P V (warp: 16 keys / tile)
    const int gq = lane >> 2, t4 = lane & 3;
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
    bool ok = true;

    for (int t = 0; t < ntiles; ++t, ++g) {
      const int st = g % kDecTmaStages;
      bool w_ok = !*abort_flag && mbar_wait_bounded(&full[st], (g / kDecTmaStages) & 1,
                                                    a.status, DEV_DEC_CONSUMER);
      if (!__all_sync(0xffffffffu, w_ok)) {
        ok = false;
        break;
      }
      const uint32_t kbase = ringa + (uint32_t)(st * Cf::STAGE);
      const uint32_t vbase = kbase + Cf::TILE;
      float s[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        const int key = 16 * warp + (lane & 7) + ((lane >> 4) & 1) * 8;
        const int c = 2 * kk + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + sw128_tile_off(key, c), b0, b1, b2, b3);
        mma_bf16_16816(s[0], qf[kk], b0, b1);
        mma_bf16_16816(s[1], qf[kk], b2, b3);
      }
      // Only mma rows g < 8 can hold a head (G <= 8); the stale running max
      // (raised only when it grows by more than 2^8) rarely rescales.
      const int j0 = k0 + t * kDecTile + 16 * warp;
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = j0 + 8 * nt + 2 * t4 + e;
          float v = s[nt][e] * a.scale_log2;
          v = (j >= kv_lo && j < k1) ? v : -INFINITY;
          s[nt][e] = v;
          mx = fmaxf(mx, v);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      if (mx > m_run + 8.0f) {
        const float corr = m_run == -INFINITY ? 0.f : ex2_ftz(m_run - mx);
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
          const float p = ex2_ftz(s[nt][e] - m_use);
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
        ldsm_x4_t(vbase + sw128_tile_off(key, c), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * dp], pa, b0, b1);
        mma_bf16_16816(o[2 * dp + 1], pa, b2, b3);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);            // this warp is done with the stage
    }
    // a bounded wait expired in some warp (its status word is set): all four
    // consumer warps agree before leaving, so none is left at a barrier
    if (!named_bar_and(1, 128, ok && !*abort_flag)) {
      *abort_flag = 1;
      break;
    }

    // ---- merge the 4 warps: row r = head, per warp (m, l, o[r][:])
    {
      float l = l_run;
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      if (t4 == 0 && gq < G) {
        sM[warp * 16 + gq] = m_run;
        sL[warp * 16 + gq] = l;
      }
      if (gq < G) {
#pragma unroll
        for (int nt = 0; nt < DH / 8; ++nt) {
          const int dim = 8 * nt + 2 * t4;
          *reinterpret_cast<float2*>(sO + (warp * kDecMaxG + gq) * DH + dim) =
              make_float2(o[nt][0], o[nt][1]);
        }
      }
    }
    csync();
    for (int idx = tid; idx < G * DH; idx += 128) {
      const int r = idx / DH, dd = idx % DH;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; ++w) M = fmaxf(M, sM[w * 16 + r]);
      float L = 0.f, acc = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float wt = sM[w * 16 + r] == -INFINITY ? 0.f : ex2_ftz(sM[w * 16 + r] - M);
        L += sL[w * 16 + r] * wt;
        acc += sO[(w * kDecMaxG + r) * DH + dd] * wt;
      }
      const long long base = ((long long)b * a.n_q + kvh * G + r) * a.n_splits + split;   // stride: max splits
      a.part_o[base * DH + dd] = acc;
      if (dd == 0) {
        a.part_ml[base * 2] = M;
        a.part_ml[base * 2 + 1] = L;
      }
    }

    // ---- ticket: the last CTA of (b, kvh) merges all splits + the new token
    __threadfence();
    csync();
    if (tid == 0) {
      const int prev = atomicAdd(&a.counter[b * a.n_kv + kvh], 1);
      *sFlag = prev == NS - 1;
    }
    csync();
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
    csync();
    // per head: global max and split weights, one lane per split (warp = head)
    for (int r = warp; r < G; r += 4) {
      const long long bh = (long long)b * a.n_q + kvh * G + r;
      float mx = sCur[r];
      for (int sp = lane; sp < NS; sp += 32) mx = fmaxf(mx, __ldcg(a.part_ml + (bh * a.n_splits + sp) * 2));
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
      float L = 0.f;
      for (int sp = lane; sp < NS; sp += 32) {
        const float ms = __ldcg(a.part_ml + (bh * a.n_splits + sp) * 2);
        const float wt = ms == -INFINITY ? 0.f : ex2_ftz(ms - mx);
        sW[r * (NS + 1) + sp] = wt;
        L += __ldcg(a.part_ml + (bh * a.n_splits + sp) * 2 + 1) * wt;
      }
      L = warp_sum(L);
      if (lane == 0) {
        const float wc = ex2_ftz(sCur[r] - mx);
        sW[r * (NS + 1) + NS] = wc;                              // new token's weight
        sM[r] = 1.0f / (L + wc);
      }
    }
    csync();
    for (int idx = tid; idx < G * DH; idx += 128) {
      const int r = idx / DH, dd = idx % DH;
      const long long bh = (long long)b * a.n_q + kvh * G + r;
      const float* wr = sW + r * (NS + 1);
      float acc = wr[NS] * sVc[dd];
      const float* po = a.part_o + bh * a.n_splits * DH + dd;
      // 16 partials in flight per round
      for (int sp0 = 0; sp0 < NS; sp0 += 16) {
        float ov[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) ov[u] = sp0 + u < NS ? __ldcg(po + (sp0 + u) * DH) : 0.f;
#pragma unroll
        for (int u = 0; u < 16; ++u)
          if (sp0 + u < NS) acc += wr[sp0 + u] * ov[u];
      }
      a.out[bh * DH + dd] = __float2bfloat16_rn(acc * sM[r] * sGate[idx]);
    }
    if (tid == 0) a.counter[b * a.n_kv + kvh] = 0;
  }
  if (first) {                                                // no item: still order the grid
    pdl_wait();
    pdl_trigger();
  }
  if (*abort_flag) {
    for (int k = 0; k < 64; ++k) __nanosleep(1000);   // let in-flight copies land
  }
}

}  // namespace dory
