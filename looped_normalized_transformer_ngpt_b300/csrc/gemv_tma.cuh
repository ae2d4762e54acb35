// gemv_tma.cuh - projections for few rows (M <= 16) with the weights
// streamed into shared memory by bulk copies.
//
// Same operation as gemv_kernel (gemv.cuh), including the SwiGLU pair and
// the fused nGPT step of the previous sublayer (PRE, "Dory1.0-4B: A Looped
// Normalized-GPT", Architecture):
//   Y[m, n] = scale[n] * sum_k X[m, k] W[n, k]               (fp32 out)
//   SwiGLU:  m_out[m, n] = u * SiLU(v),  u = X W_up[n]^T, v = X W_sl[n]^T
// With a handful of activation rows the projection streams its weights
// (2 M FLOP per 2-byte weight) and is bound by HBM bandwidth and latency.
// Each CTA (one per SM) owns a contiguous range of output features, so its
// weight rows are one contiguous byte range (two for SwiGLU: the W_up and
// W_sl rows); warp 8 copies that range into a shared-memory ring with
// cp.async.bulk in stages of whole rows, issuing the first stages before the
// wait on the previous kernel (weights never change during a forward pass),
// so a CTA's first ~200 KB are requested as soon as it starts.  Warps 0-7
// take the features of each stage round-robin, one feature per warp: every
// lane reads consecutive 16-byte chunks of the row (conflict-free), forms
// the dot product with the activation row (in shared memory) and the warp
// reduces it; the warp then releases its share of the stage.  Waits are
// bounded (status word).
//
// Used for one activation row and matrices of 8 MB or more (the 4B-class
// model's single-sequence decode: 10% faster per step than the register
// GEMV of gemv.cuh, measured at 262144 positions).  With more rows every
// weight chunk needs one activation chunk per row from shared memory, and
// with small matrices the launch is latency-bound either way; there the
// register GEMV measured as fast or faster (a variant with one warp per
// stage, reusing each activation chunk across the stage's rows, lengthened
// the tail of these short launches and was slower at every batch).
#pragma once
#include "gemv.cuh"

namespace dory {

constexpr int kGvtThreads = 288;                 // 8 consumer warps + 1 producer warp
constexpr int kGvtStageMax = 16384;              // bytes of weights per stage (at most)
constexpr int kGvtSmem = 224 * 1024;             // dynamic shared memory of a CTA
constexpr int kGvtXMax = 64 * 1024;              // activation rows kept in shared memory
constexpr int kGvtMaxK = kGvtStageMax / 2;       // a row (or SwiGLU pair of rows) fits a stage

// Ring geometry of one launch (host and device agree on it).
struct GvtGeom {
  int unit_bytes;     // bytes of one feature's weights (one row, two for SwiGLU)
  int per_stage;      // features per stage (<= 8: one per consumer warp)
  int stages;         // ring stages
  int x_in_smem;      // activation rows staged in shared memory
  int ring_off;       // shared-memory offset of the ring
};

__host__ __device__ inline GvtGeom gvt_geom(int M, int K, bool swiglu, bool pre) {
  GvtGeom g;
  g.unit_bytes = (swiglu ? 2 : 1) * K * 2;
  int r = kGvtStageMax / g.unit_bytes;
  g.per_stage = r < 1 ? 1 : (r > 8 ? 8 : r);
  const int xb = M * K * 2;
  g.x_in_smem = (pre || xb <= kGvtXMax) ? 1 : 0;
  g.ring_off = g.x_in_smem ? (xb + 1023) / 1024 * 1024 : 0;
  const int stage_bytes = g.per_stage * g.unit_bytes;
  int s = (kGvtSmem - g.ring_off - 1024) / stage_bytes;   // 1 KB: barriers
  g.stages = s > 16 ? 16 : s;
  return g;
}

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

template <int MM, bool SWIGLU, bool PRE>
__global__ void __launch_bounds__(kGvtThreads, 1) gemv_tma_kernel(const GemvArgs a, int* status) {
  extern __shared__ __align__(1024) uint8_t gvt_smem[];
  const GvtGeom geo = gvt_geom(a.M, a.K, SWIGLU, PRE);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int stage_bytes = geo.per_stage * geo.unit_bytes;
  uint8_t* ring = gvt_smem + geo.ring_off;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + geo.stages * stage_bytes);
  uint64_t* empty = full + geo.stages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + geo.stages);
  // this CTA's features [f0, f1)
  const int f0 = (int)((long long)blockIdx.x * a.N / gridDim.x);
  const int f1 = (int)((long long)(blockIdx.x + 1) * a.N / gridDim.x);
  const int nf = f1 - f0;
  const int n_stages = (nf + geo.per_stage - 1) / geo.per_stage;
  const long long row_bytes = (long long)a.K * 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < geo.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], geo.per_stage);   // one arrival per feature of the stage
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 8) {
    // ------------------------------------------------ producer: weight rows
    pdl_trigger();
    if (lane == 0) {
      const uint8_t* w = reinterpret_cast<const uint8_t*>(a.W);
      for (int s = 0; s < n_stages && !*abort_flag; ++s) {
        const int slot = s % geo.stages;
        if (s >= geo.stages &&
            !mbar_wait_bounded(&empty[slot], ((s / geo.stages) - 1) & 1, status, DEV_GEMV_PRODUCER)) {
          *abort_flag = 1;
          break;
        }
        const int u0 = f0 + s * geo.per_stage;
        const int nu = min(geo.per_stage, f1 - u0);
        uint8_t* dst = ring + slot * stage_bytes;
        const uint32_t bytes = (uint32_t)(nu * row_bytes);
        mbar_arrive_expect_tx(&full[slot], SWIGLU ? 2 * bytes : bytes);
        bulk_load(dst, w + u0 * row_bytes, bytes, &full[slot]);
        if (SWIGLU)
          bulk_load(dst + bytes, w + ((long long)u0 + a.pair_off) * row_bytes, bytes, &full[slot]);
      }
    }
    return;
  }

  // ------------------------------------------------ consumers (warps 0-7)
  pdl_wait();
  pdl_trigger();
  const __nv_bfloat16* X = a.X;
  long long ldx = a.ldx;
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(gvt_smem);
  if (PRE) {
    gemv_pre_rows(a, xs);                        // warps 0-7
    X = xs;
    ldx = a.K;
  } else if (geo.x_in_smem) {
    const int cpr = a.K / 8;
    for (int i = threadIdx.x; i < a.M * cpr; i += 256) {
      const int m = i / cpr, c = i % cpr;
      *reinterpret_cast<uint4*>(xs + (long long)m * a.K + c * 8) =
          *reinterpret_cast<const uint4*>(a.X + (long long)m * a.ldx + c * 8);
    }
    X = xs;
    ldx = a.K;
  }
  named_bar(1, 256);                             // activation rows ready

  const int nch = a.K / 8;                       // 16-byte chunks per row
  for (int j = warp; j < nf; j += 8) {
    const int s = j / geo.per_stage, r = j % geo.per_stage;
    const int slot = s % geo.stages;
    const bool ok = !*abort_flag && mbar_wait_bounded(&full[slot], (s / geo.stages) & 1, status,
                                                      DEV_GEMV_CONSUMER);
    if (!__all_sync(0xffffffffu, ok)) {
      *abort_flag = 1;
      break;
    }
    const int nu = min(geo.per_stage, nf - s * geo.per_stage);
    const uint8_t* stage = ring + slot * stage_bytes;
    const uint4* wu = reinterpret_cast<const uint4*>(stage + r * row_bytes);
    const uint4* wv = reinterpret_cast<const uint4*>(stage + (nu + r) * row_bytes);
    float acc[MM], acc2[MM];
#pragma unroll
    for (int m = 0; m < MM; ++m) acc[m] = acc2[m] = 0.f;
    for (int c = lane; c < nch; c += 32) {
      float fu[8], fv[8];
      bf16x8_to_f32(wu[c], fu);
      if (SWIGLU) bf16x8_to_f32(wv[c], fv);
#pragma unroll
      for (int m = 0; m < MM; ++m) {
        if (m < a.M) {
          float fx[8];
          const uint4 xv = geo.x_in_smem
                               ? *reinterpret_cast<const uint4*>(X + (long long)m * ldx + c * 8)
                               : __ldg(reinterpret_cast<const uint4*>(X + (long long)m * ldx + c * 8));
          bf16x8_to_f32(xv, fx);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            acc[m] = fmaf(fu[i], fx[i], acc[m]);
            if (SWIGLU) acc2[m] = fmaf(fv[i], fx[i], acc2[m]);
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
        const float u = warp_sum(acc[m]);
        if (SWIGLU) {
          const float v = warp_sum(acc2[m]);
          if (lane == 0)
            a.m_out[(long long)m * a.ldm + n] = __float2bfloat16_rn(u * (v / (1.0f + __expf(-v))));
        } else if (lane == 0) {
          a.Y[(long long)m * a.ldy + n] = u * (a.col_scale ? a.col_scale[n] : 1.f);
        }
      }
    }
  }
  if (*abort_flag) {
    for (int k = 0; k < 64; ++k) __nanosleep(1000);   // let in-flight copies land
  }
}

}  // namespace dory
