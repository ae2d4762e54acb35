// dory.cu - host side of the C ABI declared in include/dory.h: handle and
// argument validation, KV/workspace carving, TMA descriptors, and the forward
// schedule of the looped nGPT ("Dory1.0-4B: A Looped Normalized-GPT",
// Training with Loops; Last-Loop KV Caching):
//
//   h = N(E_in[tok])
//   input layers (cache slice 0)
//   x = h;  s_0 = x
//   for i = 1..k:  h = N(s_{i-1} + x); recurrent layers; s_i = N(h)
//       cache: per-loop -> slice i-1 written every loop;
//              last-loop -> slice 0 written at loop k only
//   output layers on s_k;  logits = s_z * (E_out h)
//
// Each layer: QKV+gate GEMM (RoPE, q/k norm, sigmoid fused) -> attention ->
// KV write -> output GEMM -> nGPT step -> up+gate GEMM (SwiGLU fused) -> down
// GEMM -> nGPT step.  Everything is enqueued on the caller's stream; no call
// synchronises or allocates.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "dory.h"
#include "attn.cuh"
#include "attn_tc.cuh"
#include "attn_dec.cuh"
#include "gemm_tc.cuh"
#include "gemv.cuh"
#include "gemv_tma.cuh"
#include "quant.cuh"
#include "sample.cuh"
#include "rowops.cuh"

using namespace dory;

namespace {

constexpr int kGemmBN = 256;
constexpr int kSwapBN = 64;         // activation rows per tile of the swapped GEMM
constexpr int kSwapMaxM = 128;      // batched decode through the swapped GEMM up to this
constexpr int kSwapMaxParts = 16;   // K splits of the swapped GEMM

struct WsLayout {
  size_t status, h32, h32b, x32, hb, y32, q, k, v, g, att, m, rope_swa, rope_full, ropet_swa,
      ropet_full, gy, dec_o,
      dec_ml, dec_cnt, parts, seq_pos, seq_k, save32, total;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

WsLayout ws_layout(const dory_config& c, int max_batch, int max_chunk) {
  WsLayout L{};
  const size_t M = (size_t)max_batch * max_chunk;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align256(bytes);
    return o;
  };
  const size_t hq = (size_t)c.n_q * c.head_dim, hk = (size_t)c.n_kv * c.head_dim;
  L.status = take(256);
  L.h32 = take(M * c.d * 4);
  L.h32b = take((size_t)max_batch * c.d * 4);   // decode: second hidden-state buffer
  L.x32 = take(M * c.d * 4);
  L.hb = take(M * c.d * 2);
  L.y32 = take(M * c.d * 4);
  L.q = take(M * hq * 2);
  L.k = take(M * hk * 2);
  L.v = take(M * hk * 2);
  L.g = take(M * hq * 2);
  L.att = take(M * hq * 2);
  L.m = take(M * (size_t)c.ffn * 2);
  // RoPE rows: the call's positions, (ragged decode) each sequence's, or (a
  // mixed step) decode rows followed by a chunk
  const size_t rope_rows = (size_t)max_chunk + max_batch;
  L.rope_swa = take(rope_rows * (c.head_dim / 2) * 8);
  L.rope_full = take(rope_rows * (c.head_dim / 2) * 8);
  L.ropet_swa = take(rope_rows * (c.head_dim / 2) * 8);    // transposed copies
  L.ropet_full = take(rope_rows * (c.head_dim / 2) * 8);
  // few-row projections (decode): fp32 output of the QKV+gate / up+gate GEMV
  const size_t nq = (size_t)(2 * c.n_q + 2 * c.n_kv) * c.head_dim;
  const size_t wide = nq > 2 * (size_t)c.ffn ? nq : 2 * (size_t)c.ffn;
  L.gy = take((size_t)kGemvMaxM * wide * 4);
  // split-KV decode attention partials
  L.dec_o = take((size_t)max_batch * c.n_q * kDecMaxSplits * c.head_dim * 4);
  L.dec_ml = take((size_t)max_batch * c.n_q * kDecMaxSplits * 2 * 4);
  L.dec_cnt = take((size_t)max_batch * c.n_kv * 4);   // split tickets, zero between launches
  L.seq_pos = take((size_t)max_batch * 4);            // ragged decode: positions
  L.seq_k = take((size_t)max_batch * 4);              //   and loop counts
  L.save32 = take((size_t)max_batch * c.d * 4);       //   and finished rows' states
  // batched decode (up to kSwapMaxM rows): split-K partial sums
  {
    const size_t rows = max_batch < kSwapMaxM ? max_batch : kSwapMaxM;
    const size_t w2 = wide > (size_t)c.d ? wide : (size_t)c.d;
    L.parts = take((size_t)kSwapMaxParts * rows * w2 * 4);
  }
  L.total = off;
  return L;
}

bool layer_full(const dory_config& c, int l) { return l % c.full_every == c.full_offset; }
bool layer_rec(const dory_config& c, int l) { return l >= c.n_in && l < c.n_in + c.n_rec; }
int n_layers(const dory_config& c) { return c.n_in + c.n_rec + c.n_out; }
int slots_of(const dory_config& c, int l, int max_ctx) {
  return layer_full(c, l) ? max_ctx : (max_ctx < c.window ? max_ctx : c.window);
}
int mult_of(const dory_config& c, int l, int k, int mode) {
  return (mode == DORY_CACHE_PER_LOOP && layer_rec(c, l)) ? k : 1;
}

// Offset of (layer, slice, K|V) inside the KV region.
size_t kv_offset(const dory_config& c, int max_batch, int max_ctx, int k, int mode, int layer,
                 int slice, int which) {
  const size_t per_slot = (size_t)c.n_kv * c.head_dim * 2;
  size_t off = 0;
  for (int l = 0; l < layer; ++l)
    off += 2 * (size_t)mult_of(c, l, k, mode) * slots_of(c, l, max_ctx) * per_slot * max_batch;
  const size_t blk = (size_t)slots_of(c, layer, max_ctx) * per_slot * max_batch;
  return off + (size_t)slice * 2 * blk + (size_t)which * blk;
}

int validate_config(const dory_config* c) {
  if (!c) return DORY_EINVAL;
  if (c->d <= 0 || c->n_in < 0 || c->n_rec < 0 || c->n_out < 0 || c->n_q <= 0 || c->n_kv <= 0 ||
      c->head_dim <= 0 || c->ffn <= 0 || c->vocab <= 0 || c->window <= 0 || c->full_every <= 0 ||
      c->full_offset < 0 || n_layers(*c) <= 0)
    return DORY_EINVAL;
  if (c->n_q % c->n_kv) return DORY_EINVAL;
  if (c->head_dim != 32 && c->head_dim != 64 && c->head_dim != 128) return DORY_EUNSUPPORTED;
  if (c->d % 128 || c->d > 8 * kRowThreads * kRowMaxChunks) return DORY_EUNSUPPORTED;
  if (c->ffn % (kGemmBN / 2) || c->ffn > kGemvMaxK / 2 || c->d > kGemvMaxK / 2)
    return DORY_EUNSUPPORTED;
  if (64 % (c->n_q / c->n_kv) || c->n_q / c->n_kv > kDecMaxG) return DORY_EUNSUPPORTED;
  if (c->vocab % 16) return DORY_EUNSUPPORTED;
  if (kGemmBN % c->head_dim) return DORY_EUNSUPPORTED;
  if (c->rope && (!(c->rope_base_swa > 0) || !(c->rope_base_full > 0))) return DORY_EINVAL;
  return DORY_OK;
}

// ------------------------------------------------------------ TMA encoding
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// Row-major bf16 matrix [rows, cols] with row stride ld (elements), loaded
// as 64-column x box_rows boxes with the 128-byte swizzle.
// fp32 matrix [rows][cols] (row stride ld elements) written as {32, 128}
// boxes with the 128-byte swizzle (staged fp32 GEMM epilogue).
bool encode_f32_out(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                    uint64_t ld) {
  if (!get_encoder()) return false;
  if (((uintptr_t)base & 15) || (ld * 4) % 16) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 4};
  cuuint32_t box[2] = {32, 128};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                 uint32_t box_rows) {
  if (!get_encoder()) return false;
  if (((uintptr_t)base & 15) || (ld * 2) % 16) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// uint8 matrix [rows][cols] (row stride ld bytes), loaded as unswizzled
// boxes {box_cols, box_rows} (packed quantised weights).
bool encode_u8(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
               uint32_t box_cols, uint32_t box_rows,
               CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_NONE) {
  if (!get_encoder()) return false;
  if (((uintptr_t)base & 15) || ld % 16 || box_cols % 16) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 tensor [d2][d1][d0] (d0 contiguous, strides s1 / s2 elements), loaded
// as boxes {64, box1, box2} with the 128-byte swizzle.
bool encode_bf16_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                    uint64_t s1, uint64_t s2, uint32_t box1, uint32_t box2) {
  if (!get_encoder()) return false;
  if (((uintptr_t)base & 15) || (s1 * 2) % 16 || (s2 * 2) % 16) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1 * 2, s2 * 2};
  cuuint32_t box[3] = {64, box1, box2};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch with programmatic stream serialisation (see pdl_wait in ptx.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

int g_num_sms = 0;
bool g_debug_tc_attn = true;   // dory_debug_attention: tensor-core prefill kernel where it applies
int num_sms() {
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 148;
  }
  return g_num_sms;
}

template <int BN, int EPI>
int launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, GemmArgs args, cudaStream_t st,
                const EpiMaps* maps = nullptr) {
  static bool attr = false;
  using Cf = GemmCfg<BN, EPI>;
  if (!attr) {
    if (cudaFuncSetAttribute(gemm_tc_kernel<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Cf::SMEM) != cudaSuccess)
      return DORY_ECUDA;
    attr = true;
  }
  args.tiles_m = (args.M + Cf::BM - 1) / Cf::BM;
  const int cols = EPI == EPI_SWIGLU ? args.N / 2 : args.N;
  const int bn_out = EPI == EPI_SWIGLU ? BN / 2 : BN;
  args.tiles_n = (cols + bn_out - 1) / bn_out;
  if (!Cf::PARTS) args.k_splits = 1;
  if (args.k_splits < 1) return DORY_EINVAL;
  const int tiles = args.tiles_m * args.tiles_n * args.k_splits;
  if (tiles == 0) return DORY_OK;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  EpiMaps em;
  if (maps) {
    em = *maps;
  } else {
    std::memset(&em, 0, sizeof(em));
    // the head_dim-128 QKV+gate epilogue always writes through its maps
    if (EPI == EPI_QKVG && Cf::STAGED && args.head_dim == 128) return DORY_EINVAL;
  }
  // fp32 / SwiGLU: staged stores when the caller described the output
  args.staged = maps ? 1 : 0;
  return launch_k(gemm_tc_kernel<BN, EPI>, dim3(grid), dim3(Cf::THREADS), Cf::SMEM, st, ta, tb,
                  args, em) ==
                 cudaSuccess
             ? DORY_OK
             : DORY_ECUDA;
}

template <int DH>
int launch_attn(const AttnArgs& a, int B, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(attn_prefill_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)AttnCfg<DH>::SMEM) != cudaSuccess)
      return DORY_ECUDA;
    attr = true;
  }
  const int G = a.n_q / a.n_kv, BQ = AttnCfg<DH>::BR / G;
  const int qblocks = (a.C + BQ - 1) / BQ;
  const int base = qblocks * a.n_kv * B;
  // few CTAs over many key blocks (a short chunk after a long cache): split
  // the key blocks so that about two CTAs per SM stream them, within the
  // partial buffers (part_cap splits of every (row, head) when given)
  AttnArgs aa = a;
  aa.n_split = 1;
  if (a.part_o && a.part_ml && a.part_cap > 0 && base < num_sms()) {
    const int keys = a.window > 0 ? std::min(a.P0 + a.C, a.window + BQ) : a.P0 + a.C;
    const int nblk = keys / AttnCfg<DH>::BKEY;
    int ns = (2 * num_sms() + base - 1) / base;
    ns = std::min(ns, nblk / 2);
    ns = std::min(ns, a.part_cap);
    if (ns >= 2) aa.n_split = ns;
  }
  dim3 grid(qblocks, a.n_kv, B * aa.n_split);
  if (launch_k(attn_prefill_kernel<DH>, grid, dim3(128), AttnCfg<DH>::SMEM, st, aa) != cudaSuccess)
    return DORY_ECUDA;
  if (aa.n_split == 1) return DORY_OK;
  const long long rh = (long long)B * a.C * a.n_q;
  return launch_k(attn_split_combine_kernel<DH>, dim3((unsigned)rh), dim3(DH), 0, st, aa,
                  (int)(B * a.C)) == cudaSuccess
             ? DORY_OK
             : DORY_ECUDA;
}

// Prefill attention on tcgen05 (attn_tc.cuh) when its tile rules hold:
// head_dim 128, 128 / G query positions per CTA, key tiles of 64 aligned
// positions that never mix cached and current keys (P0 % 64 == 0) and never
// wrap the ring (window and ring size multiples of 64, or a ring that is not
// full).  Returns DORY_EUNSUPPORTED otherwise (the caller then runs the
// mma.sync kernel).  cache_rows = rows of the cache block ([batch][n_kv][S]).
int launch_attn_tc(const AttnArgs& aa, int B, int head_dim, long long cache_rows, int* status,
                   cudaStream_t st) {
  constexpr int BK = AttnTcCfg::BK;
  const int G = aa.n_q / aa.n_kv;
  if (head_dim != 128 || G < 1 || 128 % G || aa.C < 2 || aa.P0 % BK) return DORY_EUNSUPPORTED;
  if (aa.window > 0 && aa.window % BK) return DORY_EUNSUPPORTED;
  if (aa.P0 > 0 && aa.window > 0 && aa.S % BK && aa.S < aa.P0) return DORY_EUNSUPPORTED;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)AttnTcCfg::SMEM) != cudaSuccess)
      return DORY_ECUDA;
    attr = true;
  }
  const long long tok = (long long)B * aa.C;
  CUtensorMap tq, tk, tv, tkc, tvc;
  const __nv_bfloat16* kc = aa.k_cache ? aa.k_cache : aa.k_cur;
  const __nv_bfloat16* vc = aa.v_cache ? aa.v_cache : aa.v_cur;
  const uint64_t crow = aa.k_cache ? (uint64_t)cache_rows : (uint64_t)tok * aa.n_kv;
  if (!encode_bf16_3d(&tq, aa.q, 128, aa.n_q, tok, 128, (uint64_t)aa.n_q * 128, G, 128 / G) ||
      !encode_bf16_3d(&tk, aa.k_cur, 128, aa.n_kv, tok, 128, (uint64_t)aa.n_kv * 128, 1, BK) ||
      !encode_bf16_3d(&tv, aa.v_cur, 128, aa.n_kv, tok, 128, (uint64_t)aa.n_kv * 128, 1, BK) ||
      !encode_bf16(&tkc, kc, crow, 128, 128, BK) || !encode_bf16(&tvc, vc, crow, 128, 128, BK))
    return DORY_ECUDA;
  AttnTcArgs a{};
  a.C = aa.C;
  a.P0 = aa.P0;
  a.S = aa.S;
  a.n_kv = aa.n_kv;
  a.G = G;
  a.window = aa.window;
  a.scale_log2 = aa.scale_log2;
  a.gate = aa.gate;
  a.out = aa.out;
  a.n_q = aa.n_q;
  a.status = status;
  a.B = B;
  // persistent: no more CTAs than are resident (two per SM), striding over
  // the work items (query block, kv head, sequence), longest first
  const int QP = 128 / G;
  const long long items = (long long)((aa.C + QP - 1) / QP) * aa.n_kv * B;
  const int cap = 2 * num_sms();
  const int grid = items < cap ? (int)items : cap;
  return launch_k(attn_tc_kernel, dim3(grid), dim3(kAttnTcThreads), AttnTcCfg::SMEM, st, tq, tk,
                  tv, tkc, tvc,
                  a) == cudaSuccess
             ? DORY_OK
             : DORY_ECUDA;
}

// Few-row projection (M <= kGemvMaxM), see gemv.cuh.  The caller fills
// X/ldx (or, for the fused nGPT step, h_in/y_in/alpha/h_out with K = d), W, N,
// K, M and either Y/ldy/col_scale or (SwiGLU) pair_off/m_out/ldm.
template <int MM, int J, bool SW, bool PRE>
cudaError_t gemv_go(const GemvArgs& a, int grid, cudaStream_t st) {
  const size_t smem = (PRE || a.stage_x) ? (size_t)a.M * a.K * 2 : 0;
  static int per_sm = 0;
  if (per_sm == 0) {
    if (cudaFuncSetAttribute(gemv_kernel<MM, J, SW, PRE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kGemvStageMax) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_kernel<MM, J, SW, PRE>,
                                                      kGemvThreads, kGemvStageMax) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
  }
  // no more CTAs than are resident at once: a partial second wave would
  // double the time of these latency-bound kernels (CTAs stride instead)
  const int cap = per_sm * num_sms();
  return launch_k(gemv_kernel<MM, J, SW, PRE>, dim3(grid < cap ? grid : cap), dim3(kGemvThreads),
                  smem, st, a);
}

template <int MM, bool SW, bool PRE>
cudaError_t gemv_j(const GemvArgs& a, int J, int grid, cudaStream_t st) {
  if (J <= 2) return gemv_go<MM, 2, SW, PRE>(a, grid, st);
  if (J <= 4) return gemv_go<MM, 4, SW, PRE>(a, grid, st);
  if (SW) return cudaErrorInvalidValue;
  if (J <= 6) return gemv_go<MM, 6, false, PRE>(a, grid, st);
  return gemv_go<MM, 8, false, PRE>(a, grid, st);
}

// One-row projection of a large matrix with the weights streamed by bulk
// copies (gemv_tma.cuh): one CTA per SM, each owning a contiguous range of
// features.  Returns DORY_EUNSUPPORTED outside the case where it measured
// faster (one activation row, >= 8 MB of weights) or its limits (a
// feature's rows above one 16 KB stage, unaligned weights).
#ifndef DORY_GEMV_TMA
#define DORY_GEMV_TMA 1
#endif
template <int MM, bool SW, bool PRE>
int gemv_tma_go(const GemvArgs& a, int* status, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(gemv_tma_kernel<MM, SW, PRE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kGvtSmem) != cudaSuccess)
      return DORY_ECUDA;
    attr = true;
  }
  const int grid = a.N < num_sms() ? a.N : num_sms();
  return launch_k(gemv_tma_kernel<MM, SW, PRE>, dim3(grid), dim3(kGvtThreads), (size_t)kGvtSmem, st,
                  a, status) == cudaSuccess
             ? DORY_OK
             : DORY_ECUDA;
}

int launch_gemv_tma(const GemvArgs& a, int* status, cudaStream_t st) {
  const bool sw = a.m_out != nullptr;
  const bool pre = a.h_in != nullptr;
  const long long wbytes = (long long)(sw ? 2 : 1) * a.N * a.K * 2;
  if (!DORY_GEMV_TMA || a.M != 1 || wbytes < (8ll << 20) || a.N <= 0 || a.K % 8 ||
      (sw ? 2 : 1) * a.K * 2 > kGvtStageMax || (reinterpret_cast<uintptr_t>(a.W) & 15) ||
      (pre && a.K > kGemvPreMaxD) || (!pre && (reinterpret_cast<uintptr_t>(a.X) & 15 || a.ldx % 8)))
    return DORY_EUNSUPPORTED;
  if (gvt_geom(a.M, a.K, sw, pre).stages < 2) return DORY_EUNSUPPORTED;
  return sw ? (pre ? gemv_tma_go<1, true, true>(a, status, st) : gemv_tma_go<1, true, false>(a, status, st))
            : (pre ? gemv_tma_go<1, false, true>(a, status, st) : gemv_tma_go<1, false, false>(a, status, st));
}

// Projection of 1-4 rows with weight-only quantised weights (quant.cuh),
// register form: the geometry of launch_gemv with 16 (MXFP8) or 32 (NVFP4)
// weights per 16-byte chunk.  Used where the bulk-copy form does not apply
// (scale rows that are not a multiple of 16 bytes).
template <int FMT, int MM, int J, bool SW, bool PRE>
cudaError_t gemv_q_go(const GemvArgs& a, int grid, cudaStream_t st) {
  const size_t smem = (PRE || a.stage_x) ? (size_t)a.M * a.K * 2 : 0;
  static int per_sm = 0;
  if (per_sm == 0) {
    if (cudaFuncSetAttribute(gemv_q_kernel<FMT, MM, J, SW, PRE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kGemvStageMax) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_q_kernel<FMT, MM, J, SW, PRE>,
                                                      kGemvThreads, kGemvStageMax) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
  }
  const int cap = per_sm * num_sms();
  return launch_k(gemv_q_kernel<FMT, MM, J, SW, PRE>, dim3(grid < cap ? grid : cap),
                  dim3(kGemvThreads), smem, st, a);
}

template <int FMT, int MM, bool SW, bool PRE>
cudaError_t gemv_q_j(const GemvArgs& a, int J, int grid, cudaStream_t st) {
  if (J <= 2) return gemv_q_go<FMT, MM, 2, SW, PRE>(a, grid, st);
  if (J <= 4) return gemv_q_go<FMT, MM, 4, SW, PRE>(a, grid, st);
  if (SW) return cudaErrorInvalidValue;
  if (J <= 6) return gemv_q_go<FMT, MM, 6, false, PRE>(a, grid, st);
  return gemv_q_go<FMT, MM, 8, false, PRE>(a, grid, st);
}

template <int FMT>
cudaError_t gemv_q_fmt(const GemvArgs& a, int J, int grid, cudaStream_t st) {
  const bool sw = a.m_out != nullptr, pre = a.h_in != nullptr;
  return sw ? (pre ? gemv_q_j<FMT, 4, true, true>(a, J, grid, st)
                   : gemv_q_j<FMT, 4, true, false>(a, J, grid, st))
            : (pre ? gemv_q_j<FMT, 4, false, true>(a, J, grid, st)
                   : gemv_q_j<FMT, 4, false, false>(a, J, grid, st));
}

int launch_gemv_q(GemvArgs a, cudaStream_t st) {
  const bool sw = a.m_out != nullptr;
  const bool pre = a.h_in != nullptr;
  const int E = a.qfmt == QF_MXFP8 ? 16 : 32;
  const int jmax = sw ? 4 : 8;
  const int kc = (a.K + 32 * E - 1) / (32 * E);   // chunk columns per row
  int S = 1;
  while ((kc + S - 1) / S > jmax && S < kGemvWarps) S *= 2;
  const int J = (kc + S - 1) / S;
  if (J > jmax || a.M > 4 || a.M <= 0 || a.K % 32 || !a.Wq || !a.Ws ||
      (a.qfmt != QF_MXFP8 && a.qfmt != QF_NVFP4))
    return DORY_EUNSUPPORTED;
  if (pre && a.K > kGemvPreMaxD) return DORY_EUNSUPPORTED;
  a.S = S;
  const int fpi = kGemvWarps / S;
  a.n_iters = (a.N + fpi - 1) / fpi;
  a.stage_x = (!pre && (size_t)a.M * a.K * 2 <= (size_t)kGemvStageMax) ? 1 : 0;
  const cudaError_t e = a.qfmt == QF_MXFP8 ? gemv_q_fmt<QF_MXFP8>(a, J, a.n_iters, st)
                                           : gemv_q_fmt<QF_NVFP4>(a, J, a.n_iters, st);
  return e == cudaSuccess ? DORY_OK : DORY_ECUDA;
}

// Projection of 1-4 rows with quantised weights, bulk-copy form (quant.cuh
// gemv_tma_q_kernel): one CTA per SM, packed code and scale rows streamed by
// cp.async.bulk.  Needs 16-byte multiples for the rows of codes and scales.
template <int FMT, int MM, bool SW, bool PRE>
int gemv_tma_q_go(const GemvArgs& a, int* status, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(gemv_tma_q_kernel<FMT, MM, SW, PRE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kGvtSmem) != cudaSuccess)
      return DORY_ECUDA;
    attr = true;
  }
  const int grid = a.N < num_sms() ? a.N : num_sms();
  return launch_k(gemv_tma_q_kernel<FMT, MM, SW, PRE>, dim3(grid), dim3(kGvtThreads),
                  (size_t)kGvtSmem, st, a, status) == cudaSuccess
             ? DORY_OK
             : DORY_ECUDA;
}

template <int FMT, int MM>
int gemv_tma_q_mm(const GemvArgs& a, int* status, cudaStream_t st) {
  const bool sw = a.m_out != nullptr, pre = a.h_in != nullptr;
  return sw ? (pre ? gemv_tma_q_go<FMT, MM, true, true>(a, status, st)
                   : gemv_tma_q_go<FMT, MM, true, false>(a, status, st))
            : (pre ? gemv_tma_q_go<FMT, MM, false, true>(a, status, st)
                   : gemv_tma_q_go<FMT, MM, false, false>(a, status, st));
}

int launch_gemv_tma_q(const GemvArgs& a, int* status, cudaStream_t st) {
  const bool sw = a.m_out != nullptr;
  const bool pre = a.h_in != nullptr;
  if (a.M < 1 || a.M > 4 || a.N <= 0 || a.K % 32 || !a.Wq || !a.Ws ||
      (a.qfmt != QF_MXFP8 && a.qfmt != QF_NVFP4))
    return DORY_EUNSUPPORTED;
  const int sb = a.qfmt == QF_MXFP8 ? a.K / 32 : a.K / 16;
  if (sb % 16 || (reinterpret_cast<uintptr_t>(a.Wq) & 15) || (reinterpret_cast<uintptr_t>(a.Ws) & 15))
    return DORY_EUNSUPPORTED;
  if (pre && a.K > kGemvPreMaxD) return DORY_EUNSUPPORTED;
  if (!pre && ((reinterpret_cast<uintptr_t>(a.X) & 15) || a.ldx % 8)) return DORY_EUNSUPPORTED;
  if (gvq_geom(a.qfmt, a.M, a.K, sw, pre).stages < 2) return DORY_EUNSUPPORTED;
  if (a.qfmt == QF_MXFP8)
    return a.M == 1 ? gemv_tma_q_mm<QF_MXFP8, 1>(a, status, st)
                    : gemv_tma_q_mm<QF_MXFP8, 4>(a, status, st);
  return a.M == 1 ? gemv_tma_q_mm<QF_NVFP4, 1>(a, status, st)
                  : gemv_tma_q_mm<QF_NVFP4, 4>(a, status, st);
}

int launch_gemv(GemvArgs a, cudaStream_t st, int* status = nullptr) {
  if (a.qfmt) {
    if (a.M <= 4) {
      const int rq = launch_gemv_tma_q(a, status, st);
      if (rq != DORY_EUNSUPPORTED) return rq;
      return launch_gemv_q(a, st);
    }
    // 5-16 rows: decoding the codes for every row makes the projection
    // compute-bound; the bf16 matrix holds the dequantised weights
    a.qfmt = 0;
  }
  const int rt = launch_gemv_tma(a, status, st);
  if (rt != DORY_EUNSUPPORTED) return rt;
  const bool sw = a.m_out != nullptr;
  const bool pre = a.h_in != nullptr;
  const int jmax = sw ? 4 : 8;
  const int kc = (a.K + 255) / 256;                // 256-element chunks per row
  int S = 1;
  while ((kc + S - 1) / S > jmax && S < kGemvWarps) S *= 2;
  const int J = (kc + S - 1) / S;
  if (J > jmax || a.M > kGemvMaxM || a.M <= 0 || a.K % 8) return DORY_EUNSUPPORTED;
  if (pre && a.K > kGemvPreMaxD) return DORY_EUNSUPPORTED;
  a.S = S;
  const int fpi = kGemvWarps / S;
  a.n_iters = (a.N + fpi - 1) / fpi;
  a.stage_x = (!pre && (size_t)a.M * a.K * 2 <= (size_t)kGemvStageMax) ? 1 : 0;
  const int grid = a.n_iters;
  cudaError_t e;
  if (a.M <= 4)
    e = sw ? (pre ? gemv_j<4, true, true>(a, J, grid, st) : gemv_j<4, true, false>(a, J, grid, st))
           : (pre ? gemv_j<4, false, true>(a, J, grid, st) : gemv_j<4, false, false>(a, J, grid, st));
  else if (a.M <= 8)   // e.g. the speculative verifier's gamma + 1 rows
    e = sw ? (pre ? gemv_j<8, true, true>(a, J, grid, st) : gemv_j<8, true, false>(a, J, grid, st))
           : (pre ? gemv_j<8, false, true>(a, J, grid, st) : gemv_j<8, false, false>(a, J, grid, st));
  else
    e = sw ? (pre ? gemv_j<16, true, true>(a, J, grid, st) : gemv_j<16, true, false>(a, J, grid, st))
           : (pre ? gemv_j<16, false, true>(a, J, grid, st)
                  : gemv_j<16, false, false>(a, J, grid, st));
  return e == cudaSuccess ? DORY_OK : DORY_ECUDA;
}

// Output / down projection with the nGPT step fused (EPI_NGPT): clusters of
// N / 256 CTAs, each cluster striding over 128-row blocks; h (fp32) is read
// and rewritten through maps.out and its bf16 copy through maps.hb.  Returns
// DORY_EUNSUPPORTED when N is not a multiple of 256 of at most 8 tiles or no
// cluster of that size fits (the caller then runs the GEMM + row kernel).
int launch_gemm_ngpt(const CUtensorMap& ta, const CUtensorMap& tb, GemmArgs args,
                     const EpiMaps& maps, cudaStream_t st) {
  using Cf = GemmCfg<kGemmBN, EPI_NGPT>;
  if (args.N % kGemmBN || args.N / kGemmBN < 1 || args.N / kGemmBN > 8) return DORY_EUNSUPPORTED;
  const int cn = args.N / kGemmBN;
  static bool attr = false;
  static int max_clusters[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
  if (!attr) {
    if (cudaFuncSetAttribute(gemm_tc_kernel<kGemmBN, EPI_NGPT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cf::SMEM) != cudaSuccess)
      return DORY_ECUDA;
    attr = true;
  }
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = cn;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = Cf::SMEM;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (max_clusters[cn] == 0) {
    int n = 0;
    cfg.gridDim = dim3(cn * (num_sms() / cn));
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<kGemmBN, EPI_NGPT>, &cfg) != cudaSuccess)
      n = 0;
    cudaGetLastError();
    max_clusters[cn] = n > 0 ? n : -1;
  }
  if (max_clusters[cn] < 1) return DORY_EUNSUPPORTED;
  args.tiles_m = (args.M + Cf::BM - 1) / Cf::BM;
  args.tiles_n = cn;
  args.k_splits = 1;
  args.staged = 1;
  if (args.tiles_m == 0) return DORY_OK;
  const int n_clusters = args.tiles_m < max_clusters[cn] ? args.tiles_m : max_clusters[cn];
  cfg.gridDim = dim3(n_clusters * cn);
  // with programmatic serialisation where the runtime accepts it together
  // with the cluster shape, else plain stream order
  static int pdl_ok = -1;
  cfg.numAttrs = pdl_ok != 0 ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_tc_kernel<kGemmBN, EPI_NGPT>, ta, tb, args, maps);
  if (e != cudaSuccess && pdl_ok != 0) {
    cudaGetLastError();
    pdl_ok = 0;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gemm_tc_kernel<kGemmBN, EPI_NGPT>, ta, tb, args, maps);
  } else if (e == cudaSuccess && pdl_ok < 0) {
    pdl_ok = 1;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    max_clusters[cn] = -1;                          // not launchable here: unfused path
    return DORY_EUNSUPPORTED;
  }
  return DORY_OK;
}

// One-token attention of the forward pass (fused split merge, gate and KV
// write), see attn_decode_kernel.  Fills chunk / n_splits.
template <int DH, bool RAW>
int launch_dec_attn(DecAttnArgs a, int B, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(attn_decode_kernel<DH, RAW>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)DecCfg<DH>::SMEM) != cudaSuccess)
      return DORY_ECUDA;
    attr = true;
  }
  const int lo = a.window > 0 ? (a.P0 - a.window + 1 > 0 ? a.P0 - a.window + 1 : 0) : 0;
  const int n_cache = a.P0 - lo;                      // cached keys (the new token is extra)
  // Work items of equal size; the grid (no more CTAs than are resident: three
  // per SM) strides over them.  The split count gives every (sequence, kv
  // head) at least kDecMinTiles tiles per split and keeps the last round of
  // items nearly full.
  const int groups = B * a.n_kv;
  const int cap = 3 * num_sms();
  const int max_sp = (n_cache + kDecMinTiles * kDecTile - 1) / (kDecMinTiles * kDecTile);
  int best_sp = 1;
  double best = -1.0;
  for (int sp = 1; sp <= kDecMaxSplits && sp <= (max_sp > 0 ? max_sp : 1); ++sp) {
    const long long items = (long long)groups * sp;
    const long long rounds = (items + cap - 1) / cap;
    // time ~ rounds x keys per split; prefer fewer, fuller rounds
    const double per = (double)rounds * (double)((n_cache + sp - 1) / sp + 1);
    if (best < 0 || per < best * 0.98) {
      best = per;
      best_sp = sp;
    }
  }
  int chunk = n_cache > 0 ? (n_cache + best_sp - 1) / best_sp : kDecTile;
  chunk = (chunk + kDecTile - 1) / kDecTile * kDecTile;
  a.chunk = chunk;
  a.n_splits = n_cache > 0 ? (n_cache + chunk - 1) / chunk : 1;
  const long long items = (long long)groups * a.n_splits;
  const int grid = items < cap ? (int)items : cap;
  a.B = B;
  return launch_k(attn_decode_kernel<DH, RAW>, dim3(grid), dim3(128), DecCfg<DH>::SMEM, st, a) ==
                 cudaSuccess
             ? DORY_OK
             : DORY_ECUDA;
}

// TMA-fed decode attention (attn_dec.cuh): head_dim 128, cache given as a
// block of 64-aligned rings ([batch][n_kv][S], S % 64 == 0).  One CTA per SM
// strides over (split, kv head, sequence) items; the split ranges are
// 64-aligned.  Returns DORY_EUNSUPPORTED when the cache does not qualify.
// Fewest 64-key tiles per CTA of the TMA decode attention: with few groups
// and short windows (one sequence, 4096-key windows: 256 tiles) two tiles
// per CTA made each CTA's fixed work (prologue, partial store, ticket) and
// the 32-way merge dominate; four tiles (16 splits per group) measured 2-5%
// shorter one-sequence decode steps and left larger batches unchanged.
constexpr int kDecTmaMinTiles = 4;

template <bool RAW>
int launch_dec_attn_tma(DecAttnArgs a, int B, cudaStream_t st) {
  if (!a.k_cache || !a.v_cache || a.cache_rows <= 0 || a.S % kDecTile) return DORY_EUNSUPPORTED;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(attn_decode_tma_kernel<RAW>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)DecTmaCfg::SMEM) != cudaSuccess)
      return DORY_ECUDA;
    attr = true;
  }
  const int lo = a.window > 0 ? (a.P0 - a.window + 1 > 0 ? a.P0 - a.window + 1 : 0) : 0;
  const int lo_a = lo / kDecTile * kDecTile;
  const int n_cache = a.P0 - lo_a;                    // cached keys from the aligned start
  const long long groups = (long long)B * a.n_kv;
  // stream-K schedule (attn_dec.cuh): T tiles cut into `grid` equal ranges,
  // at least kDecMinTiles tiles each; a group spans at most
  // ceil(tpg / floor(T / grid)) + 1 ranges, which must stay within the
  // kDecMaxSplits partials per head that the workspace holds
  // ragged batches: the caller's count, the most tiles of any sequence
  const long long tpg =
      a.p0s ? a.tpg : (n_cache > 0 ? (n_cache + kDecTile - 1) / kDecTile : 0);
  const long long T = groups * tpg;
  long long grid = num_sms();
  int max_seg = 1;
  if (tpg == 0) {
    if (grid > groups) grid = groups;
  } else {
    const long long by_min = (T + kDecTmaMinTiles - 1) / kDecTmaMinTiles;
    if (grid > by_min) grid = by_min;
    // With few groups a grid that is a multiple of the group count cuts the
    // ranges at group boundaries (no CTA pays a second prologue and merge);
    // taken when the ranges are short (latency-bound launches) or it keeps
    // nearly every SM busy.
    const long long per_group = grid / groups;
    if (per_group >= 1 && (tpg / per_group < 32 || groups * per_group * 10 >= grid * 9))
      grid = groups * per_group;
    for (;; --grid) {
      const long long per = T / grid;
      const long long segs = (tpg + per - 1) / per + 1;
      if (segs <= kDecMaxSplits || grid == 1) {
        max_seg = (int)(segs < kDecMaxSplits ? segs : kDecMaxSplits);
        break;
      }
    }
  }
  a.tpg = (int)tpg;
  a.n_splits = max_seg;
  a.chunk = 0;
  CUtensorMap tkc, tvc;
  if (!encode_bf16(&tkc, a.k_cache, (uint64_t)a.cache_rows, 128, 128, kDecTile) ||
      !encode_bf16(&tvc, a.v_cache, (uint64_t)a.cache_rows, 128, 128, kDecTile))
    return DORY_EUNSUPPORTED;
  a.B = B;
  return launch_k(attn_decode_tma_kernel<RAW>, dim3((unsigned)grid), dim3(kDecTmaThreads),
                  DecTmaCfg::SMEM,
                  st, tkc, tvc, a) == cudaSuccess
             ? DORY_OK
             : DORY_ECUDA;
}

template <bool RAW>
int dec_attn(const DecAttnArgs& a, int B, int head_dim, cudaStream_t st) {
  if (head_dim == 128) {
    const int rc = launch_dec_attn_tma<RAW>(a, B, st);
    if (rc != DORY_EUNSUPPORTED) return rc;
  }
  if (head_dim == 32) return launch_dec_attn<32, RAW>(a, B, st);
  if (head_dim == 64) return launch_dec_attn<64, RAW>(a, B, st);
  if (head_dim == 128) return launch_dec_attn<128, RAW>(a, B, st);
  return DORY_EUNSUPPORTED;
}

// Split-KV decode attention: partial kernel + combine.
template <int DH>
int launch_decode_attn(DecodeArgs a, int B, const __nv_bfloat16* gate, __nv_bfloat16* out,
                       cudaStream_t st) {
  const int lo = a.window > 0 ? (a.P0 - a.window + 1 > 0 ? a.P0 - a.window + 1 : 0) : 0;
  const int n_keys = a.P0 - lo + 1;
  int target = 2 * num_sms() / (B * a.n_kv);
  if (target < 1) target = 1;
  int chunk = (n_keys + target - 1) / target;
  const int min_chunk = (n_keys + kDecMaxSplits - 1) / kDecMaxSplits;
  if (chunk < min_chunk) chunk = min_chunk;
  chunk = (chunk + kDecTile - 1) / kDecTile * kDecTile;
  a.chunk = chunk;
  a.n_splits = (n_keys + chunk - 1) / chunk;
  if (launch_k(attn_decode_split_kernel<DH>, dim3(a.n_splits, a.n_kv, B), dim3(128), 0, st, a) !=
      cudaSuccess)
    return DORY_ECUDA;
  return launch_k(attn_decode_combine_kernel, dim3(B * a.n_q), dim3(DH), 0, st,
                  (const float*)a.part_o, (const float*)a.part_ml, a.n_splits, a.n_q, DH, gate,
                  out) == cudaSuccess
             ? DORY_OK
             : DORY_ECUDA;
}

}  // namespace

struct dory_model {
  dory_config cfg;
  std::vector<dory_layer_weights> layers;
  int qfmt = 0;                          // DORY_QUANT_* of the few-row projections
  std::vector<dory_qlayer> qlayers;
  int q_swap = 0;                        // 2-128 rows: expand the codes in the swapped GEMM
  const void* embed_in = nullptr;
  const void* embed_out = nullptr;
  const float* s_z = nullptr;
  // bound memory
  bool bound = false;
  uint8_t* kv = nullptr;
  uint8_t* ws = nullptr;
  int max_batch = 0, max_ctx = 0, max_chunk = 0, k_max = 0, cache_mode = 0;
  WsLayout L{};
  std::vector<CUtensorMap> tm_qkvg, tm_o, tm_upgate, tm_down;
  CUtensorMap tm_embed_out{};
  // sequence state
  int len = 0;
  // ragged batches: per-sequence lengths (seq_len[b] = len for every b < batch
  // while `ragged` is false), the batch slot of a one-sequence call and
  // whether the current step decodes at per-sequence positions
  std::vector<int> seq_len;
  bool ragged = false;
  int slot = 0;
  bool ragged_step = false;
  bool multi_k = false;      // the ragged step also has per-sequence loop counts
  // a mixed step: mix_bd decode rows (slots 0 .. mix_bd-1) followed by a
  // chunk of one sequence in slot mix_slot at position mix_p
  bool mixed_step = false;
  int mix_bd = 0, mix_slot = 0, mix_p = 0;
  std::vector<int> step_k;   // those counts (host copy)
  int step_loop = 0;         // recurrent loop being run (per-sequence KV stores)
  int batch = 0;       // batch of the current sequences (0 = none yet)
  int last_rows = 0;   // rows of the last processed chunk (B * C)
  int hsel_last = 0;   // hidden-state buffer holding the last step's final rows
  bool use_tc_attn = true;  // prefill attention on tcgen05 where its tile rules hold
  bool use_ngpt_fused = true;   // nGPT step in the prefill O / down GEMM epilogues
  bool next_done = false;  // the last step also wrote the greedy tokens
  int launches = 0;
  // optional per-launch event timing
  bool prof_on = false;
  int prof_used = 0;
  std::vector<cudaEvent_t> prof_ev;   // 2 per launch
  std::vector<int> prof_cls;
};

// Points a layer projection at the layer's quantised weights, if any
// (which: 0 QKV+gate, 1 output, 2 up+gate, 3 down).
void use_quant(const dory_model* m, int l, int which, GemvArgs& g) {
  if (!m->qfmt) return;
  const dory_qlayer& q = m->qlayers[l];
  const dory_qmatrix& x = which == 0 ? q.qkvg : which == 1 ? q.o : which == 2 ? q.upgate : q.down;
  g.qfmt = m->qfmt;
  g.Wq = static_cast<const uint8_t*>(x.codes);
  g.Ws = static_cast<const uint8_t*>(x.scales);
  g.Wr = x.row_scale;
}


namespace {

template <typename T>
T* wsp(dory_model* m, size_t off) {
  return reinterpret_cast<T*>(m->ws + off);
}

#define DORY_TRY(...)                 \
  do {                                \
    const int _rc = (__VA_ARGS__);    \
    if (_rc != DORY_OK) return _rc;   \
  } while (0)

// Brackets every launch: optional start/end events (profiling) and the
// launch counter.
void pb(dory_model* m, int cls, cudaStream_t st) {
  if (m->prof_on && m->prof_used < (int)m->prof_cls.size()) {
    m->prof_cls[m->prof_used] = cls;
    cudaEventRecord(m->prof_ev[2 * m->prof_used], st);
  }
}
int pe(dory_model* m, cudaStream_t st, int rc = DORY_OK) {
  if (m->prof_on && m->prof_used < (int)m->prof_cls.size()) {
    cudaEventRecord(m->prof_ev[2 * m->prof_used + 1], st);
    ++m->prof_used;
  }
  m->launches += 1;
  if (rc != DORY_OK) return rc;
  return cudaGetLastError() == cudaSuccess ? DORY_OK : DORY_ECUDA;
}

// Hidden-state bookkeeping of one forward step.  The fp32 hidden state of the
// step's rows lives in one of two workspace buffers (h32 / h32b); `pend`,
// when set, is the residual rate of an nGPT step that is still owed: the true
// hidden state is N(h + pend * (N(y32) - h)).  The decode path leaves that
// step to the next kernel (a projection forms it in its prologue, a boundary
// kernel before its own transform); the prefill path applies it at once.
struct StepState {
  int hsel = 0;
  const float* pend = nullptr;
};

float* hbuf(dory_model* m, int sel) { return wsp<float>(m, sel ? m->L.h32b : m->L.h32); }

int ngpt_update(dory_model* m, int M, float* h, const float* alpha, cudaStream_t st,
                const float* y = nullptr, int n_parts = 1, long long part_stride = 0) {
  pb(m, DORY_K_NGPT_UPDATE, st);
  return pe(m, st,
            launch_k(ngpt_update_kernel, dim3(M), dim3(kRowThreads), 0, st, h,
                     wsp<__nv_bfloat16>(m, m->L.hb),
                     y ? y : (const float*)wsp<float>(m, m->L.y32), alpha, m->cfg.d, n_parts,
                     part_stride) == cudaSuccess
                ? DORY_OK
                : DORY_ECUDA);
}

// Applies an owed nGPT step in place (h and its bf16 copy hb).
int flush_pending(dory_model* m, StepState& s, int M, cudaStream_t st) {
  if (!s.pend) return DORY_OK;
  const float* al = s.pend;
  s.pend = nullptr;
  return ngpt_update(m, M, hbuf(m, s.hsel), al, st);
}

// Cache block of (layer, slice): K (which = 0) or V (which = 1).
// K or V block of (layer, slice), from the batch slot of a one-sequence
// call (m->slot; 0 otherwise): [max_batch - slot][n_kv][slots][head_dim].
__nv_bfloat16* kv_block(dory_model* m, int l, int slice, int which) {
  const dory_config& c = m->cfg;
  return reinterpret_cast<__nv_bfloat16*>(
             m->kv + kv_offset(c, m->max_batch, m->max_ctx, m->k_max, m->cache_mode, l, slice,
                               which)) +
         (size_t)m->slot * c.n_kv * slots_of(c, l, m->max_ctx) * c.head_dim;
}

// Rows ([batch][n_kv][slots]) of a block as kv_block returns it.
long long cache_rows(const dory_model* m, int slots) {
  return (long long)(m->max_batch - m->slot) * m->cfg.n_kv * slots;
}

// Ragged decode: 64-key tiles per (sequence, kv head) group of the TMA decode
// attention's schedule, the most over the step's sequences (window <= 0:
// full layer).
int ragged_tpg(const dory_model* m, int B, int window) {
  int t = 0;
  for (int b = 0; b < B; ++b) {
    const int p0 = m->seq_len[b];
    const int lo = window > 0 ? (p0 - window + 1 > 0 ? p0 - window + 1 : 0) : 0;
    const int lo_a = lo / kDecTile * kDecTile;
    const int n = p0 > lo_a ? (p0 - lo_a + kDecTile - 1) / kDecTile : 0;
    if (n > t) t = n;
  }
  return t;
}

float attn_scale_log2(const dory_config& c) {
  const float scale = c.softmax_scale > 0.f ? c.softmax_scale : sqrtf((float)c.head_dim);
  return scale * 1.4426950408889634f;
}

// One layer for one new token per sequence through the few-row GEMVs (a
// single sequence with quantised weights, see gemv_decode):
// five kernels.  QKV + gate GEMV (owed nGPT step fused) -> attention (RoPE /
// q-k norm in its prologue, split merge, gate and KV write fused) -> output
// GEMV -> up + gate GEMV with SwiGLU (attention nGPT step fused) -> down GEMV
// (its nGPT step is owed to the next kernel).
int run_layer_decode(dory_model* m, int l, int slice, bool store, int B, int P0, StepState& s,
                     cudaStream_t st) {
  const dory_config& c = m->cfg;
  const dory_layer_weights& w = m->layers[l];
  const int M = B;
  const int hq = c.n_q * c.head_dim;
  const int nqkvg = (2 * c.n_q + 2 * c.n_kv) * c.head_dim;
  const bool full = layer_full(c, l);
  const bool fuse = c.d <= kGemvPreMaxD;
  float* y32 = wsp<float>(m, m->L.y32);
  float* gy = wsp<float>(m, m->L.gy);
  __nv_bfloat16* att = wsp<__nv_bfloat16>(m, m->L.att);
  __nv_bfloat16* mo = wsp<__nv_bfloat16>(m, m->L.m);
  if (!fuse) DORY_TRY(flush_pending(m, s, M, st));

  auto with_pending = [&](GemvArgs& g) {
    if (s.pend) {
      g.h_in = hbuf(m, s.hsel);
      g.y_in = y32;
      g.alpha = s.pend;
      g.h_out = hbuf(m, s.hsel ^ 1);
      s.hsel ^= 1;
      s.pend = nullptr;
    } else {
      g.X = wsp<__nv_bfloat16>(m, m->L.hb);
      g.ldx = c.d;
    }
  };

  // QKV + gate projection -> fp32 rows [q | k | v | g]
  GemvArgs gq{};
  gq.M = M;
  gq.W = static_cast<const __nv_bfloat16*>(w.w_qkvg);
  gq.N = nqkvg;
  gq.K = c.d;
  gq.Y = gy;
  gq.ldy = nqkvg;
  with_pending(gq);
  use_quant(m, l, 0, gq);
  pb(m, DORY_K_QKVG_GEMM, st);
  DORY_TRY(pe(m, st, launch_gemv(gq, st, wsp<int>(m, m->L.status))));

  // attention over the cached keys + the new token, KV write fused
  DecAttnArgs da{};
  da.y = gy;
  da.ldy = nqkvg;
  da.n_parts = 1;
  da.part_stride = 0;
  da.s_qk = w.s_qk;
  da.rope = c.rope ? wsp<float2>(m, full ? m->L.rope_full : m->L.rope_swa) : nullptr;
  da.k_cache = kv_block(m, l, slice, 0);
  da.v_cache = kv_block(m, l, slice, 1);
  da.store = store ? 1 : 0;
  da.P0 = P0;
  da.S = slots_of(c, l, m->max_ctx);
  da.n_q = c.n_q;
  da.n_kv = c.n_kv;
  da.window = full ? 0 : c.window;
  da.scale_log2 = attn_scale_log2(c);
  da.part_o = wsp<float>(m, m->L.dec_o);
  da.part_ml = wsp<float>(m, m->L.dec_ml);
  da.counter = wsp<int>(m, m->L.dec_cnt);
  da.out = att;
  da.cache_rows = cache_rows(m, da.S);
  da.status = wsp<int>(m, m->L.status);
  if (m->ragged_step) {
    da.p0s = wsp<int>(m, m->L.seq_pos);
    da.tpg = ragged_tpg(m, B, da.window);
    if (m->multi_k && m->step_loop > 0) {     // a recurrent layer: per-sequence stores
      da.kstore = wsp<int>(m, m->L.seq_k);
      da.loop = m->step_loop;
    }
  }
  pb(m, DORY_K_ATTENTION, st);
  DORY_TRY(pe(m, st, dec_attn<true>(da, B, c.head_dim, st)));

  // output projection; its nGPT step is owed
  GemvArgs go{};
  go.M = M;
  go.X = att;
  go.ldx = hq;
  go.W = static_cast<const __nv_bfloat16*>(w.w_o);
  go.N = c.d;
  go.K = hq;
  go.Y = y32;
  go.ldy = c.d;
  use_quant(m, l, 1, go);
  pb(m, DORY_K_O_GEMM, st);
  DORY_TRY(pe(m, st, launch_gemv(go, st, wsp<int>(m, m->L.status))));
  s.pend = w.alpha_attn;
  if (!fuse) DORY_TRY(flush_pending(m, s, M, st));

  // up + gate projection with SwiGLU
  GemvArgs gu{};
  gu.M = M;
  gu.W = static_cast<const __nv_bfloat16*>(w.w_upgate);
  gu.N = c.ffn;
  gu.K = c.d;
  gu.pair_off = c.ffn;
  gu.m_out = mo;
  gu.ldm = c.ffn;
  with_pending(gu);
  use_quant(m, l, 2, gu);
  pb(m, DORY_K_UPGATE_GEMM, st);
  DORY_TRY(pe(m, st, launch_gemv(gu, st, wsp<int>(m, m->L.status))));

  // down projection; its nGPT step is owed
  GemvArgs gd{};
  gd.M = M;
  gd.X = mo;
  gd.ldx = c.ffn;
  gd.W = static_cast<const __nv_bfloat16*>(w.w_down);
  gd.N = c.d;
  gd.K = c.ffn;
  gd.Y = y32;
  gd.ldy = c.d;
  use_quant(m, l, 3, gd);
  pb(m, DORY_K_DOWN_GEMM, st);
  DORY_TRY(pe(m, st, launch_gemv(gd, st, wsp<int>(m, m->L.status))));
  s.pend = w.alpha_mlp;
  return DORY_OK;
}

// Swapped split-K projection for a decode batch: parts[s][row][n] (fp32) =
// X[row, K range s] . W[n, K range s]^T; returns the number of splits.
int swap_gemm(dory_model* m, const CUtensorMap& tw, const CUtensorMap& tx, int n_out, int rows,
              int K, float* parts, int& n_parts, cudaStream_t st,
              const dory_qmatrix* q = nullptr) {
  GemmArgs g{};
  g.w_pre = 1;   // weight operand: loads may start before the wait
  g.M = n_out;
  g.N = rows;
  g.K = K;
  g.status = wsp<int>(m, m->L.status);
  g.out = parts;
  g.ldo = n_out;
  g.part_stride = (long long)rows * n_out;
  const int units = ((n_out + 127) / 128) * ((rows + kSwapBN - 1) / kSwapBN);
  const int kb = (K + 63) / 64;
  // K splits: the persistent CTAs take units (tile, split) round-robin, so a
  // CTA's time is (its units) x (k blocks per unit + a fixed cost per unit
  // for the pipeline fill and the partial-sum store, about two k blocks).
  // Take the split count with the smallest such time; on ties the fewer
  // partial sums.
  const int cap = num_sms();
  int sp = 1;
  long long best = -1;
  for (int c = 1; c <= kSwapMaxParts && c <= (kb / 2 > 1 ? kb / 2 : 1); ++c) {
    const long long rounds = ((long long)units * c + cap - 1) / cap;
    const long long t = rounds * ((kb + c - 1) / c + 2);
    if (best < 0 || t < best) {
      best = t;
      sp = c;
    }
  }
  g.k_splits = sp;
  n_parts = sp;
  const bool fp4 = m->qfmt == DORY_QUANT_NVFP4;
  const int spr = fp4 ? K / 16 : K / 32;             // block-scale bytes per row
  if (q && m->qfmt && K % 64 == 0 && spr % 16 == 0) {
    // weight-only quantised weights: the packed codes and block scales
    // stream in and are expanded to bf16 in shared memory (the dequantised
    // matrix's values)
    const uint64_t rb = fp4 ? K / 2 : K;
    CUtensorMap tq;
    EpiMaps em;
    std::memset(&em, 0, sizeof(em));
    // code rows with the swizzle of their width (bank-conflict-free reads)
    if (!encode_u8(&tq, q->codes, n_out, rb, rb, fp4 ? 32 : 64, 128,
                   fp4 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B) ||
        !encode_u8(&em.q, q->scales, n_out, spr, spr, 16, 128))
      return DORY_ECUDA;
    g.qfmt = m->qfmt;
    g.qscales = static_cast<const uint8_t*>(q->scales);
    g.qrow = q->row_scale;
    return launch_gemm<kSwapBN, EPI_QPARTS>(tq, tx, g, st, &em);
  }
  return launch_gemm<kSwapBN, EPI_PARTS>(tw, tx, g, st);
}

// The layer's quantised matrix (which: 0 QKV+gate, 1 output, 2 up+gate, 3
// down), or null without quantised weights.
// One-token steps run through the few-row GEMVs only for a single sequence
// with quantised weights (the GEMV streams its packed codes); every other
// one-token step takes the swapped tensor-core GEMM, which on B300 reads the
// weights faster than the GEMV from one sequence up (measured: the 4B-class
// decode step at 1, 2, 4 and 16 sequences, 9 to 75% shorter).
bool gemv_decode(const dory_model* m, int M) { return m->qfmt != 0 && M == 1; }

const dory_qmatrix* qmat(const dory_model* m, int l, int which) {
  if (!m->qfmt || !m->q_swap) return nullptr;
  const dory_qlayer& q = m->qlayers[l];
  return which == 0 ? &q.qkvg : which == 1 ? &q.o : which == 2 ? &q.upgate : &q.down;
}

// One layer for one new token per sequence (B <= kSwapMaxM, unless
// gemv_decode): weights are the 128-row operand of
// the tensor-core GEMM, the batch the 64-row one, K split over the SMs; the
// attention, nGPT-step and SwiGLU kernels add the partial sums.
int run_layer_batched(dory_model* m, int l, int slice, bool store, int B, int P0,
                      const CUtensorMap& tx_hb, const CUtensorMap& tx_att,
                      const CUtensorMap& tx_m, StepState& s, cudaStream_t st) {
  const dory_config& c = m->cfg;
  const dory_layer_weights& w = m->layers[l];
  const int hq = c.n_q * c.head_dim;
  const int nqkvg = (2 * c.n_q + 2 * c.n_kv) * c.head_dim;
  const bool full = layer_full(c, l);
  DORY_TRY(flush_pending(m, s, B, st));
  float* h = hbuf(m, s.hsel);
  float* parts = wsp<float>(m, m->L.parts);
  __nv_bfloat16* att = wsp<__nv_bfloat16>(m, m->L.att);
  __nv_bfloat16* mo = wsp<__nv_bfloat16>(m, m->L.m);
  int np = 1;

  pb(m, DORY_K_QKVG_GEMM, st);
  DORY_TRY(pe(m, st, swap_gemm(m, m->tm_qkvg[l], tx_hb, nqkvg, B, c.d, parts, np, st, qmat(m, l, 0))));

  DecAttnArgs da{};
  da.y = parts;
  da.ldy = nqkvg;
  da.n_parts = np;
  da.part_stride = (long long)B * nqkvg;
  da.s_qk = w.s_qk;
  da.rope = c.rope ? wsp<float2>(m, full ? m->L.rope_full : m->L.rope_swa) : nullptr;
  da.k_cache = kv_block(m, l, slice, 0);
  da.v_cache = kv_block(m, l, slice, 1);
  da.store = store ? 1 : 0;
  da.P0 = P0;
  da.S = slots_of(c, l, m->max_ctx);
  da.n_q = c.n_q;
  da.n_kv = c.n_kv;
  da.window = full ? 0 : c.window;
  da.scale_log2 = attn_scale_log2(c);
  da.part_o = wsp<float>(m, m->L.dec_o);
  da.part_ml = wsp<float>(m, m->L.dec_ml);
  da.counter = wsp<int>(m, m->L.dec_cnt);
  da.out = att;
  da.cache_rows = cache_rows(m, da.S);
  da.status = wsp<int>(m, m->L.status);
  if (m->ragged_step) {
    da.p0s = wsp<int>(m, m->L.seq_pos);
    da.tpg = ragged_tpg(m, B, da.window);
    if (m->multi_k && m->step_loop > 0) {     // a recurrent layer: per-sequence stores
      da.kstore = wsp<int>(m, m->L.seq_k);
      da.loop = m->step_loop;
    }
  }
  pb(m, DORY_K_ATTENTION, st);
  DORY_TRY(pe(m, st, dec_attn<true>(da, B, c.head_dim, st)));

  pb(m, DORY_K_O_GEMM, st);
  DORY_TRY(pe(m, st, swap_gemm(m, m->tm_o[l], tx_att, c.d, B, hq, parts, np, st, qmat(m, l, 1))));
  DORY_TRY(ngpt_update(m, B, h, w.alpha_attn, st, parts, np, (long long)B * c.d));

  pb(m, DORY_K_UPGATE_GEMM, st);
  DORY_TRY(pe(m, st, swap_gemm(m, m->tm_upgate[l], tx_hb, 2 * c.ffn, B, c.d, parts, np, st,
                                qmat(m, l, 2))));
  pb(m, DORY_K_UPGATE_GEMM, st);
  DORY_TRY(pe(m, st,
              launch_k(swiglu_parts_kernel, dim3((c.ffn + 8 * kRowThreads - 1) / (8 * kRowThreads), B),
                       dim3(kRowThreads), 0, st, (const float*)parts, c.ffn, np,
                       (long long)B * 2 * c.ffn, mo) == cudaSuccess
                  ? DORY_OK
                  : DORY_ECUDA));

  pb(m, DORY_K_DOWN_GEMM, st);
  DORY_TRY(pe(m, st, swap_gemm(m, m->tm_down[l], tx_m, c.d, B, c.ffn, parts, np, st, qmat(m, l, 3))));
  return ngpt_update(m, B, h, w.alpha_mlp, st, parts, np, (long long)B * c.d);
}

// One layer for C tokens per sequence (prefill chunks; also decode with more
// rows than the GEMV handles): tensor-core GEMMs with fused epilogues, or the
// GEMV for few rows; prefill or one-token attention; nGPT steps applied
// at once.
int run_layer(dory_model* m, int l, int slice, bool store, int B, int C, int P0,
              const CUtensorMap& tm_hb, const CUtensorMap& tm_att, const CUtensorMap& tm_m,
              const EpiMaps& em, StepState& s, cudaStream_t st) {
  const dory_config& c = m->cfg;
  const dory_layer_weights& w = m->layers[l];
  const int M = B * C;
  const int hq = c.n_q * c.head_dim;
  int* status = wsp<int>(m, m->L.status);
  const bool full = layer_full(c, l);
  DORY_TRY(flush_pending(m, s, M, st));
  float* h = hbuf(m, s.hsel);

  // QKV + gate projection with RoPE / q-k normalisation / sigmoid fused
  GemmArgs ga{};
  ga.w_pre = 1;   // weight operand: loads may start before the wait
  ga.M = M;
  ga.N = (2 * c.n_q + 2 * c.n_kv) * c.head_dim;
  ga.K = c.d;
  ga.status = status;
  ga.q = wsp<__nv_bfloat16>(m, m->L.q);
  ga.k = wsp<__nv_bfloat16>(m, m->L.k);
  ga.v = wsp<__nv_bfloat16>(m, m->L.v);
  ga.g = wsp<__nv_bfloat16>(m, m->L.g);
  ga.n_q = c.n_q;
  ga.n_kv = c.n_kv;
  ga.head_dim = c.head_dim;
  ga.s_qk = w.s_qk;
  ga.rope = c.rope ? wsp<float2>(m, full ? m->L.rope_full : m->L.rope_swa) : nullptr;
  ga.rope_t = c.rope && c.head_dim == 128
                  ? wsp<float4>(m, full ? m->L.ropet_full : m->L.ropet_swa)
                  : nullptr;
  ga.rows_per_seq = C;
  const bool few = M <= kGemvMaxM;
  __nv_bfloat16* hb = wsp<__nv_bfloat16>(m, m->L.hb);
  float* gy = wsp<float>(m, m->L.gy);
  if (few) {
    GemvArgs g{};
    g.M = M;
    g.X = hb;
    g.ldx = c.d;
    g.W = static_cast<const __nv_bfloat16*>(w.w_qkvg);
    g.N = ga.N;
    g.K = c.d;
    g.Y = gy;
    g.ldy = ga.N;
    use_quant(m, l, 0, g);
    pb(m, DORY_K_QKVG_GEMM, st);
    DORY_TRY(pe(m, st, launch_gemv(g, st, wsp<int>(m, m->L.status))));
    pb(m, DORY_K_QKVG_GEMM, st);
    const int nheads = 2 * c.n_q + 2 * c.n_kv;
    const int thr = c.head_dim / 2 > 32 ? c.head_dim / 2 : 32;
    DORY_TRY(pe(m, st,
                launch_k(qkvg_post_kernel, dim3(M, nheads), dim3(thr), 0, st, (const float*)gy, M,
                         c.n_q, c.n_kv, c.head_dim, w.s_qk, (const float2*)ga.rope, C, ga.q, ga.k,
                         ga.v, ga.g) == cudaSuccess
                    ? DORY_OK
                    : DORY_ECUDA));
  } else {
    pb(m, DORY_K_QKVG_GEMM, st);
    DORY_TRY(pe(m, st, launch_gemm<kGemmBN, EPI_QKVG>(tm_hb, m->tm_qkvg[l], ga, st, &em)));
  }

  // attention over cached + current keys
  const int S = slots_of(c, l, m->max_ctx);
  __nv_bfloat16* kc = kv_block(m, l, slice, 0);
  __nv_bfloat16* vc = kv_block(m, l, slice, 1);
  __nv_bfloat16* att = wsp<__nv_bfloat16>(m, m->L.att);
  if (m->mixed_step) {
    // a mixed step: the first mix_bd rows decode one token each in slots
    // 0 .. mix_bd-1 at their own positions (split-key kernel, KV write
    // fused); the remaining rows are one chunk of the sequence in slot
    // mix_slot (multi-token kernel on that slot's blocks, then its KV write)
    const int Bd = m->mix_bd, Cc = M - Bd;
    const size_t hk = (size_t)c.n_kv * c.head_dim;
    if (Bd > 0) {
      DecAttnArgs da{};
      da.q = ga.q;
      da.k_cur = ga.k;
      da.v_cur = ga.v;
      da.gate = ga.g;
      da.k_cache = kc;
      da.v_cache = vc;
      da.store = store ? 1 : 0;
      int pmax = 0;
      for (int b = 0; b < Bd; ++b) pmax = m->seq_len[b] > pmax ? m->seq_len[b] : pmax;
      da.P0 = pmax;
      da.p0s = wsp<int>(m, m->L.seq_pos);
      da.tpg = ragged_tpg(m, Bd, full ? 0 : c.window);
      da.S = S;
      da.n_q = c.n_q;
      da.n_kv = c.n_kv;
      da.window = full ? 0 : c.window;
      da.scale_log2 = attn_scale_log2(c);
      da.part_o = wsp<float>(m, m->L.dec_o);
      da.part_ml = wsp<float>(m, m->L.dec_ml);
      da.counter = wsp<int>(m, m->L.dec_cnt);
      da.out = att;
      da.cache_rows = cache_rows(m, S);
      da.status = status;
      pb(m, DORY_K_ATTENTION, st);
      DORY_TRY(pe(m, st, dec_attn<false>(da, Bd, c.head_dim, st)));
    }
    const size_t so = (size_t)m->mix_slot * c.n_kv * S * c.head_dim;
    AttnArgs aa{};
    aa.q = ga.q + (size_t)Bd * hq;
    aa.k_cur = ga.k + Bd * hk;
    aa.v_cur = ga.v + Bd * hk;
    aa.k_cache = kc + so;
    aa.v_cache = vc + so;
    aa.gate = ga.g + (size_t)Bd * hq;
    aa.out = att + (size_t)Bd * hq;
    aa.C = Cc;
    aa.P0 = m->mix_p;
    aa.S = S;
    aa.n_q = c.n_q;
    aa.n_kv = c.n_kv;
    aa.window = full ? 0 : c.window;
    aa.scale_log2 = attn_scale_log2(c);
    aa.part_o = wsp<float>(m, m->L.dec_o);
    aa.part_ml = wsp<float>(m, m->L.dec_ml);
    aa.part_cap = (int)((long long)kDecMaxSplits * m->max_batch / Cc);
    const long long rows_c = (long long)(m->max_batch - m->mix_slot) * c.n_kv * S;
    pb(m, DORY_K_ATTENTION, st);
    int arc = m->use_tc_attn ? launch_attn_tc(aa, 1, c.head_dim, rows_c, status, st)
                             : DORY_EUNSUPPORTED;
    if (arc == DORY_EUNSUPPORTED) {
      if (c.head_dim == 32) arc = launch_attn<32>(aa, 1, st);
      if (c.head_dim == 64) arc = launch_attn<64>(aa, 1, st);
      if (c.head_dim == 128) arc = launch_attn<128>(aa, 1, st);
    }
    DORY_TRY(pe(m, st, arc));
    if (store) {
      const int t_first = Cc > S ? Cc - S : 0;
      pb(m, DORY_K_KV_WRITE, st);
      DORY_TRY(pe(m, st,
                  launch_k(kv_write_kernel, dim3(Cc - t_first, 1), dim3(128), 0, st, aa.k_cur,
                           aa.v_cur, kc + so, vc + so, Cc, m->mix_p, S, t_first, c.n_kv,
                           c.head_dim) == cudaSuccess
                      ? DORY_OK
                      : DORY_ECUDA));
    }
  } else if (C == 1) {
    pb(m, DORY_K_ATTENTION, st);
    // one token per sequence: split-key kernel, KV write fused
    DecAttnArgs da{};
    da.q = ga.q;
    da.k_cur = ga.k;
    da.v_cur = ga.v;
    da.gate = ga.g;
    da.k_cache = kc;
    da.v_cache = vc;
    da.store = store ? 1 : 0;
    da.P0 = P0;
    da.S = S;
    da.n_q = c.n_q;
    da.n_kv = c.n_kv;
    da.window = full ? 0 : c.window;
    da.scale_log2 = attn_scale_log2(c);
    da.part_o = wsp<float>(m, m->L.dec_o);
    da.part_ml = wsp<float>(m, m->L.dec_ml);
    da.counter = wsp<int>(m, m->L.dec_cnt);
    da.out = att;
    da.cache_rows = cache_rows(m, S);
    da.status = status;
    DORY_TRY(pe(m, st, dec_attn<false>(da, B, c.head_dim, st)));
  } else {
    pb(m, DORY_K_ATTENTION, st);
    AttnArgs aa{};
    aa.q = ga.q;
    aa.k_cur = ga.k;
    aa.v_cur = ga.v;
    aa.k_cache = kc;
    aa.v_cache = vc;
    aa.gate = ga.g;
    aa.out = att;
    aa.C = C;
    aa.P0 = P0;
    aa.S = S;
    aa.n_q = c.n_q;
    aa.n_kv = c.n_kv;
    aa.window = full ? 0 : c.window;
    aa.scale_log2 = attn_scale_log2(c);
    // key-range split partials live in the decode attention's buffers
    aa.part_o = wsp<float>(m, m->L.dec_o);
    aa.part_ml = wsp<float>(m, m->L.dec_ml);
    aa.part_cap = (int)((long long)kDecMaxSplits * m->max_batch / ((long long)B * C));
    int arc = m->use_tc_attn ? launch_attn_tc(aa, B, c.head_dim,
                                              cache_rows(m, S), status, st)
                             : DORY_EUNSUPPORTED;
    if (arc == DORY_EUNSUPPORTED) {
      if (c.head_dim == 32) arc = launch_attn<32>(aa, B, st);
      if (c.head_dim == 64) arc = launch_attn<64>(aa, B, st);
      if (c.head_dim == 128) arc = launch_attn<128>(aa, B, st);
    }
    DORY_TRY(pe(m, st, arc));
    // KV write: the last min(C, S) positions of the call
    if (store) {
      const int t_first = C > S ? C - S : 0;
      dim3 grid(C - t_first, B);
      pb(m, DORY_K_KV_WRITE, st);
      DORY_TRY(pe(m, st,
                  launch_k(kv_write_kernel, grid, dim3(64), 0, st, (const __nv_bfloat16*)ga.k,
                           (const __nv_bfloat16*)ga.v, kc, vc, C, P0, S, t_first, c.n_kv,
                           c.head_dim) == cudaSuccess
                      ? DORY_OK
                      : DORY_ECUDA));
    }
  }

  // output projection + nGPT step
  GemmArgs go{};
  go.w_pre = 1;   // weight operand: loads may start before the wait
  go.M = M;
  go.N = c.d;
  go.K = hq;
  go.status = status;
  go.out = wsp<float>(m, m->L.y32);
  go.ldo = c.d;
  pb(m, DORY_K_O_GEMM, st);
  bool fused_o = false, fused_d = false;
  if (few) {
    GemvArgs g{};
    g.M = M;
    g.X = att;
    g.ldx = hq;
    g.W = static_cast<const __nv_bfloat16*>(w.w_o);
    g.N = c.d;
    g.K = hq;
    g.Y = go.out;
    g.ldy = c.d;
    use_quant(m, l, 1, g);
    DORY_TRY(pe(m, st, launch_gemv(g, st, wsp<int>(m, m->L.status))));
  } else if (m->use_ngpt_fused) {
    // nGPT step fused into the GEMM epilogue (cluster over the d columns)
    EpiMaps eh = em;
    eh.hb = tm_hb;
    if (!encode_f32_out(&eh.out, h, M, c.d, c.d)) return DORY_ECUDA;
    go.h32 = h;
    go.alpha = w.alpha_attn;
    const int rc = launch_gemm_ngpt(tm_att, m->tm_o[l], go, eh, st);
    if (rc != DORY_EUNSUPPORTED) {
      DORY_TRY(pe(m, st, rc));
      fused_o = true;
    }
  }
  if (!few && !fused_o)
    DORY_TRY(pe(m, st, launch_gemm<kGemmBN, EPI_F32>(tm_att, m->tm_o[l], go, st, &em)));
  if (!fused_o) DORY_TRY(ngpt_update(m, M, h, w.alpha_attn, st));

  // SwiGLU MLP + nGPT step
  GemmArgs gu{};
  gu.w_pre = 1;   // weight operand: loads may start before the wait
  gu.M = M;
  gu.N = 2 * c.ffn;
  gu.K = c.d;
  gu.b_second = c.ffn;
  gu.status = status;
  gu.m_out = wsp<__nv_bfloat16>(m, m->L.m);
  gu.ldm = c.ffn;
  pb(m, DORY_K_UPGATE_GEMM, st);
  if (few) {
    GemvArgs g{};
    g.M = M;
    g.X = hb;
    g.ldx = c.d;
    g.W = static_cast<const __nv_bfloat16*>(w.w_upgate);
    g.N = c.ffn;
    g.K = c.d;
    g.pair_off = c.ffn;
    g.m_out = gu.m_out;
    g.ldm = c.ffn;
    use_quant(m, l, 2, g);
    DORY_TRY(pe(m, st, launch_gemv(g, st, wsp<int>(m, m->L.status))));
  } else {
    EpiMaps emm = em;                              // m is written through its load map
    emm.out = tm_m;
    DORY_TRY(pe(m, st, launch_gemm<kGemmBN, EPI_SWIGLU>(tm_hb, m->tm_upgate[l], gu, st, &emm)));
  }
  GemmArgs gd{};
  gd.w_pre = 1;   // weight operand: loads may start before the wait
  gd.M = M;
  gd.N = c.d;
  gd.K = c.ffn;
  gd.status = status;
  gd.out = wsp<float>(m, m->L.y32);
  gd.ldo = c.d;
  pb(m, DORY_K_DOWN_GEMM, st);
  if (few) {
    GemvArgs g{};
    g.M = M;
    g.X = gu.m_out;
    g.ldx = c.ffn;
    g.W = static_cast<const __nv_bfloat16*>(w.w_down);
    g.N = c.d;
    g.K = c.ffn;
    g.Y = gd.out;
    g.ldy = c.d;
    use_quant(m, l, 3, g);
    DORY_TRY(pe(m, st, launch_gemv(g, st, wsp<int>(m, m->L.status))));
  } else if (m->use_ngpt_fused) {
    EpiMaps eh = em;
    eh.hb = tm_hb;
    if (!encode_f32_out(&eh.out, h, M, c.d, c.d)) return DORY_ECUDA;
    gd.h32 = h;
    gd.alpha = w.alpha_mlp;
    const int rc = launch_gemm_ngpt(tm_m, m->tm_down[l], gd, eh, st);
    if (rc != DORY_EUNSUPPORTED) {
      DORY_TRY(pe(m, st, rc));
      fused_d = true;
    }
  }
  if (!few && !fused_d)
    DORY_TRY(pe(m, st, launch_gemm<kGemmBN, EPI_F32>(tm_m, m->tm_down[l], gd, st, &em)));
  return fused_d ? DORY_OK : ngpt_update(m, M, h, w.alpha_mlp, st);
}

// Loop-boundary kernel on the current hidden buffer; an owed nGPT step is
// applied first inside the same kernel.
// With per-sequence loop counts, `loop` is the loop just finished: rows
// whose count it is keep their final state (see boundary_kernel).
int boundary(dory_model* m, int M, int mode, StepState& s, cudaStream_t st, int loop = 0) {
  const float* y = s.pend ? wsp<float>(m, m->L.y32) : nullptr;
  const float* al = s.pend;
  s.pend = nullptr;
  const bool mk = m->multi_k && (mode == BND_ENTER_NEXT || mode == BND_EXIT);
  pb(m, DORY_K_BOUNDARY, st);
  return pe(m, st,
            launch_k(boundary_kernel, dim3(M), dim3(kRowThreads), 0, st, hbuf(m, s.hsel),
                     wsp<__nv_bfloat16>(m, m->L.hb), wsp<float>(m, m->L.x32), m->cfg.d, mode, y, 1,
                     (long long)0, al, mk ? (const int*)wsp<int>(m, m->L.seq_k) : nullptr, loop,
                     wsp<float>(m, m->L.save32)) == cudaSuccess
                ? DORY_OK
                : DORY_ECUDA);
}

// One forward step over B sequences x C tokens at positions P0..P0+C-1.
// Logit rows: if logits != null, rows (b, t) for t >= C - n_logit_rows are
// written to logits + (b * ld_seq + t_out0 + t - (C - n_logit_rows)) * V.
int run_step(dory_model* m, const int32_t* tokens, int ld_tok, int B, int C, int k,
             float* logits, long long ld_seq, int t_out0, int n_logit_rows, cudaStream_t st,
             int32_t* next_tok = nullptr) {
  m->next_done = false;
  const dory_config& c = m->cfg;
  const int M = B * C;
  const int P0 = m->len;
  int* status = wsp<int>(m, m->L.status);
  const bool decode = !m->mixed_step && C == 1 && gemv_decode(m, M);
  const bool batched = !m->mixed_step && C == 1 && !decode && M <= kSwapMaxM;

  CUtensorMap tm_hb, tm_att, tm_m;
  const int hq = c.n_q * c.head_dim;
  const uint32_t box = batched ? kSwapBN / 2 : 128;   // activation rows per TMA box
  if (!encode_bf16(&tm_hb, m->ws + m->L.hb, M, c.d, c.d, box) ||
      !encode_bf16(&tm_att, m->ws + m->L.att, M, hq, hq, box) ||
      !encode_bf16(&tm_m, m->ws + m->L.m, M, c.ffn, c.ffn, box))
    return DORY_ECUDA;
  // destinations of the staged QKV+gate epilogue (q, k, v, sigmoid(g))
  EpiMaps em;
  const int hk = c.n_kv * c.head_dim;
  if (!encode_bf16(&em.q, m->ws + m->L.q, M, hq, hq, 128) ||
      !encode_bf16(&em.k, m->ws + m->L.k, M, hk, hk, 128) ||
      !encode_bf16(&em.v, m->ws + m->L.v, M, hk, hk, 128) ||
      !encode_bf16(&em.g, m->ws + m->L.g, M, hq, hq, 128) ||
      !encode_f32_out(&em.out, m->ws + m->L.y32, M, c.d, c.d))   // output / down projections
    return DORY_ECUDA;

  if (m->mixed_step) {
    SeqPos sp{};
    for (int b = 0; b < m->mix_bd; ++b) sp.p[b] = m->seq_len[b];
    const int n = 2 * M * (c.head_dim / 2);
    pb(m, DORY_K_ROPE, st);
    DORY_TRY(pe(m, st,
                launch_k(rope_mixed_kernel, dim3((n + 255) / 256), dim3(256), 0, st,
                         c.rope ? wsp<float2>(m, m->L.rope_swa) : nullptr,
                         c.rope ? wsp<float2>(m, m->L.rope_full) : nullptr,
                         wsp<float2>(m, m->L.ropet_swa), wsp<float2>(m, m->L.ropet_full), sp,
                         m->mix_bd, m->mix_p, M - m->mix_bd, c.head_dim, (double)c.rope_base_swa,
                         (double)c.rope_base_full, wsp<int>(m, m->L.seq_pos)) == cudaSuccess
                    ? DORY_OK
                    : DORY_ECUDA));
  } else if (m->ragged_step) {
    // each sequence's position: RoPE rows and the positions for the attention
    SeqPos sp{};
    for (int b = 0; b < B; ++b) {
      sp.p[b] = m->seq_len[b];
      sp.k[b] = m->multi_k ? m->step_k[b] : 0;
    }
    const int n = 2 * B * (c.head_dim / 2);
    pb(m, DORY_K_ROPE, st);
    DORY_TRY(pe(m, st,
                launch_k(rope_rows_kernel, dim3((n + 255) / 256), dim3(256), 0, st,
                         c.rope ? wsp<float2>(m, m->L.rope_swa) : nullptr,
                         c.rope ? wsp<float2>(m, m->L.rope_full) : nullptr, sp, B, c.head_dim,
                         (double)c.rope_base_swa, (double)c.rope_base_full,
                         wsp<int>(m, m->L.seq_pos),
                         m->multi_k ? wsp<int>(m, m->L.seq_k) : nullptr) == cudaSuccess
                    ? DORY_OK
                    : DORY_ECUDA));
  } else if (c.rope) {
    const int n = 2 * C * (c.head_dim / 2);
    const int blocks = (n + 255) / 256;
    pb(m, DORY_K_ROPE, st);
    DORY_TRY(pe(m, st,
                launch_k(rope_table_kernel, dim3(blocks), dim3(256), 0, st,
                         wsp<float2>(m, m->L.rope_swa), wsp<float2>(m, m->L.rope_full),
                         wsp<float2>(m, m->L.ropet_swa), wsp<float2>(m, m->L.ropet_full), C, P0,
                         c.head_dim, (double)c.rope_base_swa, (double)c.rope_base_full) ==
                        cudaSuccess
                    ? DORY_OK
                    : DORY_ECUDA));
  }
  StepState s;
  pb(m, DORY_K_EMBED, st);
  DORY_TRY(pe(m, st,
              launch_k(embed_kernel, dim3(M), dim3(kRowThreads), 0, st, tokens, ld_tok, C,
                       reinterpret_cast<const __nv_bfloat16*>(m->embed_in), c.vocab, c.d,
                       hbuf(m, s.hsel), wsp<__nv_bfloat16>(m, m->L.hb), status) == cudaSuccess
                  ? DORY_OK
                  : DORY_ECUDA));

  auto layer = [&](int l, int slice, bool store) {
    if (decode) return run_layer_decode(m, l, slice, store, B, P0, s, st);
    if (batched) return run_layer_batched(m, l, slice, store, B, P0, tm_hb, tm_att, tm_m, s, st);
    return run_layer(m, l, slice, store, B, C, P0, tm_hb, tm_att, tm_m, em, s, st);
  };
  for (int l = 0; l < c.n_in; ++l) DORY_TRY(layer(l, 0, true));
  if (c.n_rec > 0) {
    // per-sequence loop counts (last-loop cache): k is the largest; a
    // sequence stores its keys and values at its own last loop and keeps its
    // final state from there to the output block
    const bool per_loop = m->cache_mode == DORY_CACHE_PER_LOOP;
    for (int i = 1; i <= k; ++i) {
      DORY_TRY(boundary(m, M, i == 1 ? BND_SAVE_ENTER : BND_ENTER_NEXT, s, st, i - 1));
      const int slice = per_loop ? i - 1 : 0;
      const bool store = per_loop || (i == k && !m->multi_k);
      m->step_loop = i;
      for (int l = c.n_in; l < c.n_in + c.n_rec; ++l) DORY_TRY(layer(l, slice, store));
    }
    m->step_loop = 0;
    DORY_TRY(boundary(m, M, BND_EXIT, s, st, k));
  }
  for (int l = c.n_in + c.n_rec; l < n_layers(c); ++l) DORY_TRY(layer(l, 0, true));
  DORY_TRY(flush_pending(m, s, M, st));
  m->hsel_last = s.hsel;

  if (logits && n_logit_rows > 0) {
    // LM head on the selected rows: per sequence, rows C - n .. C-1 of hb
    const int first = C - n_logit_rows;
    GemmArgs gl{};
    gl.w_pre = 1;   // weight operand: loads may start before the wait
    gl.N = c.vocab;
    gl.K = c.d;
    gl.status = status;
    gl.col_scale = m->s_z;
    gl.ldo = c.vocab;
    if (n_logit_rows == 1 && decode) {
      GemvArgs g{};
      g.M = B;
      g.X = wsp<__nv_bfloat16>(m, m->L.hb) + (size_t)(C - 1) * c.d;
      g.ldx = C * c.d;
      g.W = static_cast<const __nv_bfloat16*>(m->embed_out);
      g.N = c.vocab;
      g.K = c.d;
      g.Y = logits + (long long)t_out0 * c.vocab;
      g.ldy = (int)(ld_seq * c.vocab);
      g.col_scale = m->s_z;
      pb(m, DORY_K_LM_HEAD, st);
      DORY_TRY(pe(m, st, launch_gemv(g, st, wsp<int>(m, m->L.status))));
    } else if (n_logit_rows == 1) {
      // one row per sequence: a strided view of hb (row stride C * d)
      CUtensorMap tm_last;
      if (!encode_bf16(&tm_last, m->ws + m->L.hb + (size_t)(C - 1) * c.d * 2, B, c.d,
                       (uint64_t)C * c.d, 128))
        return DORY_ECUDA;
      gl.M = B;
      gl.ldo = ld_seq * c.vocab;
      gl.out = logits + (long long)t_out0 * c.vocab;
      EpiMaps el;
      const bool st_ok = encode_f32_out(&el.out, gl.out, B, c.vocab, gl.ldo);
      pb(m, DORY_K_LM_HEAD, st);
      DORY_TRY(pe(m, st, launch_gemm<kGemmBN, EPI_F32>(tm_last, m->tm_embed_out, gl, st,
                                                        st_ok ? &el : nullptr)));
    } else {
      for (int b = 0; b < B; ++b) {
        CUtensorMap tm_rows;
        if (!encode_bf16(&tm_rows, m->ws + m->L.hb + ((size_t)b * C + first) * c.d * 2,
                         n_logit_rows, c.d, c.d, 128))
          return DORY_ECUDA;
        gl.M = n_logit_rows;
        gl.out = logits + ((long long)b * ld_seq + t_out0) * c.vocab;
        EpiMaps el;
        const bool st_ok = encode_f32_out(&el.out, gl.out, n_logit_rows, c.vocab, gl.ldo);
        pb(m, DORY_K_LM_HEAD, st);
        DORY_TRY(pe(m, st, launch_gemm<kGemmBN, EPI_F32>(tm_rows, m->tm_embed_out, gl, st,
                                                          st_ok ? &el : nullptr)));
      }
    }
  }
  m->len += C;
  m->last_rows = M;
  return DORY_OK;
}

int check_call(dory_model* m, int B, int n_new, int k, int cache_mode) {
  if (!m) return DORY_EINVAL;
  if (!m->bound) return DORY_EUNBOUND;
  if (B <= 0 || n_new <= 0 || k <= 0) return DORY_EINVAL;
  if (cache_mode != DORY_CACHE_LAST_LOOP && cache_mode != DORY_CACHE_PER_LOOP) return DORY_EINVAL;
  if (cache_mode != m->cache_mode) return DORY_EKMISMATCH;
  if (m->cache_mode == DORY_CACHE_PER_LOOP && k != m->k_max) return DORY_EKMISMATCH;
  if (B > m->max_batch) return DORY_ECAPACITY;
  if ((long long)m->len + n_new > m->max_ctx) return DORY_ECAPACITY;
  if (m->batch != 0 && m->len > 0 && B != m->batch) return DORY_EINVAL;
  return DORY_OK;
}


int dory_prefill_body(dory_t* m, const int32_t* tokens, int B, int T, int k, float* logits,
                      int all_logits, void* stream);

// Logits of n consecutive rows of the last step's final hidden states (bf16
// copy), from row row0, into out [n][vocab] (s_z applied).
int lm_head_rows(dory_model* m, int row0, int n, float* out, cudaStream_t st) {
  const dory_config& c = m->cfg;
  if (n <= kGemvMaxM) {
    GemvArgs g{};
    g.M = n;
    g.X = wsp<__nv_bfloat16>(m, m->L.hb) + (size_t)row0 * c.d;
    g.ldx = c.d;
    g.W = static_cast<const __nv_bfloat16*>(m->embed_out);
    g.N = c.vocab;
    g.K = c.d;
    g.Y = out;
    g.ldy = c.vocab;
    g.col_scale = m->s_z;
    pb(m, DORY_K_LM_HEAD, st);
    return pe(m, st, launch_gemv(g, st, wsp<int>(m, m->L.status)));
  }
  CUtensorMap tm_rows;
  if (!encode_bf16(&tm_rows, m->ws + m->L.hb + (size_t)row0 * c.d * 2, n, c.d, c.d, 128))
    return DORY_ECUDA;
  GemmArgs gl{};
  gl.w_pre = 1;
  gl.M = n;
  gl.N = c.vocab;
  gl.K = c.d;
  gl.status = wsp<int>(m, m->L.status);
  gl.col_scale = m->s_z;
  gl.ldo = c.vocab;
  gl.out = out;
  EpiMaps el;
  const bool st_ok = encode_f32_out(&el.out, out, n, c.vocab, c.vocab);
  pb(m, DORY_K_LM_HEAD, st);
  return pe(m, st, launch_gemm<kGemmBN, EPI_F32>(tm_rows, m->tm_embed_out, gl, st,
                                                 st_ok ? &el : nullptr));
}

// One decode step of batch slots 0 .. B-1 at their own lengths, with one
// loop count k for all or (ks, host array, last-loop cache) one per
// sequence, k then being the largest.
int ragged_decode(dory_model* m, const int32_t* tokens, int B, int k, const int* ks,
                  int cache_mode, float* logits, int32_t* next, void* stream) {
  if (!m || !tokens) return DORY_EINVAL;
  if (!m->bound) return DORY_EUNBOUND;
  if (B <= 0) return DORY_EINVAL;
  if (B > kRaggedMax) return DORY_EUNSUPPORTED;
  if (next && !logits) return DORY_EINVAL;
  if (B > m->max_batch) return DORY_ECAPACITY;
  if (!m->ragged) {
    for (int b = 0; b < m->max_batch; ++b) m->seq_len[b] = b < m->batch ? m->len : 0;
    m->ragged = true;
  }
  int pmax = 0;
  for (int b = 0; b < B; ++b) {
    if (m->seq_len[b] + 1 > m->max_ctx) return DORY_ECAPACITY;
    if (m->seq_len[b] > pmax) pmax = m->seq_len[b];
  }
  const int saved_len = m->len, saved_batch = m->batch;
  m->len = pmax;                        // the step's largest position (schedules)
  m->batch = 0;
  int rc = check_call(m, B, 1, k, cache_mode);
  if (rc == DORY_OK) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    m->launches = 0;
    m->ragged_step = true;
    m->multi_k = ks != nullptr;
    if (ks) m->step_k.assign(ks, ks + B);
    rc = run_step(m, tokens, 1, B, 1, k, logits, 1, 0, logits ? 1 : 0, st, next);
    m->ragged_step = false;
    m->multi_k = false;
    if (rc == DORY_OK && next && !m->next_done) {
      pb(m, DORY_K_ARGMAX, st);
      rc = pe(m, st,
              launch_k(argmax_kernel, dim3(B), dim3(1024), 0, st, (const float*)logits,
                       m->cfg.vocab, next) == cudaSuccess
                  ? DORY_OK
                  : DORY_ECUDA);
    }
    if (rc == DORY_OK)
      for (int b = 0; b < B; ++b) m->seq_len[b] += 1;
  }
  m->len = saved_len;
  m->batch = saved_batch > B ? saved_batch : B;
  return rc;
}

}  // namespace

// ====================================================================== ABI
extern "C" {

int dory_create(const dory_config* cfg, const dory_weights* w, dory_t** out) {
  if (!out) return DORY_EINVAL;
  *out = nullptr;
  const int rc = validate_config(cfg);
  if (rc != DORY_OK) return rc;
  if (!w || !w->embed_in || !w->embed_out || !w->layers) return DORY_EINVAL;
  const int L = n_layers(*cfg);
  for (int l = 0; l < L; ++l) {
    const dory_layer_weights& lw = w->layers[l];
    if (!lw.w_qkvg || !lw.w_o || !lw.w_upgate || !lw.w_down || !lw.alpha_attn || !lw.alpha_mlp ||
        !lw.s_qk)
      return DORY_EINVAL;
  }
  dory_model* m = new (std::nothrow) dory_model();
  if (!m) return DORY_ENOMEM;
  m->cfg = *cfg;
  m->layers.assign(w->layers, w->layers + L);
  m->embed_in = w->embed_in;
  m->embed_out = w->embed_out;
  m->s_z = w->s_z;
  *out = m;
  return DORY_OK;
}

size_t dory_kv_bytes(const dory_config* cfg, int max_batch, int max_ctx, int k, int cache_mode) {
  if (validate_config(cfg) != DORY_OK || max_batch <= 0 || max_ctx <= 0 || k <= 0) return 0;
  if (cache_mode != DORY_CACHE_LAST_LOOP && cache_mode != DORY_CACHE_PER_LOOP) return 0;
  return kv_offset(*cfg, max_batch, max_ctx, k, cache_mode, n_layers(*cfg), 0, 0);
}

size_t dory_workspace_bytes(const dory_config* cfg, int max_batch, int max_chunk) {
  if (validate_config(cfg) != DORY_OK || max_batch <= 0 || max_chunk <= 0) return 0;
  return ws_layout(*cfg, max_batch, max_chunk).total;
}

int dory_bind(dory_t* m, void* kv, size_t kv_bytes, void* ws, size_t ws_bytes, int max_batch,
              int max_ctx, int max_chunk, int k_max, int cache_mode) {
  if (!m || !kv || !ws || max_batch <= 0 || max_ctx <= 0 || max_chunk <= 0 || k_max <= 0)
    return DORY_EINVAL;
  if (cache_mode != DORY_CACHE_LAST_LOOP && cache_mode != DORY_CACHE_PER_LOOP) return DORY_EINVAL;
  if (((uintptr_t)kv & 255) || ((uintptr_t)ws & 255)) return DORY_EINVAL;
  const dory_config& c = m->cfg;
  if (kv_bytes < dory_kv_bytes(&c, max_batch, max_ctx, k_max, cache_mode)) return DORY_ENOMEM;
  if (ws_bytes < dory_workspace_bytes(&c, max_batch, max_chunk)) return DORY_ENOMEM;
  const int L = n_layers(c);
  std::vector<CUtensorMap> q(L), o(L), u(L), dn(L);
  const int hq = c.n_q * c.head_dim;
  const int nqkvg = (2 * c.n_q + 2 * c.n_kv) * c.head_dim;
  for (int l = 0; l < L; ++l) {
    const dory_layer_weights& w = m->layers[l];
    if (!encode_bf16(&q[l], w.w_qkvg, nqkvg, c.d, c.d, kGemmBN / 2) ||
        !encode_bf16(&o[l], w.w_o, c.d, hq, hq, kGemmBN / 2) ||
        !encode_bf16(&u[l], w.w_upgate, 2 * (uint64_t)c.ffn, c.d, c.d, kGemmBN / 2) ||
        !encode_bf16(&dn[l], w.w_down, c.d, c.ffn, c.ffn, kGemmBN / 2))
      return DORY_ECUDA;
  }
  CUtensorMap eo;
  if (!encode_bf16(&eo, m->embed_out, c.vocab, c.d, c.d, kGemmBN / 2)) return DORY_ECUDA;
  m->tm_qkvg.swap(q);
  m->tm_o.swap(o);
  m->tm_upgate.swap(u);
  m->tm_down.swap(dn);
  m->tm_embed_out = eo;
  m->kv = static_cast<uint8_t*>(kv);
  m->ws = static_cast<uint8_t*>(ws);
  m->max_batch = max_batch;
  m->max_ctx = max_ctx;
  m->max_chunk = max_chunk;
  m->k_max = k_max;
  m->cache_mode = cache_mode;
  m->L = ws_layout(c, max_batch, max_chunk);
  m->bound = true;
  m->len = 0;
  m->batch = 0;
  m->last_rows = 0;
  m->hsel_last = 0;
  m->seq_len.assign(max_batch, 0);
  m->ragged = false;
  m->slot = 0;
  // status word and split tickets start at zero (tickets return to zero
  // after every launch that uses them)
  if (cudaMemsetAsync(m->ws + m->L.status, 0, 256, 0) != cudaSuccess ||
      cudaMemsetAsync(m->ws + m->L.dec_cnt, 0, (size_t)max_batch * c.n_kv * 4, 0) != cudaSuccess ||
      cudaStreamSynchronize(0) != cudaSuccess)
    return DORY_ECUDA;
  return DORY_OK;
}

int dory_prefill(dory_t* m, const int32_t* tokens, int B, int T, int k, int cache_mode,
                 float* logits, int all_logits, void* stream) {
  int rc = check_call(m, B, T, k, cache_mode);
  if (rc != DORY_OK) return rc;
  if (!tokens) return DORY_EINVAL;
  if (m->ragged) return DORY_EINVAL;     // per-sequence lengths: dory_prefill_slot
  rc = dory_prefill_body(m, tokens, B, T, k, logits, all_logits, stream);
  if (rc == DORY_OK)
    for (int b = 0; b < B; ++b) m->seq_len[b] = m->len;
  return rc;
}
}  // extern "C"

namespace {
// The chunk loop of a prefill of B sequences at m->len (from batch slot
// m->slot when B == 1).
int dory_prefill_body(dory_t* m, const int32_t* tokens, int B, int T, int k, float* logits,
                      int all_logits, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  m->launches = 0;
  m->batch = B;
  for (int t0 = 0; t0 < T; t0 += m->max_chunk) {
    const int C = T - t0 < m->max_chunk ? T - t0 : m->max_chunk;
    const bool last = t0 + C == T;
    float* lg = nullptr;
    int nrows = 0;
    long long ld_seq = 1;
    int t_out0 = 0;
    if (logits && all_logits) {
      lg = logits;
      nrows = C;
      ld_seq = T;
      t_out0 = t0;
    } else if (logits && last) {
      lg = logits;
      nrows = 1;
      ld_seq = 1;
      t_out0 = 0;
    }
    const int r = run_step(m, tokens + t0, T, B, C, k, lg, ld_seq, t_out0, nrows, st);
    if (r != DORY_OK) return r;
  }
  return DORY_OK;
}
}  // namespace

extern "C" {

int dory_decode_step(dory_t* m, const int32_t* tokens, int B, int k, int cache_mode,
                     float* logits, int32_t* next, void* stream) {
  const int rc = check_call(m, B, 1, k, cache_mode);
  if (rc != DORY_OK) return rc;
  if (!tokens) return DORY_EINVAL;
  if (m->ragged) return DORY_EINVAL;     // per-sequence lengths: dory_decode_step_ragged
  if (next && !logits) return DORY_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  m->launches = 0;
  m->batch = B;
  const int r = run_step(m, tokens, 1, B, 1, k, logits, 1, 0, logits ? 1 : 0, st, next);
  if (r != DORY_OK) return r;
  for (int b = 0; b < B; ++b) m->seq_len[b] = m->len;
  if (next && !m->next_done) {
    pb(m, DORY_K_ARGMAX, st);
    return pe(m, st,
              launch_k(argmax_kernel, dim3(B), dim3(1024), 0, st, (const float*)logits,
                       m->cfg.vocab, next) == cudaSuccess
                  ? DORY_OK
                  : DORY_ECUDA);
  }
  return DORY_OK;
}

// ---------------------------------------------------------------- speculative
}  // extern "C"

namespace {
constexpr int kSpecMaxGamma = 16;

// Sliding-window blocks of the bound KV region (every slice): the ring slots
// a speculative step overwrites and may have to put back.
std::vector<SpecRing> spec_rings(const dory_model* m) {
  std::vector<SpecRing> r;
  const dory_config& c = m->cfg;
  for (int l = 0; l < n_layers(c); ++l) {
    if (layer_full(c, l)) continue;
    for (int sl = 0; sl < mult_of(c, l, m->k_max, m->cache_mode); ++sl) {
      SpecRing g{};
      g.k_off = (long long)kv_offset(c, m->max_batch, m->max_ctx, m->k_max, m->cache_mode, l, sl, 0);
      g.v_off = (long long)kv_offset(c, m->max_batch, m->max_ctx, m->k_max, m->cache_mode, l, sl, 1);
      g.slots = slots_of(c, l, m->max_ctx);
      r.push_back(g);
    }
  }
  return r;
}

struct SpecScratch {
  size_t logits, drafts, vin, g, n, table, backup, dlogits, stats, kept, total;
};

SpecScratch spec_layout(const dory_model* m, int B, int gamma, size_t n_rings) {
  const dory_config& c = m->cfg;
  SpecScratch L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += align256(bytes);
    return at;
  };
  L.logits = take((size_t)B * (gamma + 1) * c.vocab * 4);
  L.drafts = take((size_t)gamma * B * 4);
  L.vin = take((size_t)B * (gamma + 1) * 4);
  L.g = take((size_t)B * (gamma + 1) * 4);
  L.n = take(4);
  L.table = take(n_rings * sizeof(SpecRing));
  L.backup = take(n_rings * 2 * (size_t)B * c.n_kv * (gamma + 1) * c.head_dim * 2);
  // sampling only: the drafter's logits, softmax statistics, kept counts
  L.dlogits = take((size_t)gamma * B * c.vocab * 4);
  L.stats = take((size_t)(2 * gamma + 1) * B * sizeof(float2));
  L.kept = take((size_t)B * 4);
  L.total = off;
  return L;
}
}  // namespace

extern "C" {

size_t dory_speculative_scratch_bytes(const dory_t* m, int B, int gamma) {
  if (!m || !m->bound || B <= 0 || gamma < 1 || gamma > kSpecMaxGamma) return 0;
  return spec_layout(m, B, gamma, spec_rings(m).size()).total;
}

}  // extern "C"

namespace {
// Greedy (temperature 0, u null) or sampled self-speculative step.
int speculative_step(dory_t* m, const int32_t* tokens, int B, int k_draft, int k_verify,
                     int gamma, float temperature, const float* u, void* scratch,
                     size_t scratch_bytes, int32_t* out, int* n_out, int32_t* kept_out,
                     void* stream) {
  if (!m || !tokens || !scratch || !out || !n_out) return DORY_EINVAL;
  if (!m->bound) return DORY_EUNBOUND;
  if (gamma < 1 || gamma > kSpecMaxGamma || k_draft < 1 || k_draft > k_verify) return DORY_EINVAL;
  if (m->cache_mode != DORY_CACHE_PER_LOOP || k_verify != m->k_max) return DORY_EKMISMATCH;
  if (reinterpret_cast<uintptr_t>(scratch) & 255) return DORY_EINVAL;
  if (m->ragged) return DORY_EINVAL;     // sequences of one length only
  // the verifying pass is one chunk of gamma + 1 tokens per sequence
  int rc = check_call(m, B, gamma + 1, k_verify, DORY_CACHE_PER_LOOP);
  if (rc != DORY_OK) return rc;
  if (gamma + 1 > m->max_chunk) return DORY_ECAPACITY;
  const std::vector<SpecRing> rings = spec_rings(m);
  const SpecScratch S = spec_layout(m, B, gamma, rings.size());
  if (scratch_bytes < S.total) return DORY_ENOMEM;
  const dory_config& c = m->cfg;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* sc = static_cast<uint8_t*>(scratch);
  float* logits = reinterpret_cast<float*>(sc + S.logits);
  int32_t* drafts = reinterpret_cast<int32_t*>(sc + S.drafts);
  int32_t* vin = reinterpret_cast<int32_t*>(sc + S.vin);
  int32_t* g = reinterpret_cast<int32_t*>(sc + S.g);
  int* n_dev = reinterpret_cast<int*>(sc + S.n);
  SpecRing* table = reinterpret_cast<SpecRing*>(sc + S.table);
  uint4* backup = reinterpret_cast<uint4*>(sc + S.backup);
  float* dlogits = reinterpret_cast<float*>(sc + S.dlogits);
  float2* stats = reinterpret_cast<float2*>(sc + S.stats);
  int32_t* kept = reinterpret_cast<int32_t*>(sc + S.kept);
  const bool sampled = u != nullptr;
  const float inv_t = sampled ? 1.0f / temperature : 0.0f;
  const int L = m->len;
  const int nr = (int)rings.size();
  m->launches = 0;
  m->batch = B;
  auto ring_copy = [&](int dir, const int* i0) -> int {
    if (nr == 0) return DORY_OK;
    const long long chunks = (long long)nr * 2 * B * c.n_kv * (gamma + 1) * (c.head_dim / 8);
    long long blocks = (chunks + 255) / 256;
    if (blocks > 4 * num_sms()) blocks = 4 * num_sms();
    return launch_k(spec_ring_copy_kernel, dim3((unsigned)blocks), dim3(256), 0, st, m->kv,
                    (const SpecRing*)table, nr, B, c.n_kv, c.head_dim, L, gamma + 1, backup, dir,
                    i0) == cudaSuccess
               ? DORY_OK
               : DORY_ECUDA;
  };
  if (nr > 0 &&
      cudaMemcpyAsync(table, rings.data(), rings.size() * sizeof(SpecRing), cudaMemcpyHostToDevice,
                      st) != cudaSuccess)
    return DORY_ECUDA;
  // the window-ring slots of positions L .. L + gamma, which drafting and
  // verifying overwrite (slot p mod W held position p - W, still visible)
  DORY_TRY(ring_copy(0, nullptr));
  // drafts: gamma decode steps at k_draft (per-loop slices 1..k_draft),
  // greedy or drawn from softmax(z / T) with uniform column i
  for (int i = 0; i < gamma; ++i) {
    const int32_t* in = i == 0 ? tokens : drafts + (i - 1) * B;
    if (sampled) {
      float* dl = dlogits + (size_t)i * B * c.vocab;
      DORY_TRY(run_step(m, in, 1, B, 1, k_draft, dl, 1, 0, 1, st));
      DORY_TRY(launch_k(sample_kernel, dim3(B), dim3(kSampleThreads), 0, st, (const float*)dl,
                        c.vocab, inv_t, u + i, 2 * gamma + 1, drafts + i * B) == cudaSuccess
                   ? DORY_OK
                   : DORY_ECUDA);
      continue;
    }
    DORY_TRY(run_step(m, in, 1, B, 1, k_draft, logits, 1, 0, 1, st, drafts + i * B));
    if (!m->next_done) {
      pb(m, DORY_K_ARGMAX, st);
      DORY_TRY(pe(m, st,
                  launch_k(argmax_kernel, dim3(B), dim3(1024), 0, st, (const float*)logits, c.vocab,
                           drafts + i * B) == cudaSuccess
                      ? DORY_OK
                      : DORY_ECUDA));
    }
  }
  // back to the state before drafting; one verifying pass over the last
  // emitted token and the drafts at k_verify, logits at every position
  DORY_TRY(ring_copy(1, nullptr));
  m->len = L;
  DORY_TRY(launch_k(spec_gather_kernel, dim3(1), dim3(256), 0, st, tokens, (const int32_t*)drafts,
                    B, gamma, vin) == cudaSuccess
               ? DORY_OK
               : DORY_ECUDA);
  DORY_TRY(run_step(m, vin, gamma + 1, B, gamma + 1, k_verify, logits, gamma + 1, 0, gamma + 1,
                    st));
  if (sampled) {
    // softmax statistics of the verifier's and the drafter's rows, kept
    // drafts, emitted tokens (rejection sampling)
    float2* sp = stats;
    float2* sq = stats + (size_t)B * (gamma + 1);
    DORY_TRY(launch_k(row_stats_kernel, dim3(B * (gamma + 1)), dim3(kSampleThreads), 0, st,
                      (const float*)logits, c.vocab, inv_t, sp) == cudaSuccess
                 ? DORY_OK
                 : DORY_ECUDA);
    DORY_TRY(launch_k(row_stats_kernel, dim3(B * gamma), dim3(kSampleThreads), 0, st,
                      (const float*)dlogits, c.vocab, inv_t, sq) == cudaSuccess
                 ? DORY_OK
                 : DORY_ECUDA);
    DORY_TRY(launch_k(spec_keep_kernel, dim3(1), dim3(256), 0, st, (const float*)logits,
                      (const float2*)sp, (const float*)dlogits, (const float2*)sq,
                      (const int32_t*)drafts, u, B, gamma, c.vocab, inv_t, kept) == cudaSuccess
                 ? DORY_OK
                 : DORY_ECUDA);
    DORY_TRY(launch_k(spec_emit_kernel, dim3(B), dim3(kSampleThreads), 0, st,
                      (const float*)logits, (const float2*)sp, (const float*)dlogits,
                      (const float2*)sq, (const int32_t*)drafts, u, (const int32_t*)kept, B, gamma,
                      c.vocab, inv_t, out, n_dev) == cudaSuccess
                 ? DORY_OK
                 : DORY_ECUDA);
    if (kept_out && cudaMemcpyAsync(kept_out, kept, (size_t)B * 4, cudaMemcpyDeviceToDevice, st) !=
                        cudaSuccess)
      return DORY_ECUDA;
  } else {
    pb(m, DORY_K_ARGMAX, st);
    DORY_TRY(pe(m, st,
                launch_k(argmax_kernel, dim3(B * (gamma + 1)), dim3(1024), 0, st,
                         (const float*)logits, c.vocab, g) == cudaSuccess
                    ? DORY_OK
                    : DORY_ECUDA));
    DORY_TRY(launch_k(spec_accept_kernel, dim3(1), dim3(256), 0, st, (const int32_t*)drafts,
                      (const int32_t*)g, B, gamma, out, n_dev) == cudaSuccess
                 ? DORY_OK
                 : DORY_ECUDA);
  }
  // positions past the accepted ones go back to what the rings held
  DORY_TRY(ring_copy(1, n_dev));
  int n = 0;
  if (cudaMemcpyAsync(&n, n_dev, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return DORY_ECUDA;
  if (n < 1 || n > gamma + 1) return DORY_EDEVICE;
  m->len = L + n;
  for (int b = 0; b < B; ++b) m->seq_len[b] = m->len;
  *n_out = n;
  return DORY_OK;
}

}  // namespace

extern "C" {

int dory_speculative_step(dory_t* m, const int32_t* tokens, int B, int k_draft, int k_verify,
                          int gamma, void* scratch, size_t scratch_bytes, int32_t* out, int* n_out,
                          void* stream) {
  return speculative_step(m, tokens, B, k_draft, k_verify, gamma, 0.0f, nullptr, scratch,
                          scratch_bytes, out, n_out, nullptr, stream);
}

int dory_speculative_sample_step(dory_t* m, const int32_t* tokens, int B, int k_draft,
                                 int k_verify, int gamma, float temperature, const float* u,
                                 void* scratch, size_t scratch_bytes, int32_t* out, int* n_out,
                                 int32_t* kept, void* stream) {
  if (!u || !(temperature > 0.0f)) return DORY_EINVAL;
  return speculative_step(m, tokens, B, k_draft, k_verify, gamma, temperature, u, scratch,
                          scratch_bytes, out, n_out, kept, stream);
}

int dory_debug_speculative_layout(const dory_t* m, int B, int gamma, size_t* offsets) {
  if (!m || !offsets || !m->bound || B <= 0 || gamma < 1 || gamma > kSpecMaxGamma)
    return DORY_EINVAL;
  const SpecScratch S = spec_layout(m, B, gamma, spec_rings(m).size());
  offsets[0] = S.logits;
  offsets[1] = S.dlogits;
  offsets[2] = S.drafts;
  return DORY_OK;
}

int dory_sample_tokens(const float* logits, int rows, int V, float temperature, const float* u,
                       int32_t* out, void* stream) {
  if (!logits || !u || !out || rows <= 0 || V <= 0 || !(temperature > 0.0f)) return DORY_EINVAL;
  return launch_k(sample_kernel, dim3(rows), dim3(kSampleThreads), 0,
                  static_cast<cudaStream_t>(stream), logits, V, 1.0f / temperature, u, 1,
                  out) == cudaSuccess
             ? DORY_OK
             : DORY_ECUDA;
}

int dory_copy_prefix(dory_t* m, int src, const int* dst, int n_dst, int len, void* stream) {
  if (!m || !dst || n_dst <= 0 || n_dst > kKvCopyMaxDst || len <= 0) return DORY_EINVAL;
  if (!m->bound) return DORY_EUNBOUND;
  if (src < 0 || src >= m->max_batch) return DORY_EINVAL;
  if (len > m->max_ctx) return DORY_ECAPACITY;
  const dory_config& c = m->cfg;
  KvCopyTable t;
  t.n_dst = n_dst;
  t.src = src;
  t.max_batch = m->max_batch;
  for (int i = 0; i < n_dst; ++i) {
    if (dst[i] < 0 || dst[i] >= m->max_batch || dst[i] == src) return DORY_EINVAL;
    t.dst[i] = dst[i];
  }
  int nb = 0, max_rows = 0;
  for (int l = 0; l < n_layers(c); ++l) {
    for (int sl = 0; sl < mult_of(c, l, m->k_max, m->cache_mode); ++sl) {
      if (nb == kKvCopyMaxBlocks) return DORY_EUNSUPPORTED;
      t.k_off[nb] = (long long)kv_offset(c, m->max_batch, m->max_ctx, m->k_max, m->cache_mode, l,
                                         sl, 0);
      t.slots[nb] = slots_of(c, l, m->max_ctx);
      // positions 0 .. len-1: slots 0 .. len-1 on full layers; on a window
      // ring the whole ring once it has wrapped (slot p mod slots)
      t.rows[nb] = len < t.slots[nb] ? len : t.slots[nb];
      if (t.rows[nb] > max_rows) max_rows = t.rows[nb];
      ++nb;
    }
  }
  t.n_blocks = nb;
  const long long chunks = 2ll * c.n_kv * max_rows * (c.head_dim / 8);
  const dim3 grid((unsigned)((chunks + 255) / 256), (unsigned)nb, (unsigned)n_dst);
  return launch_k(kv_copy_kernel, grid, dim3(256), 0, static_cast<cudaStream_t>(stream), m->kv, t,
                  c.n_kv, c.head_dim) == cudaSuccess
             ? DORY_OK
             : DORY_ECUDA;
}

int dory_quant_bytes(int fmt, int rows, int K, size_t* codes_bytes, size_t* scales_bytes) {
  if ((fmt != DORY_QUANT_MXFP8 && fmt != DORY_QUANT_NVFP4) || rows <= 0 || K <= 0 || K % 32 ||
      !codes_bytes || !scales_bytes)
    return DORY_EINVAL;
  const size_t n = (size_t)rows * K;
  *codes_bytes = fmt == DORY_QUANT_MXFP8 ? n : n / 2;
  *scales_bytes = fmt == DORY_QUANT_MXFP8 ? n / 32 : n / 16;
  return DORY_OK;
}

int dory_quantize_matrix(int fmt, const void* W, int rows, int K, void* codes, void* scales,
                         float* row_scale, void* deq, void* stream) {
  size_t cb = 0, sb = 0;
  if (dory_quant_bytes(fmt, rows, K, &cb, &sb) != DORY_OK || !W || !codes || !scales)
    return DORY_EINVAL;
  if (fmt == DORY_QUANT_NVFP4 && !row_scale) return DORY_EINVAL;
  auto al = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
  if (!al(W, 16) || !al(codes, 16) || (deq && !al(deq, 16)) || (row_scale && !al(row_scale, 4)))
    return DORY_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long n = (long long)rows * K;
  const __nv_bfloat16* w = static_cast<const __nv_bfloat16*>(W);
  __nv_bfloat16* dq = static_cast<__nv_bfloat16*>(deq);
  // plain launches: these kernels do not take part in programmatic
  // dependent launch, so each waits for all earlier work on the stream
  if (fmt == DORY_QUANT_MXFP8) {
    const long long nb = n / 32;
    quant_mxfp8_kernel<<<(unsigned)((nb + 127) / 128), 128, 0, st>>>(
        w, nb, static_cast<uint8_t*>(codes), static_cast<uint8_t*>(scales), dq, row_scale, K);
  } else {
    const long long nb = n / 16;
    if (cudaMemsetAsync(row_scale, 0, sizeof(float), st) != cudaSuccess) return DORY_ECUDA;
    long long g = (n / 8 + 255) / 256;
    if (g > 4ll * num_sms()) g = 4ll * num_sms();
    quant_amax_kernel<<<(unsigned)g, 256, 0, st>>>(w, n, reinterpret_cast<unsigned*>(row_scale));
    quant_gscale_kernel<<<1, 256, 0, st>>>(row_scale, rows);
    quant_nvfp4_kernel<<<(unsigned)((nb + 127) / 128), 128, 0, st>>>(
        w, nb, K, row_scale, static_cast<uint8_t*>(codes), static_cast<uint8_t*>(scales), dq);
  }
  return cudaGetLastError() == cudaSuccess ? DORY_OK : DORY_ECUDA;
}

int dory_set_quantized_weights(dory_t* m, int fmt, const dory_qlayer* layers) {
  if (!m) return DORY_EINVAL;
  if (fmt == DORY_QUANT_NONE) {
    m->qfmt = 0;
    m->qlayers.clear();
    return DORY_OK;
  }
  if ((fmt != DORY_QUANT_MXFP8 && fmt != DORY_QUANT_NVFP4) || !layers) return DORY_EINVAL;
  const dory_config& c = m->cfg;
  if (c.d % 32 || (c.n_q * c.head_dim) % 32 || c.ffn % 32) return DORY_EINVAL;
  auto al = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
  for (int l = 0; l < n_layers(c); ++l) {
    const dory_qmatrix* q[4] = {&layers[l].qkvg, &layers[l].o, &layers[l].upgate, &layers[l].down};
    for (const dory_qmatrix* x : q) {
      if (!x->codes || !x->scales || !al(x->codes, 16)) return DORY_EINVAL;
      if (fmt == DORY_QUANT_NVFP4 && (!x->row_scale || !al(x->scales, 2))) return DORY_EINVAL;
    }
  }
  m->qlayers.assign(layers, layers + n_layers(c));
  m->qfmt = fmt;
  return DORY_OK;
}

int dory_set_quantized_swap(dory_t* m, int stream_codes) {
  if (!m || (stream_codes != 0 && stream_codes != 1)) return DORY_EINVAL;
  m->q_swap = stream_codes;
  return DORY_OK;
}

int dory_length(const dory_t* m, int* out) {
  if (!m || !out) return DORY_EINVAL;
  *out = m->len;
  return DORY_OK;
}

int dory_set_length(dory_t* m, int B, int len) {
  if (!m) return DORY_EINVAL;
  if (!m->bound) return DORY_EUNBOUND;
  if (B <= 0 || len < 0) return DORY_EINVAL;
  if (B > m->max_batch || len > m->max_ctx) return DORY_ECAPACITY;
  m->len = len;
  m->batch = len > 0 ? B : 0;
  m->ragged = false;
  std::fill(m->seq_len.begin(), m->seq_len.end(), 0);
  for (int b = 0; b < B; ++b) m->seq_len[b] = len;
  return DORY_OK;
}

int dory_reset(dory_t* m) {
  if (!m) return DORY_EINVAL;
  m->len = 0;
  m->batch = 0;
  m->last_rows = 0;
  m->ragged = false;
  std::fill(m->seq_len.begin(), m->seq_len.end(), 0);
  return DORY_OK;
}

int dory_set_lengths(dory_t* m, int B, const int* lengths) {
  if (!m || !lengths) return DORY_EINVAL;
  if (!m->bound) return DORY_EUNBOUND;
  if (B <= 0) return DORY_EINVAL;
  if (B > m->max_batch) return DORY_ECAPACITY;
  for (int b = 0; b < B; ++b) {
    if (lengths[b] < 0) return DORY_EINVAL;
    if (lengths[b] > m->max_ctx) return DORY_ECAPACITY;
  }
  std::fill(m->seq_len.begin(), m->seq_len.end(), 0);
  for (int b = 0; b < B; ++b) m->seq_len[b] = lengths[b];
  m->ragged = true;
  m->batch = B;
  m->len = 0;
  return DORY_OK;
}

int dory_get_lengths(const dory_t* m, int B, int* out) {
  if (!m || !out || B <= 0) return DORY_EINVAL;
  if (!m->bound) return DORY_EUNBOUND;
  if (B > m->max_batch) return DORY_ECAPACITY;
  for (int b = 0; b < B; ++b) out[b] = m->ragged ? m->seq_len[b] : (b < m->batch ? m->len : 0);
  return DORY_OK;
}

int dory_prefill_slot(dory_t* m, int slot, const int32_t* tokens, int T, int k, int cache_mode,
                      float* logits, int all_logits, void* stream) {
  if (!m || !tokens) return DORY_EINVAL;
  if (!m->bound) return DORY_EUNBOUND;
  if (slot < 0 || slot >= m->max_batch) return DORY_EINVAL;
  if (!m->ragged) {
    // from the uniform state: every sequence of the batch keeps its length
    for (int b = 0; b < m->max_batch; ++b) m->seq_len[b] = b < m->batch ? m->len : 0;
    m->ragged = true;
  }
  const int saved_len = m->len, saved_batch = m->batch;
  m->len = m->seq_len[slot];
  m->batch = 0;
  m->slot = slot;
  int rc = check_call(m, 1, T, k, cache_mode);
  if (rc == DORY_OK) rc = dory_prefill_body(m, tokens, 1, T, k, logits, all_logits, stream);
  if (rc == DORY_OK) m->seq_len[slot] = m->len;
  m->slot = 0;
  m->len = saved_len;
  m->batch = saved_batch > slot + 1 ? saved_batch : slot + 1;
  return rc;
}

int dory_decode_step_ragged(dory_t* m, const int32_t* tokens, int B, int k, int cache_mode,
                            float* logits, int32_t* next, void* stream) {
  return ragged_decode(m, tokens, B, k, nullptr, cache_mode, logits, next, stream);
}

int dory_step_mixed(dory_t* m, const int32_t* tokens, int Bd, int slot, int C, int k,
                    int cache_mode, float* logits, int32_t* next, void* stream) {
  if (!m || !tokens) return DORY_EINVAL;
  if (!m->bound) return DORY_EUNBOUND;
  if (Bd < 0 || C < 1 || slot < Bd || slot >= m->max_batch) return DORY_EINVAL;
  if (Bd > kRaggedMax) return DORY_EUNSUPPORTED;
  if (next && (!logits || Bd == 0)) return DORY_EINVAL;
  if (C > m->max_chunk) return DORY_ECAPACITY;
  if (!m->ragged) {
    for (int b = 0; b < m->max_batch; ++b) m->seq_len[b] = b < m->batch ? m->len : 0;
    m->ragged = true;
  }
  for (int b = 0; b < Bd; ++b)
    if (m->seq_len[b] + 1 > m->max_ctx) return DORY_ECAPACITY;
  const int saved_len = m->len, saved_batch = m->batch;
  m->len = m->seq_len[slot];
  m->batch = 0;
  int rc = check_call(m, 1, C, k, cache_mode);
  if (rc == DORY_OK) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int M = Bd + C;
    m->launches = 0;
    m->mixed_step = true;
    m->mix_bd = Bd;
    m->mix_slot = slot;
    m->mix_p = m->seq_len[slot];
    rc = run_step(m, tokens, M, 1, M, k, nullptr, 1, 0, 0, st);
    m->mixed_step = false;
    if (rc == DORY_OK && logits && Bd > 0) rc = lm_head_rows(m, 0, Bd, logits, st);
    if (rc == DORY_OK && logits)
      rc = lm_head_rows(m, M - 1, 1, logits + (size_t)Bd * m->cfg.vocab, st);
    if (rc == DORY_OK && next) {
      pb(m, DORY_K_ARGMAX, st);
      rc = pe(m, st,
              launch_k(argmax_kernel, dim3(Bd), dim3(1024), 0, st, (const float*)logits,
                       m->cfg.vocab, next) == cudaSuccess
                  ? DORY_OK
                  : DORY_ECUDA);
    }
    if (rc == DORY_OK) {
      for (int b = 0; b < Bd; ++b) m->seq_len[b] += 1;
      m->seq_len[slot] += C;
    }
  }
  m->len = saved_len;
  m->batch = saved_batch > slot + 1 ? saved_batch : slot + 1;
  return rc;
}

int dory_decode_step_multi(dory_t* m, const int32_t* tokens, int B, const int* ks,
                           int cache_mode, float* logits, int32_t* next, void* stream) {
  if (!ks) return DORY_EINVAL;
  if (m && m->bound && cache_mode != DORY_CACHE_LAST_LOOP) return DORY_EKMISMATCH;
  int kmax = 0;
  for (int b = 0; b < B && B <= kRaggedMax; ++b) {
    if (ks[b] < 1) return DORY_EINVAL;
    if (ks[b] > kmax) kmax = ks[b];
  }
  return ragged_decode(m, tokens, B, kmax, ks, cache_mode, logits, next, stream);
}

int dory_destroy(dory_t* m) {
  if (!m) return DORY_EINVAL;
  for (cudaEvent_t e : m->prof_ev) cudaEventDestroy(e);
  delete m;
  return DORY_OK;
}

int dory_profile_begin(dory_t* m, int max_launches) {
  if (!m || max_launches <= 0) return DORY_EINVAL;
  if ((int)m->prof_cls.size() < max_launches) {
    while ((int)m->prof_ev.size() < 2 * max_launches) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return DORY_ECUDA;
      m->prof_ev.push_back(e);
    }
    m->prof_cls.assign(max_launches, 0);
  }
  m->prof_used = 0;
  m->prof_on = true;
  return DORY_OK;
}

int dory_profile_end(dory_t* m, double* ms, int* launches) {
  if (!m || !ms || !launches) return DORY_EINVAL;
  if (!m->prof_on) return DORY_EINVAL;
  m->prof_on = false;
  for (int c = 0; c < DORY_K_COUNT; ++c) {
    ms[c] = 0.0;
    launches[c] = 0;
  }
  for (int i = 0; i < m->prof_used; ++i) {
    if (cudaEventSynchronize(m->prof_ev[2 * i + 1]) != cudaSuccess) return DORY_ECUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, m->prof_ev[2 * i], m->prof_ev[2 * i + 1]) != cudaSuccess)
      return DORY_ECUDA;
    ms[m->prof_cls[i]] += t;
    launches[m->prof_cls[i]] += 1;
  }
  m->prof_used = 0;
  return DORY_OK;
}

const char* dory_strerror(int s) {
  switch (s) {
    case DORY_OK: return "ok";
    case DORY_EINVAL: return "invalid argument";
    case DORY_ENOMEM: return "buffer too small";
    case DORY_ECUDA: return "CUDA call failed";
    case DORY_ECAPACITY: return "batch or context capacity exceeded";
    case DORY_EKMISMATCH: return "per-loop cache needs the bound k and cache mode";
    case DORY_EUNBOUND: return "memory not bound (call dory_bind first)";
    case DORY_EDEVICE: return "device status word set (a bounded wait expired or bad token)";
    case DORY_EUNSUPPORTED: return "configuration not supported by the kernels";
    default: return "unknown status";
  }
}

int dory_device_status(dory_t* m, int* out, void* stream) {
  if (!m || !out) return DORY_EINVAL;
  if (!m->bound) return DORY_EUNBOUND;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, m->ws + m->L.status, sizeof(int), cudaMemcpyDeviceToHost, st) !=
          cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return DORY_ECUDA;
  if (cudaMemsetAsync(m->ws + m->L.status, 0, sizeof(int), st) != cudaSuccess) return DORY_ECUDA;
  *out = v;
  return DORY_OK;
}

int dory_last_launch_count(const dory_t* m, int* out) {
  if (!m || !out) return DORY_EINVAL;
  *out = m->launches;
  return DORY_OK;
}

int dory_debug_hidden(dory_t* m, float* dst, int max_rows, void* stream) {
  if (!m || !dst) return DORY_EINVAL;
  if (!m->bound) return DORY_EUNBOUND;
  const int rows = m->last_rows < max_rows ? m->last_rows : max_rows;
  if (rows <= 0) return DORY_EINVAL;
  return cudaMemcpyAsync(dst, m->ws + (m->hsel_last ? m->L.h32b : m->L.h32),
                         (size_t)rows * m->cfg.d * 4,
                         cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DORY_OK
             : DORY_ECUDA;
}

}  // extern "C"

namespace {
// Test-only: thread 0 waits for phase 0 of an mbarrier that expects one
// arrival and never gets it, through the same bounded wait the TMA and
// tcgen05 kernels use, with a short limit; the wait gives up, writes
// DEV_PROBE_WAIT to the status word and the kernel returns.
__global__ void expire_wait_kernel(unsigned long long limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, status, DEV_PROBE_WAIT, limit_ns);
}
}  // namespace

extern "C" {

int dory_debug_expire_wait(dory_t* m, int limit_us, void* stream) {
  if (!m || limit_us < 1 || limit_us > 100000) return DORY_EINVAL;
  if (!m->bound) return DORY_EUNBOUND;
  expire_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      (unsigned long long)limit_us * 1000ull, wsp<int>(m, m->L.status));
  return cudaGetLastError() == cudaSuccess ? DORY_OK : DORY_ECUDA;
}

int dory_debug_kv_offset(const dory_t* m, int layer, int slice, int which, size_t* offset,
                         int* slots) {
  if (!m || !offset || !slots) return DORY_EINVAL;
  if (!m->bound) return DORY_EUNBOUND;
  const dory_config& c = m->cfg;
  if (layer < 0 || layer >= n_layers(c) || which < 0 || which > 1) return DORY_EINVAL;
  if (slice < 0 || slice >= mult_of(c, layer, m->k_max, m->cache_mode)) return DORY_EINVAL;
  *offset = kv_offset(c, m->max_batch, m->max_ctx, m->k_max, m->cache_mode, layer, slice, which);
  *slots = slots_of(c, layer, m->max_ctx);
  return DORY_OK;
}

int dory_debug_gemm(const void* A, const void* B, float* C, int M, int N, int K, int ldc,
                    void* stream) {
  if (!A || !B || !C || M <= 0 || N <= 0 || K <= 0 || K % 8 || ldc < N) return DORY_EINVAL;
  CUtensorMap ta, tb;
  if (!encode_bf16(&ta, A, M, K, K, 128) || !encode_bf16(&tb, B, N, K, K, kGemmBN / 2))
    return DORY_ECUDA;
  GemmArgs g{};
  g.M = M;
  g.N = N;
  g.K = K;
  g.out = C;
  g.ldo = ldc;
  // output written through a TMA map where its alignment allows, else directly
  EpiMaps eo;
  const bool st_ok = encode_f32_out(&eo.out, C, M, N, ldc);
  return launch_gemm<kGemmBN, EPI_F32>(ta, tb, g, static_cast<cudaStream_t>(stream),
                                       st_ok ? &eo : nullptr);
}

size_t dory_debug_attention_scratch_bytes(int B, int n_q, int head_dim) {
  if (B <= 0 || n_q <= 0 || head_dim <= 0) return 0;
  return align256((size_t)B * n_q * kDecMaxSplits * head_dim * 4) +
         align256((size_t)B * n_q * kDecMaxSplits * 2 * 4) + align256((size_t)B * n_q * 4);
}

int dory_debug_attention(const void* q, const void* k_cur, const void* v_cur, const void* k_cache,
                         const void* v_cache, const void* gate, void* out, int B, int C, int P0,
                         int S, int n_q, int n_kv, int head_dim, int window, float scale,
                         void* scratch, size_t scratch_bytes, void* stream) {
  if (!q || !k_cur || !v_cur || !gate || !out || B <= 0 || C <= 0 || P0 < 0 || n_q <= 0 ||
      n_kv <= 0 || n_q % n_kv || 64 % (n_q / n_kv) || n_q / n_kv > kDecMaxG)
    return DORY_EINVAL;
  if (C == 1 && (!scratch || ((uintptr_t)scratch & 255) ||
                 scratch_bytes < dory_debug_attention_scratch_bytes(B, n_q, head_dim)))
    return DORY_EINVAL;
  if (P0 > 0 && (!k_cache || !v_cache || S <= 0)) return DORY_EINVAL;
  AttnArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k_cur = static_cast<const __nv_bfloat16*>(k_cur);
  a.v_cur = static_cast<const __nv_bfloat16*>(v_cur);
  a.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  a.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
  a.gate = static_cast<const __nv_bfloat16*>(gate);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.C = C;
  a.P0 = P0;
  a.S = S > 0 ? S : 1;
  a.n_q = n_q;
  a.n_kv = n_kv;
  a.window = window > 0 ? window : 0;
  a.scale_log2 = (scale > 0.f ? scale : sqrtf((float)head_dim)) * 1.4426950408889634f;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (C == 1) {
    // the forward pass's one-token kernel (ready inputs, no KV write)
    DecAttnArgs da{};
    da.q = a.q;
    da.k_cur = a.k_cur;
    da.v_cur = a.v_cur;
    da.gate = a.gate;
    da.k_cache = const_cast<__nv_bfloat16*>(a.k_cache);
    da.v_cache = const_cast<__nv_bfloat16*>(a.v_cache);
    da.store = 0;
    da.P0 = P0;
    da.S = a.S;
    da.n_q = n_q;
    da.n_kv = n_kv;
    da.window = a.window;
    da.scale_log2 = a.scale_log2;
    uint8_t* sc = static_cast<uint8_t*>(scratch);
    const size_t o_bytes = align256((size_t)B * n_q * kDecMaxSplits * head_dim * 4);
    const size_t ml_bytes = align256((size_t)B * n_q * kDecMaxSplits * 2 * 4);
    da.part_o = reinterpret_cast<float*>(sc);
    da.part_ml = reinterpret_cast<float*>(sc + o_bytes);
    da.counter = reinterpret_cast<int*>(sc + o_bytes + ml_bytes);
    da.out = a.out;
    da.cache_rows = P0 > 0 ? (long long)B * n_kv * a.S : 0;
    if (cudaMemsetAsync(da.counter, 0, (size_t)B * n_kv * 4, st) != cudaSuccess) return DORY_ECUDA;
    return dec_attn<false>(da, B, head_dim, st);
  }
  if (g_debug_tc_attn) {
    const int rc = launch_attn_tc(a, B, head_dim, (long long)B * n_kv * a.S, nullptr, st);
    if (rc != DORY_EUNSUPPORTED) return rc;
  }
  if (scratch && !((uintptr_t)scratch & 255)) {
    // key-range splits of the mma.sync kernel, with partials in the scratch
    const size_t per = (size_t)B * C * n_q * (head_dim + 2) * 4;   // bytes per split
    const size_t cap = scratch_bytes / (per + 512);
    if (cap >= 2) {
      a.part_cap = cap > kDecMaxSplits ? kDecMaxSplits : (int)cap;
      uint8_t* sc = static_cast<uint8_t*>(scratch);
      a.part_o = reinterpret_cast<float*>(sc);
      a.part_ml = reinterpret_cast<float*>(
          sc + align256((size_t)B * C * n_q * a.part_cap * head_dim * 4));
    }
  }
  if (head_dim == 32) return launch_attn<32>(a, B, st);
  if (head_dim == 64) return launch_attn<64>(a, B, st);
  if (head_dim == 128) return launch_attn<128>(a, B, st);
  return DORY_EUNSUPPORTED;
}

int dory_set_fused_ngpt(dory_t* m, int enable) {
  if (!m || (enable != 0 && enable != 1)) return DORY_EINVAL;
  m->use_ngpt_fused = enable != 0;
  return DORY_OK;
}

int dory_set_tc_attention(dory_t* m, int enable) {
  if (enable != 0 && enable != 1) return DORY_EINVAL;
  if (m)
    m->use_tc_attn = enable != 0;
  else
    g_debug_tc_attn = enable != 0;
  return DORY_OK;
}

}  // extern "C"

// ------------------------------------------------------------------------
// Decode attention without caller scratch: the split-key partials go to a
// fixed array in device memory that the library owns for the process's life.
// ------------------------------------------------------------------------
static constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;   // 16 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
// Device address of the array in the current device's context.  Host code
// cannot use the symbol itself as a device pointer.  The address is looked up
// on every call (a host-side table lookup once the module is loaded), so a
// context torn down and created again never leaves a stale pointer behind.
int noalloc_scratch(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return DORY_ECUDA;
  *out = p;
  return DORY_OK;
}

bool aligned_to(const void* p, uintptr_t bytes) {
  return (reinterpret_cast<uintptr_t>(p) & (bytes - 1)) == 0;
}
}  // namespace

extern "C" int dory_decode_attention_noalloc(const void* q, const void* k_cur, const void* v_cur,
                                             const void* k_cache, const void* v_cache,
                                             const void* gate, void* out, int B, int P0, int S,
                                             int n_q, int n_kv, int head_dim, int window,
                                             float scale, void* stream) {
  if (!q || !k_cur || !v_cur || !gate || !out || B <= 0 || P0 < 0 || n_q <= 0 || n_kv <= 0 ||
      n_q % n_kv || n_q / n_kv > kDecMaxG)
    return DORY_EINVAL;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128) return DORY_EUNSUPPORTED;
  if (P0 > 0 && (!k_cache || !v_cache || S <= 0)) return DORY_EINVAL;
  // keys and values are read as 16-byte vectors, q, gate and out as bf16
  if (!aligned_to(k_cur, 16) || !aligned_to(v_cur, 16) || !aligned_to(q, 2) ||
      !aligned_to(gate, 2) || !aligned_to(out, 2))
    return DORY_EINVAL;
  if (P0 > 0 && (!aligned_to(k_cache, 16) || !aligned_to(v_cache, 16))) return DORY_EINVAL;
  // the ring must still hold every cached key the mask shows: P0 of them
  // under full attention, min(P0, window - 1) under a window
  if (P0 > 0 && S < (window > 0 ? (P0 < window - 1 ? P0 : window - 1) : P0)) return DORY_EINVAL;
  const size_t need = dory_debug_attention_scratch_bytes(B, n_q, head_dim);
  if (need == 0 || need > kNoAllocScratchBytes) return DORY_ECAPACITY;
  void* scratch = nullptr;
  const int rc = noalloc_scratch(&scratch);
  if (rc != DORY_OK) return rc;
  DecodeArgs da{};
  da.q = static_cast<const __nv_bfloat16*>(q);
  da.k_cur = static_cast<const __nv_bfloat16*>(k_cur);
  da.v_cur = static_cast<const __nv_bfloat16*>(v_cur);
  da.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  da.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
  da.P0 = P0;
  da.S = S > 0 ? S : 1;
  da.n_q = n_q;
  da.n_kv = n_kv;
  da.window = window > 0 ? window : 0;
  da.scale_log2 = (scale > 0.f ? scale : sqrtf((float)head_dim)) * 1.4426950408889634f;
  // every split writes the partials the combine step reads: nothing to clear
  da.part_o = static_cast<float*>(scratch);
  da.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) +
                                        align256((size_t)B * n_q * kDecMaxSplits * head_dim * 4));
  const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(gate);
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (head_dim == 32) return launch_decode_attn<32>(da, B, g, o, st);
  if (head_dim == 64) return launch_decode_attn<64>(da, B, g, o, st);
  return launch_decode_attn<128>(da, B, g, o, st);
}
