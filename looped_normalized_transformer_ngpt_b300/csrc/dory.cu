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
#include "gemm_tc.cuh"
#include "gemv.cuh"
#include "rowops.cuh"

using namespace dory;

namespace {

constexpr int kGemmBN = 256;

struct WsLayout {
  size_t status, h32, x32, hb, y32, q, k, v, g, att, m, rope_swa, rope_full, gy, dec_o, dec_ml,
      total;
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
  L.x32 = take(M * c.d * 4);
  L.hb = take(M * c.d * 2);
  L.y32 = take(M * c.d * 4);
  L.q = take(M * hq * 2);
  L.k = take(M * hk * 2);
  L.v = take(M * hk * 2);
  L.g = take(M * hq * 2);
  L.att = take(M * hq * 2);
  L.m = take(M * (size_t)c.ffn * 2);
  L.rope_swa = take((size_t)max_chunk * (c.head_dim / 2) * 8);
  L.rope_full = take((size_t)max_chunk * (c.head_dim / 2) * 8);
  // few-row projections (decode): fp32 output of the QKV+gate / up+gate GEMV
  const size_t nq = (size_t)(2 * c.n_q + 2 * c.n_kv) * c.head_dim;
  const size_t wide = nq > 2 * (size_t)c.ffn ? nq : 2 * (size_t)c.ffn;
  L.gy = take((size_t)kGemvMaxM * wide * 4);
  // split-KV decode attention partials
  L.dec_o = take((size_t)max_batch * c.n_q * kDecMaxSplits * c.head_dim * 4);
  L.dec_ml = take((size_t)max_batch * c.n_q * kDecMaxSplits * 2 * 4);
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
int launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, GemmArgs args, cudaStream_t st) {
  static bool attr = false;
  using Cf = GemmCfg<BN>;
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
  const int tiles = args.tiles_m * args.tiles_n;
  if (tiles == 0) return DORY_OK;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  return launch_k(gemm_tc_kernel<BN, EPI>, dim3(grid), dim3(192), Cf::SMEM, st, ta, tb, args) ==
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
  dim3 grid((a.C + BQ - 1) / BQ, a.n_kv, B);
  return launch_k(attn_prefill_kernel<DH>, grid, dim3(128), AttnCfg<DH>::SMEM, st, a) ==
                 cudaSuccess
             ? DORY_OK
             : DORY_ECUDA;
}

// Y[M, N] (row stride ldy) = scale * X[M, K] . W[N, K]^T for M <= kGemvMaxM, or,
// with pair_off > 0, m_out[M, N] = (X W[n]^T) * SiLU(X W[n + pair_off]^T).
template <int MM, int J, bool SW>
cudaError_t gemv_go(int grid, cudaStream_t st, const __nv_bfloat16* X, int ldx, int M,
                    const __nv_bfloat16* W, int N, int K, int S, float* Y, int ldy,
                    const float* scale, int pair_off, __nv_bfloat16* m_out, int ldm) {
  return launch_k(gemv_kernel<MM, J, SW>, dim3(grid), dim3(kGemvThreads), 0, st, X, ldx, M, W, N,
                  K, S, Y, ldy, scale, pair_off, m_out, ldm);
}

template <int MM, bool SW>
cudaError_t gemv_j(int J, int grid, cudaStream_t st, const __nv_bfloat16* X, int ldx, int M,
                   const __nv_bfloat16* W, int N, int K, int S, float* Y, int ldy,
                   const float* scale, int pair_off, __nv_bfloat16* m_out, int ldm) {
  if (J <= 2) return gemv_go<MM, 2, SW>(grid, st, X, ldx, M, W, N, K, S, Y, ldy, scale, pair_off, m_out, ldm);
  if (J <= 4) return gemv_go<MM, 4, SW>(grid, st, X, ldx, M, W, N, K, S, Y, ldy, scale, pair_off, m_out, ldm);
  if (SW) return cudaErrorInvalidValue;
  if (J <= 6) return gemv_go<MM, 6, false>(grid, st, X, ldx, M, W, N, K, S, Y, ldy, scale, pair_off, m_out, ldm);
  return gemv_go<MM, 8, false>(grid, st, X, ldx, M, W, N, K, S, Y, ldy, scale, pair_off, m_out, ldm);
}

int launch_gemv(const __nv_bfloat16* X, int ldx, int M, const void* W, int N, int K, float* Y,
                int ldy, const float* scale, cudaStream_t st, int pair_off = 0,
                __nv_bfloat16* m_out = nullptr, int ldm = 0) {
  const bool sw = pair_off > 0;
  const int jmax = sw ? 4 : 8;
  const int kc = (K + 255) / 256;                  // 256-element chunks per row
  int S = 1;
  while ((kc + S - 1) / S > jmax && S < kGemvWarps) S *= 2;
  const int J = (kc + S - 1) / S;
  if (J > jmax || M > kGemvMaxM) return DORY_EUNSUPPORTED;
  const int rows_per_cta = kGemvWarps / S;
  const int grid = (N + rows_per_cta - 1) / rows_per_cta;
  const __nv_bfloat16* w = static_cast<const __nv_bfloat16*>(W);
  cudaError_t e;
  if (M <= 4)
    e = sw ? gemv_j<4, true>(J, grid, st, X, ldx, M, w, N, K, S, Y, ldy, scale, pair_off, m_out, ldm)
           : gemv_j<4, false>(J, grid, st, X, ldx, M, w, N, K, S, Y, ldy, scale, 0, m_out, ldm);
  else
    e = sw ? gemv_j<16, true>(J, grid, st, X, ldx, M, w, N, K, S, Y, ldy, scale, pair_off, m_out, ldm)
           : gemv_j<16, false>(J, grid, st, X, ldx, M, w, N, K, S, Y, ldy, scale, 0, m_out, ldm);
  return e == cudaSuccess ? DORY_OK : DORY_ECUDA;
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
  int batch = 0;       // batch of the current sequences (0 = none yet)
  int last_rows = 0;   // rows of the last processed chunk (B * C)
  int launches = 0;
  // optional per-launch event timing
  bool prof_on = false;
  int prof_used = 0;
  std::vector<cudaEvent_t> prof_ev;   // 2 per launch
  std::vector<int> prof_cls;
};

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

int ngpt_update(dory_model* m, int M, const float* alpha, cudaStream_t st) {
  return launch_k(ngpt_update_kernel, dim3(M), dim3(kRowThreads), 0, st, wsp<float>(m, m->L.h32),
                  wsp<__nv_bfloat16>(m, m->L.hb), (const float*)wsp<float>(m, m->L.y32), alpha,
                  m->cfg.d) == cudaSuccess
             ? DORY_OK
             : DORY_ECUDA;
}

int run_layer(dory_model* m, int l, int slice, bool store, int B, int C, int P0,
              const CUtensorMap& tm_hb, const CUtensorMap& tm_att, const CUtensorMap& tm_m,
              cudaStream_t st) {
  const dory_config& c = m->cfg;
  const dory_layer_weights& w = m->layers[l];
  const int M = B * C;
  const int hq = c.n_q * c.head_dim;
  int* status = wsp<int>(m, m->L.status);
  const bool full = layer_full(c, l);

  // QKV + gate projection with RoPE / q-k normalisation / sigmoid fused
  GemmArgs ga{};
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
  ga.rows_per_seq = C;
  const bool few = M <= kGemvMaxM;
  __nv_bfloat16* hb = wsp<__nv_bfloat16>(m, m->L.hb);
  float* gy = wsp<float>(m, m->L.gy);
  if (few) {
    pb(m, DORY_K_QKVG_GEMM, st);
    DORY_TRY(pe(m, st, launch_gemv(hb, c.d, M, w.w_qkvg, ga.N, c.d, gy, ga.N, nullptr, st)));
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
    DORY_TRY(pe(m, st, launch_gemm<kGemmBN, EPI_QKVG>(tm_hb, m->tm_qkvg[l], ga, st)));
  }

  // attention over cached + current keys
  const int S = slots_of(c, l, m->max_ctx);
  const size_t koff = kv_offset(c, m->max_batch, m->max_ctx, m->k_max, m->cache_mode, l, slice, 0);
  const size_t voff = kv_offset(c, m->max_batch, m->max_ctx, m->k_max, m->cache_mode, l, slice, 1);
  __nv_bfloat16* kc = reinterpret_cast<__nv_bfloat16*>(m->kv + koff);
  __nv_bfloat16* vc = reinterpret_cast<__nv_bfloat16*>(m->kv + voff);
  AttnArgs aa{};
  aa.q = ga.q;
  aa.k_cur = ga.k;
  aa.v_cur = ga.v;
  aa.k_cache = kc;
  aa.v_cache = vc;
  aa.gate = ga.g;
  aa.out = wsp<__nv_bfloat16>(m, m->L.att);
  aa.C = C;
  aa.P0 = P0;
  aa.S = S;
  aa.n_q = c.n_q;
  aa.n_kv = c.n_kv;
  aa.window = full ? 0 : c.window;
  const float scale = c.softmax_scale > 0.f ? c.softmax_scale : sqrtf((float)c.head_dim);
  aa.scale_log2 = scale * 1.4426950408889634f;
  pb(m, DORY_K_ATTENTION, st);
  int arc = DORY_EUNSUPPORTED;
  if (C == 1) {
    DecodeArgs da{};
    da.q = aa.q;
    da.k_cur = aa.k_cur;
    da.v_cur = aa.v_cur;
    da.k_cache = aa.k_cache;
    da.v_cache = aa.v_cache;
    da.P0 = P0;
    da.S = S;
    da.n_q = c.n_q;
    da.n_kv = c.n_kv;
    da.window = aa.window;
    da.scale_log2 = aa.scale_log2;
    da.part_o = wsp<float>(m, m->L.dec_o);
    da.part_ml = wsp<float>(m, m->L.dec_ml);
    if (c.head_dim == 32) arc = launch_decode_attn<32>(da, B, aa.gate, aa.out, st);
    if (c.head_dim == 64) arc = launch_decode_attn<64>(da, B, aa.gate, aa.out, st);
    if (c.head_dim == 128) arc = launch_decode_attn<128>(da, B, aa.gate, aa.out, st);
  } else {
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

  // output projection + nGPT step
  GemmArgs go{};
  go.M = M;
  go.N = c.d;
  go.K = hq;
  go.status = status;
  go.out = wsp<float>(m, m->L.y32);
  go.ldo = c.d;
  pb(m, DORY_K_O_GEMM, st);
  if (few)
    DORY_TRY(pe(m, st, launch_gemv(aa.out, hq, M, w.w_o, c.d, hq, go.out, c.d, nullptr, st)));
  else
    DORY_TRY(pe(m, st, launch_gemm<kGemmBN, EPI_F32>(tm_att, m->tm_o[l], go, st)));
  pb(m, DORY_K_NGPT_UPDATE, st);
  DORY_TRY(pe(m, st, ngpt_update(m, M, w.alpha_attn, st)));

  // SwiGLU MLP + nGPT step
  GemmArgs gu{};
  gu.M = M;
  gu.N = 2 * c.ffn;
  gu.K = c.d;
  gu.b_second = c.ffn;
  gu.status = status;
  gu.m_out = wsp<__nv_bfloat16>(m, m->L.m);
  gu.ldm = c.ffn;
  if (few) {
    pb(m, DORY_K_UPGATE_GEMM, st);
    DORY_TRY(pe(m, st, launch_gemv(hb, c.d, M, w.w_upgate, c.ffn, c.d, nullptr, 0, nullptr, st,
                                   c.ffn, gu.m_out, c.ffn)));
  } else {
    pb(m, DORY_K_UPGATE_GEMM, st);
    DORY_TRY(pe(m, st, launch_gemm<kGemmBN, EPI_SWIGLU>(tm_hb, m->tm_upgate[l], gu, st)));
  }
  GemmArgs gd{};
  gd.M = M;
  gd.N = c.d;
  gd.K = c.ffn;
  gd.status = status;
  gd.out = wsp<float>(m, m->L.y32);
  gd.ldo = c.d;
  pb(m, DORY_K_DOWN_GEMM, st);
  if (few)
    DORY_TRY(pe(m, st, launch_gemv(gu.m_out, c.ffn, M, w.w_down, c.d, c.ffn, gd.out, c.d, nullptr,
                                   st)));
  else
    DORY_TRY(pe(m, st, launch_gemm<kGemmBN, EPI_F32>(tm_m, m->tm_down[l], gd, st)));
  pb(m, DORY_K_NGPT_UPDATE, st);
  return pe(m, st, ngpt_update(m, M, w.alpha_mlp, st));
}

int boundary(dory_model* m, int M, int mode, cudaStream_t st) {
  pb(m, DORY_K_BOUNDARY, st);
  return pe(m, st,
            launch_k(boundary_kernel, dim3(M), dim3(kRowThreads), 0, st, wsp<float>(m, m->L.h32),
                     wsp<__nv_bfloat16>(m, m->L.hb), wsp<float>(m, m->L.x32), m->cfg.d, mode) ==
                    cudaSuccess
                ? DORY_OK
                : DORY_ECUDA);
}

// One forward step over B sequences x C tokens at positions P0 .. P0+C-1.
// Logit rows: if logits != null, rows (b, t) for t >= C - n_logit_rows are
// written to logits + (b * ld_seq + t_out0 + t - (C - n_logit_rows)) * V.
int run_step(dory_model* m, const int32_t* tokens, int ld_tok, int B, int C, int k,
             float* logits, long long ld_seq, int t_out0, int n_logit_rows, cudaStream_t st) {
  const dory_config& c = m->cfg;
  const int M = B * C;
  const int P0 = m->len;
  int* status = wsp<int>(m, m->L.status);

  CUtensorMap tm_hb, tm_att, tm_m;
  const int hq = c.n_q * c.head_dim;
  if (!encode_bf16(&tm_hb, m->ws + m->L.hb, M, c.d, c.d, 128) ||
      !encode_bf16(&tm_att, m->ws + m->L.att, M, hq, hq, 128) ||
      !encode_bf16(&tm_m, m->ws + m->L.m, M, c.ffn, c.ffn, 128))
    return DORY_ECUDA;

  if (c.rope) {
    const int n = C * (c.head_dim / 2);
    const int blocks = (n + 255) / 256;
    pb(m, DORY_K_ROPE, st);
    DORY_TRY(pe(m, st,
                launch_k(rope_table_kernel, dim3(blocks), dim3(256), 0, st,
                         wsp<float2>(m, m->L.rope_swa), C, P0, c.head_dim,
                         (double)c.rope_base_swa) == cudaSuccess
                    ? DORY_OK
                    : DORY_ECUDA));
    pb(m, DORY_K_ROPE, st);
    DORY_TRY(pe(m, st,
                launch_k(rope_table_kernel, dim3(blocks), dim3(256), 0, st,
                         wsp<float2>(m, m->L.rope_full), C, P0, c.head_dim,
                         (double)c.rope_base_full) == cudaSuccess
                    ? DORY_OK
                    : DORY_ECUDA));
  }
  pb(m, DORY_K_EMBED, st);
  DORY_TRY(pe(m, st,
              launch_k(embed_kernel, dim3(M), dim3(kRowThreads), 0, st, tokens, ld_tok, C,
                       reinterpret_cast<const __nv_bfloat16*>(m->embed_in), c.vocab, c.d,
                       wsp<float>(m, m->L.h32), wsp<__nv_bfloat16>(m, m->L.hb), status) ==
                      cudaSuccess
                  ? DORY_OK
                  : DORY_ECUDA));

  for (int l = 0; l < c.n_in; ++l)
    DORY_TRY(run_layer(m, l, 0, true, B, C, P0, tm_hb, tm_att, tm_m, st));
  if (c.n_rec > 0) {
    DORY_TRY(boundary(m, M, BND_SAVE_X, st));
    for (int i = 1; i <= k; ++i) {
      DORY_TRY(boundary(m, M, i == 1 ? BND_ENTER_FIRST : BND_ENTER_NEXT, st));
      const bool per_loop = m->cache_mode == DORY_CACHE_PER_LOOP;
      const int slice = per_loop ? i - 1 : 0;
      const bool store = per_loop || i == k;
      for (int l = c.n_in; l < c.n_in + c.n_rec; ++l)
        DORY_TRY(run_layer(m, l, slice, store, B, C, P0, tm_hb, tm_att, tm_m, st));
    }
    DORY_TRY(boundary(m, M, BND_EXIT, st));
  }
  for (int l = c.n_in + c.n_rec; l < n_layers(c); ++l)
    DORY_TRY(run_layer(m, l, 0, true, B, C, P0, tm_hb, tm_att, tm_m, st));

  if (logits && n_logit_rows > 0) {
    // LM head on the selected rows: per sequence, rows C - n .. C-1 of hb
    const int first = C - n_logit_rows;
    GemmArgs gl{};
    gl.N = c.vocab;
    gl.K = c.d;
    gl.status = status;
    gl.col_scale = m->s_z;
    gl.ldo = c.vocab;
    if (n_logit_rows == 1 && B <= kGemvMaxM) {
      pb(m, DORY_K_LM_HEAD, st);
      DORY_TRY(pe(m, st, launch_gemv(wsp<__nv_bfloat16>(m, m->L.hb) + (size_t)(C - 1) * c.d,
                                     C * c.d, B, m->embed_out, c.vocab, c.d,
                                     logits + (long long)t_out0 * c.vocab,
                                     (int)(ld_seq * c.vocab), m->s_z, st)));
    } else if (n_logit_rows == 1) {
      // one row per sequence: a strided view of hb (row stride C * d)
      CUtensorMap tm_last;
      if (!encode_bf16(&tm_last, m->ws + m->L.hb + (size_t)(C - 1) * c.d * 2, B, c.d,
                       (uint64_t)C * c.d, 128))
        return DORY_ECUDA;
      gl.M = B;
      gl.ldo = ld_seq * c.vocab;
      gl.out = logits + (long long)t_out0 * c.vocab;
      pb(m, DORY_K_LM_HEAD, st);
      DORY_TRY(pe(m, st, launch_gemm<kGemmBN, EPI_F32>(tm_last, m->tm_embed_out, gl, st)));
    } else {
      for (int b = 0; b < B; ++b) {
        CUtensorMap tm_rows;
        if (!encode_bf16(&tm_rows, m->ws + m->L.hb + ((size_t)b * C + first) * c.d * 2,
                         n_logit_rows, c.d, c.d, 128))
          return DORY_ECUDA;
        gl.M = n_logit_rows;
        gl.out = logits + ((long long)b * ld_seq + t_out0) * c.vocab;
        pb(m, DORY_K_LM_HEAD, st);
        DORY_TRY(pe(m, st, launch_gemm<kGemmBN, EPI_F32>(tm_rows, m->tm_embed_out, gl, st)));
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
  if (cudaMemsetAsync(m->ws + m->L.status, 0, 256, 0) != cudaSuccess) return DORY_ECUDA;
  return DORY_OK;
}

int dory_prefill(dory_t* m, const int32_t* tokens, int B, int T, int k, int cache_mode,
                 float* logits, int all_logits, void* stream) {
  const int rc = check_call(m, B, T, k, cache_mode);
  if (rc != DORY_OK) return rc;
  if (!tokens) return DORY_EINVAL;
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

int dory_decode_step(dory_t* m, const int32_t* tokens, int B, int k, int cache_mode,
                     float* logits, int32_t* next, void* stream) {
  const int rc = check_call(m, B, 1, k, cache_mode);
  if (rc != DORY_OK) return rc;
  if (!tokens) return DORY_EINVAL;
  if (next && !logits) return DORY_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  m->launches = 0;
  m->batch = B;
  const int r = run_step(m, tokens, 1, B, 1, k, logits, 1, 0, logits ? 1 : 0, st);
  if (r != DORY_OK) return r;
  if (next) {
    pb(m, DORY_K_ARGMAX, st);
    return pe(m, st,
              launch_k(argmax_kernel, dim3(B), dim3(1024), 0, st, (const float*)logits,
                       m->cfg.vocab, next) == cudaSuccess
                  ? DORY_OK
                  : DORY_ECUDA);
  }
  return DORY_OK;
}

int dory_length(const dory_t* m, int* out) {
  if (!m || !out) return DORY_EINVAL;
  *out = m->len;
  return DORY_OK;
}

int dory_reset(dory_t* m) {
  if (!m) return DORY_EINVAL;
  m->len = 0;
  m->batch = 0;
  m->last_rows = 0;
  return DORY_OK;
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
  return cudaMemcpyAsync(dst, m->ws + m->L.h32, (size_t)rows * m->cfg.d * 4,
                         cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DORY_OK
             : DORY_ECUDA;
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
  return launch_gemm<kGemmBN, EPI_F32>(ta, tb, g, static_cast<cudaStream_t>(stream));
}

size_t dory_debug_attention_scratch_bytes(int B, int n_q, int head_dim) {
  if (B <= 0 || n_q <= 0 || head_dim <= 0) return 0;
  return align256((size_t)B * n_q * kDecMaxSplits * head_dim * 4) +
         align256((size_t)B * n_q * kDecMaxSplits * 2 * 4);
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
    DecodeArgs da{};
    da.q = a.q;
    da.k_cur = a.k_cur;
    da.v_cur = a.v_cur;
    da.k_cache = a.k_cache;
    da.v_cache = a.v_cache;
    da.P0 = P0;
    da.S = a.S;
    da.n_q = n_q;
    da.n_kv = n_kv;
    da.window = a.window;
    da.scale_log2 = a.scale_log2;
    da.part_o = static_cast<float*>(scratch);
    da.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) +
                                          align256((size_t)B * n_q * kDecMaxSplits * head_dim * 4));
    if (head_dim == 32) return launch_decode_attn<32>(da, B, a.gate, a.out, st);
    if (head_dim == 64) return launch_decode_attn<64>(da, B, a.gate, a.out, st);
    if (head_dim == 128) return launch_decode_attn<128>(da, B, a.gate, a.out, st);
    return DORY_EUNSUPPORTED;
  }
  if (head_dim == 32) return launch_attn<32>(a, B, st);
  if (head_dim == 64) return launch_attn<64>(a, B, st);
  if (head_dim == 128) return launch_attn<128>(a, B, st);
  return DORY_EUNSUPPORTED;
}

}  // extern "C"

// ------------------------------------------------------------------------
// Decode attention without caller scratch: the split-key partials go to a
// fixed array in device memory that the library owns for the process's life.
// ------------------------------------------------------------------------
static constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;   // 16 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kNoAllocMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device (host code cannot use the symbol itself as a device pointer).
int noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices)
    return DORY_ECUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return DORY_ECUDA;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return DORY_OK;
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
