/*
 * dory.h - C ABI of the looped normalized-GPT forward pass on one B300 GPU.
 *
 * The operation is the inference forward pass of the looped nGPT described in
 * "Dory1.0-4B: A Looped Normalized-GPT":
 *   - Architecture: every hidden state lives on the unit sphere and each
 *     sublayer moves it with the nGPT residual step
 *         h <- N(h + alpha * (N(y) - h)),   N(v) = v / ||v||_2 per token;
 *     grouped-query attention with an input-dependent sigmoid output gate,
 *     per-head L2-normalised queries and keys, the gated concatenated output
 *     normalised before the output projection, a SwiGLU MLP whose activation
 *     is normalised before the down projection, and a 3:1 interleave of
 *     sliding-window and full causal attention layers.
 *   - Training with Loops: an input block runs once, a shared recurrent
 *     block runs k times, an output block runs once.  With x the input
 *     block's output, s_0 = x and s_i = N(F(N(s_{i-1} + x))); the output
 *     block receives s_k.  No adapter weights, no outer residual.
 *   - Long-Context Extension: rotary positions, base 1e4 on sliding-window
 *     layers and 1e7 on full layers.
 *   - Last-Loop KV Caching: a per-loop cache keeps one K/V slice per loop for
 *     each recurrent layer (a loop-i query sees loop-i keys of earlier
 *     tokens); a last-loop cache keeps one slice whose entries are those of
 *     the final loop.  Tokens of the current call are always seen with their
 *     current-loop keys and values.  Input and output layers keep one slice.
 *
 * Readings fixed where the paper is silent: layer i uses full attention iff
 * i % full_every == full_offset; the window W counts the query itself (key j
 * visible from query t iff j <= t and t - j < W); RoPE is rotate-half over the
 * whole head, applied before the q/k normalisation, then q and k are scaled
 * by s_qk; softmax scale sqrt(head_dim) unless set; the gate is elementwise
 * over the n_q * head_dim attention output; m = (W_up h) * SiLU(W_sl h);
 * logits = s_z * (E_out h); greedy decoding picks the lowest index among
 * equal maxima.
 *
 * Conventions
 *   - All pointers named "device" are CUDA device pointers on the current
 *     device.  The library never allocates device memory and never owns the
 *     weights, the KV cache or the workspace: the caller allocates them (sizes
 *     from dory_kv_bytes / dory_workspace_bytes) and keeps them alive while
 *     the handle uses them.
 *   - Every compute call is asynchronous on the caller's stream (a
 *     cudaStream_t passed as void*; NULL = legacy default stream) and makes no
 *     host/device synchronisation, so calls may be captured in a CUDA graph.
 *   - Argument, capacity and state errors are detected on the host before any
 *     launch and returned as a negative dory_status; the handle is unchanged.
 *     Device-side failures (a bounded wait that expired) set a status word
 *     that dory_device_status reads.  No call aborts or throws.
 *   - All sequences of one call share the same current length (they are
 *     prefilled and decoded together), except in the ragged-batch calls
 *     (dory_prefill_slot, dory_decode_step_ragged) below.
 */
#ifndef DORY_H
#define DORY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DORY_OK = 0,
    DORY_EINVAL = -1,       /* bad argument (null pointer, bad size, bad config) */
    DORY_ENOMEM = -2,       /* a caller buffer is smaller than required */
    DORY_ECUDA = -3,        /* a CUDA runtime/driver call failed */
    DORY_ECAPACITY = -4,    /* batch > max_batch, or length would exceed max_ctx */
    DORY_EKMISMATCH = -5,   /* per-loop cache used with a k other than the bound one,
                               or a cache mode other than the bound one */
    DORY_EUNBOUND = -6,     /* compute call before dory_bind */
    DORY_EDEVICE = -7,      /* device status word set (bounded wait expired) */
    DORY_EUNSUPPORTED = -8  /* config outside what the kernels implement */
} dory_status;

typedef enum { DORY_CACHE_LAST_LOOP = 0, DORY_CACHE_PER_LOOP = 1 } dory_cache_mode;

/* Model dimensions.  Supported: head_dim in {32, 64, 128}; d, ffn multiples
 * of 128; n_q a multiple of n_kv; vocab a multiple of 16. */
typedef struct {
    int d, n_in, n_rec, n_out;   /* model width; layers in input/recurrent/output blocks */
    int n_q, n_kv, head_dim;     /* query heads, kv heads, head width */
    int ffn, vocab, window;      /* SwiGLU width, vocabulary, sliding window W */
    int full_every, full_offset; /* layer i full-attention iff i % full_every == full_offset */
    int rope;                    /* 1 = rotary positions on, 0 = off */
    float rope_base_swa, rope_base_full;
    float softmax_scale;         /* <= 0 selects sqrt(head_dim) */
} dory_config;

/* One layer.  Matrices are bf16, row-major [out, in], device. */
typedef struct {
    const void* w_qkvg;       /* [(2 n_q + 2 n_kv) head_dim, d]: rows W_q | W_k | W_v | W_g */
    const void* w_o;          /* [d, n_q head_dim] */
    const void* w_upgate;     /* [2 ffn, d]: rows W_up | W_sl (W_sl feeds the SiLU) */
    const void* w_down;       /* [d, ffn] */
    const float* alpha_attn;  /* [d] effective residual rate of the attention step */
    const float* alpha_mlp;   /* [d] effective residual rate of the MLP step */
    const float* s_qk;        /* [head_dim] query/key scale */
} dory_layer_weights;

typedef struct {
    const void* embed_in;     /* bf16 [vocab, d], device */
    const void* embed_out;    /* bf16 [vocab, d], device */
    const float* s_z;         /* [vocab] logit scale, device; NULL means 1 */
    const dory_layer_weights* layers; /* HOST array of n_in + n_rec + n_out entries (copied) */
} dory_weights;

typedef struct dory_model dory_t;

#if defined(__GNUC__)
#define DORY_API __attribute__((visibility("default")))
#else
#define DORY_API
#endif

/* Validates the config, copies the pointer tables.  No CUDA call is made.
 * On success *out receives a handle to release with dory_destroy. */
DORY_API int dory_create(const dory_config* cfg, const dory_weights* w, dory_t** out);

/* Bytes of the KV region for max_batch sequences of up to max_ctx positions,
 * k loops and the given cache mode (pure host function):
 *   2 (K,V) * n_kv * head_dim * 2 B * max_batch *
 *   sum over layers l of mult_l * slots_l,
 * slots_l = max_ctx on full layers and min(max_ctx, window) on sliding-window
 * layers (a ring: position p lives in slot p mod slots_l); mult_l = k for
 * recurrent layers in per-loop mode, else 1.  Returns 0 on bad arguments.
 * Layout: for l = 0..L-1, for slice = 0..mult_l-1: K then V, each
 * [max_batch][n_kv][slots_l][head_dim] bf16. */
DORY_API size_t dory_kv_bytes(const dory_config* cfg, int max_batch, int max_ctx, int k, int cache_mode);

/* Bytes of scratch for calls of up to max_batch sequences x max_chunk tokens
 * (pure host function).  Returns 0 on bad arguments. */
DORY_API size_t dory_workspace_bytes(const dory_config* cfg, int max_batch, int max_chunk);

/* Attaches caller memory (device, 256-byte aligned) and capacities to the
 * handle and resets every sequence to length 0.  kv_bytes must be at least
 * dory_kv_bytes(cfg, max_batch, max_ctx, k_max, cache_mode) and ws_bytes at
 * least dory_workspace_bytes(cfg, max_batch, max_chunk).  In per-loop mode
 * every later call must use cache_mode and the same k (<= k_max). */
DORY_API int dory_bind(dory_t* m, void* kv, size_t kv_bytes, void* ws, size_t ws_bytes,
              int max_batch, int max_ctx, int max_chunk, int k_max, int cache_mode);

/* Prefill: appends T tokens to each of B sequences (all at the same current
 * length P0) and runs the forward at loop count k.  tokens: device int32
 * [B, T].  Prompts longer than max_chunk are processed in chunks of max_chunk
 * tokens (chunked prefill).  logits: device fp32, [B, vocab] for the last
 * position of each sequence, or [B, T, vocab] when all_logits != 0; may be
 * NULL.  Requires B <= max_batch and P0 + T <= max_ctx. */
DORY_API int dory_prefill(dory_t* m, const int32_t* tokens, int B, int T, int k, int cache_mode,
                 float* logits, int all_logits, void* stream);

/* Decode: appends one token to each of B sequences at the current length and
 * runs the forward at loop count k.  tokens: device int32 [B].  logits:
 * device fp32 [B, vocab] or NULL; next: device int32 [B] greedy tokens or
 * NULL (requires logits).
 * Decode steps of up to 128 sequences run the tensor-core projections with
 * the weights as the 128-row operand and K split over the SMs (on B300 this
 * streams the weights faster than a GEMV, from one sequence up); a single
 * sequence with quantised weights runs five kernels per layer application
 * instead (GEMVs streaming the packed codes, one attention kernel); larger
 * batches run the prefill GEMMs.  With
 * head_dim 128 and ring sizes that are multiples of 64 (max_ctx and window,
 * as given to dory_bind / dory_create) the attention streams the cached K/V
 * with TMA through a 4-stage ring; otherwise a cp.async kernel does (same
 * results up to rounding order, slower on long contexts). */
DORY_API int dory_decode_step(dory_t* m, const int32_t* tokens, int B, int k, int cache_mode,
                     float* logits, int32_t* next, void* stream);

/* ---- self-speculative decoding ---------------------------------------- */

/* One greedy self-speculative decoding step ("Dory1.0-4B: A Looped
 * Normalized-GPT", Self-Speculative Decoding): the same weights draft gamma
 * tokens, one decode step at a time at loop count k_draft, then verify them
 * in one forward pass at k_verify over the last emitted token and the
 * drafts; drafts are accepted while each equals the verifier's greedy token
 * at the position before it, and the verifier's token after the last
 * accepted draft is emitted as well.  The emitted tokens are those of plain
 * greedy decoding at k_verify.
 *   Per-loop caching bound with k_max == k_verify is required
 * (DORY_EKMISMATCH otherwise): drafting reads and writes the slices of loops
 * 1..k_draft, which the verifier shares, and the verifier rewrites every
 * slice of the positions it processes.  The sliding-window ring slots that
 * drafting and the rejected positions overwrite are saved and put back.
 *   tokens: device int32 [B], the last emitted token of each sequence (not
 * yet in the cache).  out: device int32 [B, gamma + 1]; row b receives the
 * emitted tokens in its first *n_out entries (-1 after).  n_out: host; the
 * same count for every sequence, 1 .. gamma + 1: the smallest accepted count
 * of the batch plus one (a sequence that accepted more would emit the same
 * token there).  The sequences' length grows by *n_out; the last emitted
 * token is the next call's input.
 *   scratch: device memory, 256-byte aligned, of at least
 * dory_speculative_scratch_bytes(m, B, gamma) bytes (verifier and drafter
 * logits, drafts, saved ring slots).  Requires 1 <= k_draft <= k_verify, 1 <= gamma <= 16,
 * gamma + 1 <= max_chunk and length + gamma + 1 <= max_ctx.
 *   Unlike the other compute calls this one synchronises `stream` once, to
 * read the accepted count. */
DORY_API int dory_speculative_step(dory_t* m, const int32_t* tokens, int B, int k_draft,
                                   int k_verify, int gamma, void* scratch, size_t scratch_bytes,
                                   int32_t* out, int* n_out, void* stream);

/* The same step with rejection sampling instead of greedy acceptance
 * ("Dory1.0-4B: A Looped Normalized-GPT", Self-Speculative Decoding: the
 * shallow loop count drafts, the full count verifies in one pass, and
 * rejection sampling keeps the verifier's distribution).  Distributions are
 * softmax(logits / temperature), temperature > 0.  A draw from weights w
 * with uniform v is the smallest index whose running sum (vocabulary order)
 * exceeds v * sum(w).  Draft i of sequence b is drawn with u[b][i] from the
 * drafter's distribution q; it is kept iff u[b][gamma + i] * q(x) < p(x) (p:
 * the verifier's distribution at that position), and only while every
 * earlier draft was kept.  The batch advances by n = (fewest kept drafts) +
 * 1; at the last emitted position a sequence emits its kept draft, else a
 * draw with u[b][2 gamma] from max(0, p - q) (its first rejected position)
 * or, when every draft was kept, from the verifier's distribution after the
 * last draft.  Every emitted token then follows the verifier's conditional
 * distribution.
 *   u: device fp32 [B][2 gamma + 1] uniforms in [0, 1) (the caller's random
 * numbers).  out, n_out, scratch, requirements and the synchronisation as
 * for dory_speculative_step; kept (device int32 [B], may be NULL) receives
 * each sequence's count of leading kept drafts.  DORY_EINVAL for u NULL or
 * temperature <= 0. */
DORY_API int dory_speculative_sample_step(dory_t* m, const int32_t* tokens, int B, int k_draft,
                                          int k_verify, int gamma, float temperature,
                                          const float* u, void* scratch, size_t scratch_bytes,
                                          int32_t* out, int* n_out, int32_t* kept, void* stream);

/* Scratch bytes dory_speculative_step and dory_speculative_sample_step need
 * for B sequences and gamma drafts with the handle's current binding; 0 on
 * bad arguments or before dory_bind. */
DORY_API size_t dory_speculative_scratch_bytes(const dory_t* m, int B, int gamma);

/* Test-only: byte offsets inside the speculative scratch of the verifier
 * logits (fp32 [B][gamma + 1][V]), the drafter logits (fp32 [gamma][B][V],
 * written by the sampled step) and the drafts (int32 [gamma][B]):
 * offsets[0..2].  DORY_EINVAL on bad arguments or before dory_bind. */
DORY_API int dory_debug_speculative_layout(const dory_t* m, int B, int gamma, size_t* offsets);

/* One token per row of logits (device fp32 [rows][V]) drawn from
 * softmax(logits / temperature) with the uniform u[row] (device fp32 [rows],
 * in [0, 1)), by the rule of dory_speculative_sample_step; out: device int32
 * [rows].  Asynchronous on `stream`.  DORY_EINVAL for null pointers,
 * rows or V <= 0, temperature <= 0. */
DORY_API int dory_sample_tokens(const float* logits, int rows, int V, float temperature,
                                const float* u, int32_t* out, void* stream);

/* Prefix caching: copies the cached keys and values of positions 0 .. len-1
 * of sequence src into each sequence dst[i] (host array of n_dst distinct
 * indices other than src, all below max_batch; n_dst <= 256), for every
 * layer and every slice of the bound cache mode, so that those sequences can
 * continue from the same prompt without recomputing it (the serving setup
 * of "Dory1.0-4B: A Looped Normalized-GPT", Last-Loop KV Caching, reuses
 * cached prompt prefixes).  Full-layer
 * slots 0 .. len-1 are copied, and window-layer rings as they stand (slot
 * p mod ring size).  Asynchronous on `stream`; host state is not changed:
 * declare the new length with dory_set_length(B, len) before continuing all
 * B sequences together.  Requires len <= max_ctx (DORY_ECAPACITY). */
DORY_API int dory_copy_prefix(dory_t* m, int src, const int* dst, int n_dst, int len,
                              void* stream);

/* ------------------------------------------------------------------------
 * Weight-only quantised decode ("Dory1.0-4B: A Looped Normalized-GPT",
 * Quantization: post-training quantisation of every weight matrix except
 * the token embeddings and the LM head, weights only; MXFP8 with maximum
 * scaling, NVFP4 with each block's E4M3 scale chosen to minimise the block's
 * squared error over all 126 positive finite E4M3 values).
 *
 * Formats of a row-major [rows, K] matrix (blocks run along K):
 *   DORY_QUANT_MXFP8: codes [rows][K] E4M3 (sign in bit 7); scales
 *     [rows][K/32] E8M0 (value 2^(s - 127)); weight = code * 2^(s - 127).
 *     The block exponent is floor(log2 max|x|) - 8, clamped to [-127, 127]
 *     (-127 for a block whose maximum is 0 or subnormal); elements round to
 *     nearest even, saturating at 448.
 *   DORY_QUANT_NVFP4: codes [rows][K/2] E2M1 (element 2i in the low nibble,
 *     sign in bit 3 of a nibble); scales [rows][K/16] E4M3 block scales s;
 *     row_scale [rows] fp32, the tensor's scale s_g = max|x| / 2688 (1 for
 *     an all-zero tensor) on every row; weight = code * s * s_g.  The block
 *     scale is the first candidate, in increasing order, with the smallest
 *     float32 error sum over the block of (x - q*d)^2, d = s*s_g, q = E2M1
 *     rounding (nearest even, at most 6) of x/d, each operation rounded in
 *     float32, elements in order.
 * ---------------------------------------------------------------------- */
typedef enum { DORY_QUANT_NONE = 0, DORY_QUANT_MXFP8 = 1, DORY_QUANT_NVFP4 = 2 } dory_quant_format;

/* Bytes of the codes and block scales of a rows x K matrix in format fmt
 * (pure host function).  K must be a multiple of 32.  DORY_EINVAL for a bad
 * format or size. */
DORY_API int dory_quant_bytes(int fmt, int rows, int K, size_t* codes_bytes,
                              size_t* scales_bytes);

/* Quantises the bf16 matrix W [rows, K] (device, 16-byte aligned, K a
 * multiple of 32) as ONE tensor: codes and scales (device, sizes from
 * dory_quant_bytes; codes 16-byte aligned) and row_scale (device fp32
 * [rows]; NVFP4: required, receives s_g on every row; MXFP8: may be NULL,
 * else receives 1.0).  deq (device bf16 [rows, K], may be NULL, may equal
 * W) receives the dequantised weights rounded to bf16 (exact for MXFP8).
 * Asynchronous on `stream`.  Sub-tensors that share one packed matrix (the
 * q, k, v and gate rows of w_qkvg; the up and SiLU-gate rows of w_upgate)
 * are quantised by one call each, at their row offsets. */
DORY_API int dory_quantize_matrix(int fmt, const void* W, int rows, int K, void* codes,
                                  void* scales, float* row_scale, void* deq, void* stream);

/* The quantised form of one projection matrix (device pointers, layout as
 * above; row_scale may be NULL for MXFP8). */
typedef struct {
    const void* codes;
    const void* scales;
    const float* row_scale;
} dory_qmatrix;

typedef struct {
    dory_qmatrix qkvg, o, upgate, down;   /* same rows and K as the bf16 matrices */
} dory_qlayer;

/* From now on the decode projections stream these quantised weights
 * instead of the bf16 ones: through the few-row GEMVs for decode steps of
 * one sequence and prefill chunks of up to 4 rows, and, when
 * dory_set_quantized_swap enables it, for decode steps of 2 to 128
 * sequences through the swapped tensor-core GEMM, which expands each
 * tile's codes to bf16 in shared memory.  The other projections (decode of
 * 2 to 128 sequences by default, prefill chunks of 5 or more rows, where
 * decoding the codes per row made the GEMV compute-bound) keep reading the
 * bf16 matrices, which should then hold the dequantised values
 * (dory_quantize_matrix's deq): the expanded tiles equal those values
 * exactly, so every path computes with the same weights.  The LM head and the embeddings are never
 * quantised.  layers: HOST array of n_layers entries (copied); fmt
 * DORY_QUANT_NONE switches back to the bf16 weights (layers may be NULL).
 * DORY_EINVAL for null pointers, misaligned codes (16 bytes) or NVFP4
 * scales (2 bytes), or d, n_q*head_dim or ffn not multiples of 32. */
DORY_API int dory_set_quantized_weights(dory_t* m, int fmt, const dory_qlayer* layers);

/* stream_codes 1: decode steps of 2 to 128 sequences run their quantised
 * projections through the swapped GEMM that expands the codes in shared
 * memory (projections whose K is a multiple of 512 for MXFP8 or 256 for
 * NVFP4, so that a row's block scales come in 16-byte groups; the others
 * keep the bf16 matrices); 0 (the default): they read the dequantised bf16
 * matrices.  Both
 * give bit-identical results.  The default is the faster one on B300 for
 * the 4B-class decode shapes: those GEMMs are short and latency-bound, so
 * halving or quartering their weight bytes does not shorten them, and the
 * expansion adds its own latency.  Host state only; applies to later
 * steps.  DORY_EINVAL for a null handle or a value other than 0 / 1. */
DORY_API int dory_set_quantized_swap(dory_t* m, int stream_codes);

/* ------------------------------------------------------------------------
 * Ragged batches: sequences of different lengths in one decode step (the
 * serving setting of "Dory1.0-4B: A Looped Normalized-GPT", Last-Loop KV
 * Caching; each sequence computes exactly what it computes alone).  The
 * handle then keeps one length per batch slot.  The uniform calls
 * (dory_prefill, dory_decode_step, dory_speculative_step /
 * _sample_step) return DORY_EINVAL while the lengths are per sequence;
 * dory_set_length or dory_reset returns to one shared length.
 * ---------------------------------------------------------------------- */

/* Declares per-sequence lengths: batch slots 0 .. B-1 hold lengths[b]
 * positions (host array; host state only, as dory_set_length).  Requires
 * B <= max_batch and lengths <= max_ctx (DORY_ECAPACITY). */
DORY_API int dory_set_lengths(dory_t* m, int B, const int* lengths);

/* The lengths of batch slots 0 .. B-1 (host array out; no CUDA call). */
DORY_API int dory_get_lengths(const dory_t* m, int B, int* out);

/* Prefill of ONE sequence in batch slot `slot` (< max_batch), continuing from
 * that slot's own length: T tokens (device int32), loop count k, logits of
 * the last position [V] or, with all_logits, of every position [T][V].
 * The other slots are untouched.  Asynchronous on `stream`.  From the
 * uniform state, every slot keeps its length and the handle switches to
 * per-sequence lengths. */
DORY_API int dory_prefill_slot(dory_t* m, int slot, const int32_t* tokens, int T, int k,
                               int cache_mode, float* logits, int all_logits, void* stream);

/* One decode step of batch slots 0 .. B-1 (B <= 128), each at its own
 * length: token b is the next token of slot b; RoPE, the visible keys, the
 * window and the ring slot of its new key and value follow its own
 * position.  Arguments and outputs as for dory_decode_step.  Each slot's
 * length grows by one.  The decode attention's schedule gives every
 * (sequence, kv head) group as many key tiles as the longest sequence has,
 * so a batch costs about what the same batch at its longest length costs. */
DORY_API int dory_decode_step_ragged(dory_t* m, const int32_t* tokens, int B, int k,
                                     int cache_mode, float* logits, int32_t* next, void* stream);

/* The same step with one loop count per sequence: ks (host int[B], each
 * >= 1), last-loop cache only (else DORY_EKMISMATCH).  Sequence b runs the
 * recurrent block ks[b] times, stores its key and value of each recurrent
 * layer at its own last loop and enters the output block with s_(ks[b]),
 * exactly as a step at k = ks[b] alone.  The recurrent block runs max(ks)
 * times for the whole batch (rows past their count compute values that are
 * discarded). */
DORY_API int dory_decode_step_multi(dory_t* m, const int32_t* tokens, int B, const int* ks,
                                    int cache_mode, float* logits, int32_t* next, void* stream);

/* A mixed step: one forward pass over Bd decode rows (batch slots 0 ..
 * Bd-1, one token each at its own length) and a chunk of C tokens of the
 * sequence in batch slot `slot` (slot >= Bd, continuing from its own
 * length), so that the decode tokens and the chunk share every weight read
 * (chunked prefill piggybacking on decode).  tokens: device int32 [Bd + C],
 * the decode tokens then the chunk.  logits (may be NULL): device fp32
 * [Bd + 1][V], the decode rows then the chunk's last position; next (may be
 * NULL, needs logits and Bd >= 1): greedy tokens of the decode rows [Bd].
 * One loop count k; the cache mode's rules as for dory_prefill.  Lengths
 * grow by 1 (decode slots) and C (the chunk's slot).  Every row computes
 * what it computes alone.  Requires C <= max_chunk. */
DORY_API int dory_step_mixed(dory_t* m, const int32_t* tokens, int Bd, int slot, int C, int k,
                             int cache_mode, float* logits, int32_t* next, void* stream);

/* Current length of the sequences (host state; no CUDA call). */
DORY_API int dory_length(const dory_t* m, int* out);

/* Declares that the bound KV region already holds positions 0 .. len-1 of B
 * sequences (for instance a cache saved earlier and copied back, in the
 * layout dory_kv_bytes describes); later calls continue at position len.
 * Host state only: the caller is responsible for the cache contents.
 * Requires B <= max_batch and len <= max_ctx (else DORY_ECAPACITY). */
DORY_API int dory_set_length(dory_t* m, int B, int len);

/* Resets every sequence to length 0 (host state only; cache contents are
 * simply overwritten by later calls). */
DORY_API int dory_reset(dory_t* m);

/* Releases the handle (not the caller's memory). */
DORY_API int dory_destroy(dory_t* m);

/* Static description of a status code. */
DORY_API const char* dory_strerror(int status);

/* Synchronises `stream` and reads the device status word of the bound
 * workspace: *out = 0 if every bounded device wait completed, else a code
 * naming the kernel and wait that expired.  The word is cleared. */
DORY_API int dory_device_status(dory_t* m, int* out, void* stream);

/* Number of kernels the last dory_prefill / dory_decode_step launched. */
DORY_API int dory_last_launch_count(const dory_t* m, int* out);

/* ---- per-kernel timing ------------------------------------------------ */

/* Kernel classes for dory_profile_end (one per step of the forward pass). */
typedef enum {
    DORY_K_EMBED = 0,       /* token gather + normalisation */
    DORY_K_ROPE = 1,        /* RoPE cos/sin table for the call's positions */
    DORY_K_QKVG_GEMM = 2,   /* QKV + gate projection, RoPE / q-k norm / sigmoid fused */
    DORY_K_ATTENTION = 3,   /* masked GQA attention over cached + current keys */
    DORY_K_KV_WRITE = 4,    /* KV-cache writer */
    DORY_K_O_GEMM = 5,      /* output projection */
    DORY_K_NGPT_UPDATE = 6, /* nGPT residual step */
    DORY_K_UPGATE_GEMM = 7, /* up + SiLU-gate projection, SwiGLU fused */
    DORY_K_DOWN_GEMM = 8,   /* down projection */
    DORY_K_BOUNDARY = 9,    /* loop-boundary re-injection / normalisation */
    DORY_K_LM_HEAD = 10,    /* logits */
    DORY_K_ARGMAX = 11,     /* greedy token */
    DORY_K_COUNT = 12
} dory_kernel_class;

/* Starts recording a CUDA-event pair around each of the next max_launches
 * kernel launches of this handle (events are created on first use; no device
 * memory).  Launches beyond max_launches are not timed.  Not for use inside
 * stream capture. */
DORY_API int dory_profile_begin(dory_t* m, int max_launches);

/* Stops recording, synchronises the recorded events and writes, per kernel
 * class, the summed elapsed milliseconds (ms[DORY_K_COUNT]) and the number of
 * timed launches (launches[DORY_K_COUNT]). */
DORY_API int dory_profile_end(dory_t* m, double* ms, int* launches);

/* ---- inspection entry points used by the tests (same conventions) ----- */

/* Copies the final hidden states of the last call (the LM-head input, fp32)
 * for all processed rows of the last chunk: [B * C, d], row = b * C + t,
 * C = tokens per sequence in that chunk.  dst: device fp32. */
DORY_API int dory_debug_hidden(dory_t* m, float* dst, int max_rows, void* stream);

/* Test-only: launches one block whose mbarrier wait is never completed,
 * bounded by limit_us microseconds (1 .. 100000) instead of the kernels' 2 s.
 * The wait gives up, writes 0x71 to the handle's device status word (read
 * and cleared by dory_device_status) and the kernel returns, leaving the
 * context usable.  It runs the bounded-wait routine every TMA / tcgen05
 * kernel of the library uses.  DORY_EUNBOUND before dory_bind. */
DORY_API int dory_debug_expire_wait(dory_t* m, int limit_us, void* stream);

/* Byte offset of the K (which = 0) or V (which = 1) block of (layer, slice)
 * inside the KV region, and its ring size in slots. */
DORY_API int dory_debug_kv_offset(const dory_t* m, int layer, int slice, int which,
                         size_t* offset, int* slots);

/* C[M, N] (fp32, row stride ldc) = A[M, K] . B[N, K]^T with A and B bf16
 * row-major (device), through the tensor-core GEMM of the forward pass. */
DORY_API int dory_debug_gemm(const void* A, const void* B, float* C, int M, int N, int K, int ldc,
                    void* stream);

/* The attention step alone, as the forward pass runs it (test inspection):
 * q [B*C, n_q, head_dim], k_cur / v_cur [B*C, n_kv, head_dim], gate
 * [B*C, n_q*head_dim] (already sigmoid), k_cache / v_cache
 * [B, n_kv, S, head_dim] holding positions < P0 in ring slot p mod S;
 * out [B*C, n_q*head_dim] = softmax-weighted values times gate.  window <= 0
 * means full causal; scale <= 0 means sqrt(head_dim).  All bf16, device.
 * With C == 1 the split-key decode kernels run and need `scratch`: device
 * memory of at least dory_debug_attention_scratch_bytes(B, n_q, head_dim)
 * bytes.  With C > 1 a scratch (256-byte aligned, may be NULL) lets the
 * mma.sync kernel split the key range of a short chunk over more CTAs, as
 * the forward pass does with its workspace: up to scratch_bytes /
 * (B*C*n_q*(head_dim + 2)*4 + 512) splits, merged by a second kernel. */
DORY_API int dory_debug_attention(const void* q, const void* k_cur, const void* v_cur,
                                  const void* k_cache, const void* v_cache, const void* gate,
                                  void* out, int B, int C, int P0, int S, int n_q, int n_kv,
                                  int head_dim, int window, float scale, void* scratch,
                                  size_t scratch_bytes, void* stream);

/* Multi-token (prefill) attention runs on the tcgen05 tensor cores when
 * head_dim is 128 and the key tiles of 64 positions line up (P0 a multiple
 * of 64, window and ring size multiples of 64), else on the mma.sync
 * kernel.  enable = 0 forces the mma.sync kernel (for comparison): for the
 * handle m, or, with m = NULL, for dory_debug_attention.  Host state only. */
DORY_API int dory_set_tc_attention(dory_t* m, int enable);

/* Multi-token (prefill) output and down projections: enable = 1 (the
 * default) fuses the nGPT step h <- N(h + alpha (N(y) - h)) ("Dory1.0-4B:
 * A Looped Normalized-GPT", Architecture) into the GEMM epilogue when d is a
 * multiple of 256 with d / 256 <= 8: a thread-block cluster of d / 256 CTAs
 * holds whole rows and sums both row norms through distributed shared
 * memory.  enable = 0 runs the GEMM and a separate row kernel.  Both give
 * the same results up to rounding order.  Host state only; EINVAL for m =
 * NULL or enable not 0 / 1. */
DORY_API int dory_set_fused_ngpt(dory_t* m, int enable);

/* Scratch bytes dory_debug_attention needs for one-token (decode) calls. */
DORY_API size_t dory_debug_attention_scratch_bytes(int B, int n_q, int head_dim);

/* One-token (decode) attention that needs no memory from the caller beyond
 * its inputs and outputs, and allocates none.  The paper has no counterpart:
 * this exists for callers that cannot hand the library any scratch memory,
 * such as a plug-in running inside a host program that owns every device
 * allocation and gives its extensions neither an allocator nor a workspace,
 * or a latency-critical serving loop that forbids cudaMalloc after start-up
 * because it can block and synchronise the device.
 *
 * Arguments: q [B, n_q, head_dim] (queries already rotated, normalised and
 * scaled), k_cur / v_cur [B, n_kv, head_dim] (the new token's key and value,
 * at position P0), gate and out [B, n_q * head_dim], k_cache / v_cache
 * [B, n_kv, S, head_dim] holding positions < P0 in ring slot p mod S; all
 * bf16, device.  out = gate * softmax-weighted values over the keys that the
 * mask shows (positions j <= P0, and P0 - j < window when window > 0).
 * It runs the split-key kernel pair of attn.cuh (attn_decode_split_kernel:
 * one CTA per (split, kv head, sequence), scalar fp32 dot products; then
 * attn_decode_combine_kernel merges the splits and applies the gate), not
 * the TMA-fed kernel of the forward pass; results agree with
 * dory_debug_attention with C == 1 up to rounding order.
 *
 * Refusals, all before any launch: DORY_EINVAL for null pointers, n_q not a
 * multiple of n_kv or n_q / n_kv > 8, k_cur / v_cur / k_cache / v_cache not
 * 16-byte aligned (q, gate, out: 2-byte), or a ring too small for the keys
 * the mask shows (S < P0 with window <= 0, S < min(P0, window - 1) with a
 * window); DORY_EUNSUPPORTED for head_dim outside {32, 64, 128};
 * DORY_ECAPACITY when the partials would not fit the array (below).
 *
 * The split-key partial results live in a fixed 16 MiB array inside the
 * library; every GPU that loads the library holds it until the process
 * exits.  Calls with dory_debug_attention_scratch_bytes(B, n_q, head_dim) >
 * 16 MiB are refused (for head_dim 128 that is B * n_q > 252).  Every call
 * looks up the array's device address in the current device's context
 * (cudaGetSymbolAddress); the first call on a device also loads the module
 * there, so make that first call before any stream capture.  All calls share
 * the one array and leave it holding their partials; nothing in it needs to
 * start at zero, but calls whose kernels overlap on the GPU (other streams,
 * other threads) race on it, so serialise them. */
DORY_API int dory_decode_attention_noalloc(const void* q, const void* k_cur, const void* v_cur,
                                           const void* k_cache, const void* v_cache,
                                           const void* gate, void* out, int B, int P0, int S,
                                           int n_q, int n_kv, int head_dim, int window,
                                           float scale, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DORY_H */
