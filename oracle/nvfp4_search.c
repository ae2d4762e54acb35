/*
 * nvfp4_search.c - the squared-error block-scale search of NVFP4 weight
 * quantisation, for the CPU oracle (TEST INFRASTRUCTURE ONLY: loaded by
 * oracle/quant.py; the product path never uses it).
 *
 * "Dory1.0-4B: A Looped Normalized-GPT", Quantization (Post-Training
 * Quantization): for NVFP4, each block's scale is the positive finite E4M3
 * value that minimises the squared quantisation error of the block.
 *
 * The same float32 expression, in the same order, as nvfp4_block_error in
 * oracle/quant.py (which is the readable definition; this file only makes
 * it fast enough for whole matrices):
 *   d = fl(s * s_g);  v = fl(x / d);  q = E2M1 rounding of v (nearest,
 *   ties to the even code, saturating at 6, sign of v kept);
 *   e = fl(x - fl(q * d));  err = fl(err + fl(e * e)), elements in order;
 * candidates in increasing order of s, the first smallest error wins.
 * Build without floating-point contraction (-ffp-contract=off) so that no
 * multiply-add is fused.
 */
#include <math.h>
#include <stdint.h>

/* E2M1 magnitude code (0..7) of a >= 0: nearest of 0, .5, 1, 1.5, 2, 3, 4, 6
 * with ties to the even code.  Midpoints: 0.25 0.75 1.25 1.75 2.5 3.5 5. */
static int e2m1_mag_code(float a) {
    if (a <= 0.25f) return 0;     /* tie 0.25 -> code 0 */
    if (a < 0.75f) return 1;      /* tie 0.75 -> code 2 */
    if (a <= 1.25f) return 2;     /* tie 1.25 -> code 2 */
    if (a < 1.75f) return 3;      /* tie 1.75 -> code 4 */
    if (a <= 2.5f) return 4;      /* tie 2.5  -> code 4 */
    if (a < 3.5f) return 5;       /* tie 3.5  -> code 6 */
    if (a <= 5.0f) return 6;      /* tie 5    -> code 6 */
    return 7;
}

static const float E2M1_MAG[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

/* x: n_blocks x 16 float32 (bf16-exact weights); cand: n_cand block-scale
 * values in increasing order; s_g: the tensor's float32 scale.
 * Out: best[b] = index of the chosen candidate; codes[b * 16 + i] = E2M1
 * code (sign in bit 3) of element i under that scale. */
void nvfp4_search(const float* x, long n_blocks, const float* cand, int n_cand, float s_g,
                  uint8_t* best, uint8_t* codes) {
#pragma omp parallel for schedule(static)
    for (long b = 0; b < n_blocks; ++b) {
        const float* xb = x + b * 16;
        float best_err = INFINITY;
        int bc = 0;
        for (int c = 0; c < n_cand; ++c) {
            const float d = cand[c] * s_g;
            float err = 0.0f;
            for (int i = 0; i < 16; ++i) {
                const float v = xb[i] / d;
                const float q = copysignf(E2M1_MAG[e2m1_mag_code(fabsf(v))], v);
                const float qd = q * d;
                const float e = xb[i] - qd;
                const float ee = e * e;
                err = err + ee;
            }
            if (err < best_err) {
                best_err = err;
                bc = c;
            }
        }
        best[b] = (uint8_t)bc;
        const float d = cand[bc] * s_g;
        for (int i = 0; i < 16; ++i) {
            const float v = xb[i] / d;
            codes[b * 16 + i] = (uint8_t)(e2m1_mag_code(fabsf(v)) | (signbit(v) ? 8 : 0));
        }
    }
}
