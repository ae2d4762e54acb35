"""Weight-only quantisation of the projection matrices (MXFP8, NVFP4).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module;
only the tests and the benchmark's CPU-baseline leg do.

"Dory1.0-4B: A Looped Normalized-GPT", Quantization (Post-Training
Quantization): every weight matrix except the token embeddings and the LM
head is quantised, weights only (activations stay in high precision), and
every learned vector stays in high precision.  MXFP8 uses plain maximum
scaling; NVFP4 picks each block's scale as the one, among all 126 positive
finite E4M3 values, that gives the smallest squared error over the block.

The formats themselves are not defined on the pages; they are the published
ones:
  * E4M3 (OCP 8-bit floating point, "FN" variant): sign, 4 exponent bits
    (bias 7), 3 mantissa bits; exponent field 0 is subnormal (m/8 * 2^-6);
    no infinities; S.1111.111 is NaN, so the largest finite value is
    1.75 * 2^8 = 448.  Codes 0x01..0x7E are the 126 positive finite values.
  * E2M1 (OCP Microscaling formats): sign, 2 exponent bits (bias 1), 1
    mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 for codes 0..7.
  * MXFP8 (OCP Microscaling formats v1.0): blocks of 32 consecutive elements
    along a row share one E8M0 scale 2^e (stored as e + 127).  Maximum
    scaling sets e = floor(log2(max |x|)) - 8 (8 = the exponent of E4M3's
    largest power of two), and each element is x / 2^e rounded to E4M3.
  * NVFP4: blocks of 16 consecutive elements share one E4M3 scale s, and
    the tensor has one fp32 scale s_g; an element is stored as an E2M1 value
    q with x ~ q * s * s_g.  s_g = max |x| over the tensor / (6 * 448), so
    that the largest block scale the maximum-scaling rule would need is
    E4M3's largest value.

Readings where neither the pages nor the format documents fix a detail
(each listed in the design notes):
  * rounding to E4M3 / E2M1 is to nearest, ties to the even code, and
    saturates at the largest finite magnitude; the sign of x is kept even
    when the magnitude rounds to zero;
  * MXFP8: e is clamped to [-127, 127]; a block whose maximum is 0 or
    below the normal range gets e = -127;
  * NVFP4: an all-zero tensor gets s_g = 1.  The squared error of a
    candidate scale s is evaluated in float32, exactly as written in
    nvfp4_block_error (d = fl(s * s_g); v = fl(x / d); e = fl(x - fl(q * d));
    err = fl(err + fl(e * e)) over the 16 elements in order), and the first
    candidate in increasing order of s with the smallest error wins.  The
    decision is an integer taken from floating point, so it is pinned to one
    precision and order; the GPU quantiser evaluates the same expression.
  * the dequantised weight is q * s * s_g (NVFP4) or code * 2^e (MXFP8),
    exact in float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

MXFP8 = 1
NVFP4 = 2
E4M3_MAX = 448.0
E2M1_MAX = 6.0
MX_BLOCK = 32
NV_BLOCK = 16


def e4m3_magnitudes() -> np.ndarray:
    """Magnitude of E4M3 codes 0x00..0x7E (index = code without the sign)."""
    out = np.empty(127, np.float64)
    for code in range(127):
        e, m = code >> 3, code & 7
        out[code] = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


def e2m1_magnitudes() -> np.ndarray:
    """Magnitude of E2M1 codes 0..7 (index = code without the sign)."""
    out = np.empty(8, np.float64)
    for code in range(8):
        e, m = code >> 1, code & 1
        out[code] = (m / 2.0) * 1.0 if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return out


_E4M3 = e4m3_magnitudes()
_E2M1 = e2m1_magnitudes()


def _round_to_grid(a: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the nearest grid value to each non-negative a (grid ascending,
    index = code): ties go to the even index; beyond the last value, the
    last index (saturation)."""
    a = np.asarray(a, np.float64)
    hi = np.clip(np.searchsorted(grid, a, side="left"), 1, len(grid) - 1)
    lo = hi - 1
    dlo = a - grid[lo]
    dhi = grid[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    idx = np.where(pick_hi, hi, lo)
    return np.where(a >= grid[-1], len(grid) - 1, idx)


def round_e4m3(x: np.ndarray) -> np.ndarray:
    """E4M3 codes (uint8, sign in bit 7) of x: nearest, ties to even, saturating."""
    x = np.asarray(x, np.float64)
    mag = _round_to_grid(np.abs(x), _E4M3).astype(np.uint8)
    return np.where(np.signbit(x), mag | np.uint8(0x80), mag).astype(np.uint8)


def e4m3_value(code: np.ndarray) -> np.ndarray:
    code = np.asarray(code, np.uint8)
    v = _E4M3[code & 0x7F]
    return np.where(code & 0x80, -v, v)


def round_e2m1(x: np.ndarray) -> np.ndarray:
    """E2M1 codes (0..15, sign in bit 3) of x: nearest, ties to even, saturating."""
    x = np.asarray(x, np.float64)
    mag = _round_to_grid(np.abs(x), _E2M1).astype(np.uint8)
    return np.where(np.signbit(x), mag | np.uint8(0x8), mag).astype(np.uint8)


def e2m1_value(code: np.ndarray) -> np.ndarray:
    code = np.asarray(code, np.uint8)
    v = _E2M1[code & 0x7]
    return np.where(code & 0x8, -v, v)


# ---------------------------------------------------------------- MXFP8
def quantize_mxfp8(w: np.ndarray):
    """MXFP8 quantisation of a [rows, K] matrix (K a multiple of 32).

    Returns (codes uint8 [rows, K], scales uint8 [rows, K / 32]) with
    scales = e + 127, the block's shared exponent."""
    w = np.asarray(w, np.float64)
    rows, K = w.shape
    assert K % MX_BLOCK == 0
    blk = w.reshape(rows, K // MX_BLOCK, MX_BLOCK)
    amax = np.abs(blk).max(axis=-1)
    _, p = np.frexp(amax)                       # amax = f * 2^p, f in [0.5, 1)
    e = (p - 1) - 8                             # floor(log2 amax) - emax(E4M3)
    e = np.where(amax < 2.0 ** -126, -127, np.clip(e, -127, 127))
    v = blk / np.exp2(e)[..., None]
    codes = round_e4m3(v).reshape(rows, K)
    return codes, (e + 127).astype(np.uint8)


def dequantize_mxfp8(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    rows, K = codes.shape
    v = e4m3_value(codes).reshape(rows, K // MX_BLOCK, MX_BLOCK)
    return (v * np.exp2(scales.astype(np.float64) - 127)[..., None]).reshape(rows, K)


# ---------------------------------------------------------------- NVFP4
def nvfp4_global_scale(w: np.ndarray) -> np.float32:
    """s_g = max |w| / (6 * 448), in float32 (1 for an all-zero tensor)."""
    amax = np.float32(np.max(np.abs(np.asarray(w, np.float32)))) if w.size else np.float32(0)
    if amax == 0:
        return np.float32(1.0)
    return np.float32(amax / np.float32(E2M1_MAX * E4M3_MAX))


def nvfp4_block_error(x: np.ndarray, s: np.float32, s_g: np.float32):
    """Float32 squared error of quantising the blocks x [n, 16] with block
    scale s (E4M3 value) under global scale s_g; returns (err [n], q codes
    [n, 16]).  The operations and their order are part of the definition."""
    x = np.asarray(x, np.float32)
    d = np.float32(np.float32(s) * np.float32(s_g))
    v = (x / d).astype(np.float32)
    codes = round_e2m1(v)
    q = e2m1_value(codes).astype(np.float32)
    err = np.zeros(x.shape[0], np.float32)
    for i in range(x.shape[1]):
        qd = (q[:, i] * d).astype(np.float32)
        e = (x[:, i] - qd).astype(np.float32)
        err = (err + (e * e).astype(np.float32)).astype(np.float32)
    return err, codes


_HERE = os.path.dirname(os.path.abspath(__file__))
_SEARCH_SRC = os.path.join(_HERE, "nvfp4_search.c")
_SEARCH_LIB = os.path.join(_HERE, "_nvfp4_search.so")
_search = None


def _search_lib():
    """The C form of the NVFP4 scale search (nvfp4_search.c), compiled with
    gcc on first use (or by the package build)."""
    global _search
    if _search is None:
        if (not os.path.exists(_SEARCH_LIB)
                or os.path.getmtime(_SEARCH_LIB) < os.path.getmtime(_SEARCH_SRC)):
            subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC",
                            "-o", _SEARCH_LIB + ".tmp", _SEARCH_SRC, "-lm"], check=True)
            os.replace(_SEARCH_LIB + ".tmp", _SEARCH_LIB)
        lib = ctypes.CDLL(_SEARCH_LIB)
        P = ctypes.c_void_p
        lib.nvfp4_search.argtypes = [P, ctypes.c_long, P, ctypes.c_int, ctypes.c_float, P, P]
        lib.nvfp4_search.restype = None
        _search = lib
    return _search


def quantize_nvfp4(w: np.ndarray, s_g=None, fast: bool = True, chunk_rows: int = 1024):
    """NVFP4 quantisation of a [rows, K] matrix (K a multiple of 16) with
    the squared-error scale search.  s_g: the tensor's scale when w holds
    only some of its rows (default: computed from w).  fast: run the search
    in its C form (same arithmetic, whole matrices in seconds); False runs
    nvfp4_block_error over every candidate.

    Returns (codes uint8 [rows, K] (one E2M1 code per element, 0..15),
    scales uint8 [rows, K / 16] (E4M3 codes 0x01..0x7E), s_g float32)."""
    w = np.ascontiguousarray(w, np.float32)
    rows, K = w.shape
    assert K % NV_BLOCK == 0
    s_g = nvfp4_global_scale(w) if s_g is None else np.float32(s_g)
    cand = np.arange(1, 127, dtype=np.uint8)                  # increasing magnitude
    cand_val = np.ascontiguousarray(e4m3_value(cand), np.float32)
    if fast:
        nb = rows * K // NV_BLOCK
        best = np.empty(nb, np.uint8)
        codes = np.empty((rows, K), np.uint8)
        _search_lib().nvfp4_search(w.ctypes.data, nb, cand_val.ctypes.data, len(cand_val),
                                   float(s_g), best.ctypes.data, codes.ctypes.data)
        return codes, cand[best].reshape(rows, K // NV_BLOCK), s_g
    codes = np.empty((rows, K), np.uint8)
    scales = np.empty((rows, K // NV_BLOCK), np.uint8)
    for r0 in range(0, rows, chunk_rows):
        x = w[r0:r0 + chunk_rows].reshape(-1, NV_BLOCK)
        best = np.full(x.shape[0], np.inf, np.float32)
        best_code = np.zeros(x.shape[0], np.uint8)
        best_q = np.zeros(x.shape, np.uint8)
        for c, s in zip(cand, cand_val):
            err, q = nvfp4_block_error(x, s, s_g)
            better = err < best                                # first minimum wins
            best = np.where(better, err, best)
            best_code = np.where(better, c, best_code)
            best_q = np.where(better[:, None], q, best_q)
        n = x.shape[0] * NV_BLOCK // K
        codes[r0:r0 + n] = best_q.reshape(n, K)
        scales[r0:r0 + n] = best_code.reshape(n, K // NV_BLOCK)
    return codes, scales, s_g


def dequantize_nvfp4(codes: np.ndarray, scales: np.ndarray, s_g) -> np.ndarray:
    rows, K = codes.shape
    q = e2m1_value(codes).reshape(rows, K // NV_BLOCK, NV_BLOCK)
    s = e4m3_value(scales)[..., None]
    return (q * s * np.float64(s_g)).reshape(rows, K)


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """Two E2M1 codes per byte: element 2i in the low nibble, 2i + 1 in the high."""
    c = np.asarray(codes, np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


# ---------------------------------------------------------------- model
QUANTISED = ("w_q", "w_k", "w_v", "w_g", "w_o", "w_up", "w_sl", "w_down")


def quantize_matrix(w: np.ndarray, fmt: int) -> dict:
    if fmt == MXFP8:
        codes, scales = quantize_mxfp8(w)
        return {"codes": codes, "scales": scales, "deq": dequantize_mxfp8(codes, scales)}
    if fmt == NVFP4:
        codes, scales, s_g = quantize_nvfp4(w)
        return {"codes": codes, "scales": scales, "s_g": s_g,
                "deq": dequantize_nvfp4(codes, scales, s_g)}
    raise ValueError(fmt)


def quantize_weights(weights: dict, fmt: int, keep=None):
    """The model with every projection matrix replaced by its dequantised
    quantisation (embeddings, LM head and vectors unchanged).  Returns
    (weights, per-layer dict of quantize_matrix results)."""
    out = {k: v for k, v in weights.items() if k != "layers"}
    layers, q = [], []
    for lw in weights["layers"]:
        nl, ql = dict(lw), {}
        for name in QUANTISED:
            ql[name] = quantize_matrix(lw[name], fmt)
            nl[name] = ql[name]["deq"]
        layers.append(nl)
        q.append(ql)
    out["layers"] = layers
    return out, q
