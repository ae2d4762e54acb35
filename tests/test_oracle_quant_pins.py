"""Pins of the oracle's weight-only quantisers (oracle/quant.py) against
facts that do not come from the oracle itself: the published E4M3 / E2M1
code tables, torch's float8_e4m3fn conversion (round to nearest even),
closed forms of maximum scaling, exactly representable blocks, and a
float64 brute force over all 126 block scales ("Dory1.0-4B: A Looped
Normalized-GPT", Quantization: Post-Training Quantization)."""
import numpy as np
import pytest
import torch

import synth
from oracle import quant

RNG = np.random.default_rng(1234)


# ------------------------------------------------------------ element formats
def test_e4m3_code_table():
    v = quant.e4m3_magnitudes()
    # values fixed by the format: subnormals m * 2^-9, min normal 2^-6,
    # 1.0 at exponent field 7, largest finite 1.75 * 2^8
    assert v[0x00] == 0.0 and v[0x01] == 2.0 ** -9 and v[0x07] == 7 * 2.0 ** -9
    assert v[0x08] == 2.0 ** -6 and v[0x38] == 1.0 and v[0x3F] == 1.875
    assert v[0x40] == 2.0 and v[0x7E] == 448.0
    assert len(v) == 127 and np.all(np.diff(v) > 0)       # 126 positive finite values
    # the same values as torch's float8_e4m3fn
    t = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(t.astype(np.float64), v)


def test_e2m1_code_table():
    assert list(quant.e2m1_magnitudes()) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_round_e4m3_matches_torch_round_to_nearest_even():
    # every midpoint between neighbouring magnitudes, the values themselves,
    # and dense random values, both signs, within the finite range
    v = quant.e4m3_magnitudes()
    mids = (v[1:] + v[:-1]) / 2
    rnd = RNG.uniform(0, 448, 20000) * np.exp2(RNG.integers(-14, 1, 20000))
    x = np.concatenate([v, mids, rnd, np.nextafter(mids, 0), np.nextafter(mids, 1000)])
    x = np.concatenate([x, -x]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(quant.round_e4m3(x), ref)


def test_round_e4m3_saturates():
    x = np.array([448.0, 449.0, 463.9, 464.0, 1e6, -500.0])
    assert list(quant.round_e4m3(x)) == [0x7E] * 5 + [0xFE]


def test_round_e2m1_ties_and_saturation():
    x = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.5, 100.0, -0.25, -5.0, -0.1])
    got = quant.e2m1_value(quant.round_e2m1(x))
    assert list(got) == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0, -0.0, -4.0, -0.0]
    assert quant.round_e2m1(np.array([-0.1]))[0] == 0x8        # sign kept on zero


def test_round_e2m1_is_nearest():
    x = RNG.uniform(-7, 7, 50000)
    q = quant.e2m1_value(quant.round_e2m1(x))
    grid = np.concatenate([-quant.e2m1_magnitudes(), quant.e2m1_magnitudes()])
    best = np.min(np.abs(x[:, None] - grid[None, :]), axis=1)
    assert np.all(np.abs(x - q) == best)


# ------------------------------------------------------------------- MXFP8
def test_mxfp8_scale_is_max_scaling():
    w = synth.round_bf16(RNG.standard_normal((64, 256)).astype(np.float32) * 0.02)
    codes, scales = quant.quantize_mxfp8(w)
    e = scales.astype(np.int64) - 127
    amax = np.abs(w.reshape(64, 8, 32)).max(-1)
    # 2^(e + 8) <= amax < 2^(e + 9): the block maximum scales into [256, 512)
    assert np.all(np.exp2(e + 8) <= amax) and np.all(amax < np.exp2(e + 9))


def test_mxfp8_elements_match_torch_conversion():
    w = synth.round_bf16(RNG.standard_normal((128, 512)).astype(np.float32) * 0.02)
    codes, scales = quant.quantize_mxfp8(w)
    e = (scales.astype(np.float64) - 127).repeat(32, axis=1)
    v = (w / np.exp2(e)).astype(np.float32)
    ok = np.abs(v) <= 448                                   # torch does not saturate
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes[ok], ref[ok])
    assert np.all(codes[~ok] & 0x7F == 0x7E)


def test_mxfp8_exactly_representable_blocks_round_trip():
    rows, nb = 32, 6
    mags = quant.e4m3_magnitudes()
    c = RNG.integers(0, 127, (rows, nb, 32)).astype(np.uint8)
    c[:, :, 5] = RNG.integers(0x78, 0x7F, (rows, nb))        # a block maximum in [256, 448]
    c |= (RNG.integers(0, 2, c.shape) << 7).astype(np.uint8)
    e = RNG.integers(-20, 5, (rows, nb))
    w = (quant.e4m3_value(c) * np.exp2(e)[..., None]).reshape(rows, nb * 32)
    codes, scales = quant.quantize_mxfp8(w)
    assert np.array_equal(scales.astype(np.int64) - 127, e)
    nz = mags[c & 0x7F] != 0                                 # zeros may carry either sign
    assert np.array_equal(codes.reshape(c.shape)[nz], c[nz])
    assert np.array_equal(quant.dequantize_mxfp8(codes, scales), w)


def test_mxfp8_error_bound():
    w = synth.round_bf16(RNG.standard_normal((64, 1024)).astype(np.float32) * 0.02)
    codes, scales = quant.quantize_mxfp8(w)
    deq = quant.dequantize_mxfp8(codes, scales)
    e = np.exp2(scales.astype(np.float64) - 127).repeat(32, axis=1)
    normal = np.abs(w) >= 2.0 ** -6 * e
    sat = np.abs(w) > 448 * e
    err = np.abs(w - deq)
    assert np.all(err[normal & ~sat] <= 2.0 ** -4 * np.abs(w[normal & ~sat]))   # half ulp, 3 bits
    assert np.all(err[~normal] <= 2.0 ** -10 * e[~normal])                      # half subnormal step
    assert np.all(err[sat] < 64 * e[sat])


def test_mxfp8_zero_block():
    codes, scales = quant.quantize_mxfp8(np.zeros((2, 64)))
    assert np.all(codes == 0) and np.all(scales == 0)


# ------------------------------------------------------------------- NVFP4
def test_nvfp4_global_scale():
    w = synth.round_bf16(RNG.standard_normal((16, 64)).astype(np.float32))
    assert quant.nvfp4_global_scale(w) == np.float32(np.float32(np.abs(w).max()) / np.float32(2688))
    assert quant.nvfp4_global_scale(np.zeros((2, 16))) == 1.0


def test_nvfp4_exactly_representable_blocks_have_zero_error():
    rows, nb = 64, 8
    g = 2.0 ** -12
    q = quant.e2m1_value(RNG.integers(0, 16, (rows, nb, 16)).astype(np.uint8))
    s = quant.e4m3_value(RNG.integers(1, 127, (rows, nb)).astype(np.uint8))
    q[0, 0, 0], s[0, 0] = 6.0, 448.0                         # max |w| = 6 * 448 * g: s_g = g
    w = q * s[..., None] * g
    w = w.reshape(rows, nb * 16).astype(np.float32)
    codes, scales, s_g = quant.quantize_nvfp4(w)
    assert s_g == np.float32(g)
    assert np.array_equal(quant.dequantize_nvfp4(codes, scales, s_g), w.astype(np.float64))


def _mse64(x, s, s_g):
    d = s * np.float64(s_g)
    q = quant.e2m1_value(quant.round_e2m1(x / d))
    return np.sum((x - q * d) ** 2, axis=-1)


def test_nvfp4_scale_search_is_optimal_in_float64():
    w = synth.round_bf16(RNG.standard_normal((32, 256)).astype(np.float32) * 0.02)
    w[3, 17] = 0.2                                           # one large value: varied block ranges
    codes, scales, s_g = quant.quantize_nvfp4(w)
    x = w.reshape(-1, 16).astype(np.float64)
    cand = quant.e4m3_value(np.arange(1, 127, dtype=np.uint8))
    all_err = np.stack([_mse64(x, s, s_g) for s in cand], axis=1)
    chosen = _mse64(x, quant.e4m3_value(scales.reshape(-1))[:, None], s_g)
    best = all_err.min(axis=1)
    assert np.all(chosen <= best * (1 + 1e-5) + 1e-30)
    # and never worse than maximum scaling (one of the candidates)
    amax = np.abs(x).max(axis=1)
    smax = quant.e4m3_value(quant.round_e4m3(amax / (6 * np.float64(s_g))))
    smax = np.where(smax == 0, cand[0], smax)
    assert np.all(chosen <= _mse64(x, smax[:, None], s_g) * (1 + 1e-5) + 1e-30)
    # the stored codes are the rounding of x under the chosen scale
    d = (quant.e4m3_value(scales.reshape(-1))[:, None] * np.float64(s_g))
    deq = quant.dequantize_nvfp4(codes, scales, s_g).reshape(-1, 16)
    assert np.all(np.abs(x - deq) <= np.abs(x - quant.e2m1_value(quant.round_e2m1(x / d)) * d) + 1e-12 * d)


def test_nvfp4_first_minimum_wins():
    # a block of zeros has zero error under every scale: the smallest is taken
    codes, scales, _ = quant.quantize_nvfp4(np.array([[0.0] * 15 + [1.0], [0.0] * 16]))
    assert scales[1, 0] == 0x01 and np.all(codes[1] == 0)


def test_pack_e2m1_nibble_order():
    assert list(quant.pack_e2m1(np.array([[1, 2, 15, 8]], np.uint8))[0]) == [0x21, 0x8F]


# ------------------------------------------------------------------- model
@pytest.mark.parametrize("fmt", [quant.MXFP8, quant.NVFP4])
def test_quantize_weights_replaces_matrices_only(fmt):
    shape = synth.TINY
    w = synth.make_weights(shape)
    qw, q = quant.quantize_weights(w, fmt)
    for k in ("embed_in", "embed_out", "s_z"):
        assert np.array_equal(qw[k], w[k])
    for lw, ql, lq in zip(w["layers"], qw["layers"], q):
        for name, v in lw.items():
            if name in quant.QUANTISED:
                assert ql[name].shape == v.shape and not np.array_equal(ql[name], v)
                rel = np.linalg.norm(ql[name] - v) / np.linalg.norm(v)
                assert rel < (0.04 if fmt == quant.MXFP8 else 0.15), (name, rel)
            else:
                assert np.array_equal(ql[name], v)


def test_nvfp4_search_c_form_equals_definition():
    """The C form of the scale search takes the same decisions as the numpy
    definition: random blocks, exactly representable blocks (many scales
    tie at zero error) and blocks with zeros."""
    w = synth.round_bf16(RNG.standard_normal((48, 128)).astype(np.float32) * 0.02)
    q = quant.e2m1_value(RNG.integers(0, 16, (16, 8, 16)).astype(np.uint8))
    s = quant.e4m3_value(RNG.integers(1, 127, (16, 8)).astype(np.uint8))
    w[:16] = (q * s[..., None] * 2.0 ** -14).reshape(16, 128)
    w[20, :40] = 0.0
    for s_g in (None, np.float32(3.1e-6)):
        a = quant.quantize_nvfp4(w, s_g=s_g, fast=True)
        b = quant.quantize_nvfp4(w, s_g=s_g, fast=False)
        assert a[2] == b[2]
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
