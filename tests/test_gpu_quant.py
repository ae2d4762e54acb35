"""Weight-only quantised decode through the C ABI ("Dory1.0-4B: A Looped
Normalized-GPT", Quantization: Post-Training Quantization; MXFP8 with
maximum scaling, NVFP4 with the squared-error scale search).

* The GPU quantiser against the oracle's, bit for bit: codes, block scales
  and the NVFP4 tensor scale, on 4B-width matrices and on blocks built to
  hit the edge cases (zeros, signed zeros, powers of two, outliers that
  saturate, values far below the block maximum); the dequantised bf16
  output equals the oracle's dequantised weights rounded to bf16.
* The model with quantised weights against the oracle run on the
  dequantised weights: prefill (tensor-core projections on the dequantised
  bf16 copy), decode steps and a prefill chunk of at most 4 rows
  (projections streaming the packed codes: the register form on the tiny
  shape, the bulk-copy form at the 4B width, with 1 and with 2-4 rows) and a
  chunk of 15 rows (the dequantised bf16 copy), both cache modes on the tiny
  shape with a full layer in the loop, and at the 4B-class width (3 layers),
  where every projection of the 4B-class model has its full size; decode of
  20 sequences through the swapped tensor-core GEMM that expands the codes
  in shared memory, against the oracle and bit for bit against the same
  GEMM on the dequantised bf16 matrices.  Tolerances as in test_gpu_parity."""
import numpy as np
import pytest

import oracle
import synth
from oracle import quant
from test_gpu_parity import check_greedy, check_hidden, check_logits, _tok

pytestmark = pytest.mark.gpu

FMTS = [quant.MXFP8, quant.NVFP4]
IDS = ["mxfp8", "nvfp4"]


@pytest.fixture(scope="module")
def dev(cuda_ok):
    import looped_normalized_transformer_ngpt_b300 as dory
    from looped_normalized_transformer_ngpt_b300 import _build
    _build.build()
    dory.lib()
    return dory


def _edge_matrix():
    """8 x 128 bf16-exact values with hand-placed edge cases."""
    rng = np.random.default_rng(5)
    w = synth.round_bf16(rng.standard_normal((8, 128)).astype(np.float32) * 0.02)
    w[0, :32] = 0.0                                   # an all-zero MXFP8 block
    w[0, 32:48] = -0.0                                # signed zeros
    w[1, :32] = 2.0 ** rng.integers(-12, -2, 32)      # powers of two
    w[1, 5] = 0.25                                    # the block maximum, a power of two
    w[2, 7] = 3.0                                     # an outlier: the tensor's max
    w[2, 40] = -1.5
    w[2, 70] = 1.875 * 2.0 ** -4                      # a block maximum that saturates in E4M3
    w[3, :32] *= 1e-3                                 # a block far below the others
    w[4, 0:32] = synth.round_bf16(np.linspace(-1, 1, 32).astype(np.float32) * 0.01)
    w[5, 16:32] = synth.round_bf16(np.full(16, 0.0117, np.float32))   # a constant block
    w[6, :] = synth.round_bf16(rng.uniform(-1e-30, 1e-30, 128).astype(np.float32))
    return w


def _gpu_quantize(dev, fmt, w):
    import torch
    W = torch.tensor(w, dtype=torch.bfloat16, device="cuda")
    deq = torch.empty_like(W)
    codes, scales, rs = dev.quantize_matrix(fmt, W, deq=deq)
    torch.cuda.synchronize()
    return (codes.cpu().numpy(), scales.cpu().numpy(), rs.cpu().numpy(),
            deq.float().cpu().numpy())


@pytest.fixture(scope="module")
def layer4b():
    return synth.layer_weights(synth.DORY4B, 3)


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
@pytest.mark.parametrize("which", ["edge", "w_q", "w_down", "w_up"])
def test_quantizer_bit_exact(dev, layer4b, fmt, which):
    w = _edge_matrix() if which == "edge" else layer4b[which]
    codes, scales, rs, deq = _gpu_quantize(dev, fmt, w)
    rows, K = w.shape
    if fmt == quant.MXFP8:
        c, s = quant.quantize_mxfp8(w)
        assert np.array_equal(codes.reshape(rows, K), c)
        assert np.array_equal(scales.reshape(rows, K // 32), s)
        assert np.all(rs == 1.0)
        want = quant.dequantize_mxfp8(c, s)
        assert np.array_equal(deq, want.astype(np.float32))          # exact in bf16
    else:
        c, s, g = quant.quantize_nvfp4(w)
        assert np.all(rs.view(np.uint32) == np.float32(g).view(np.uint32))
        assert np.array_equal(scales.reshape(rows, K // 16), s)
        assert np.array_equal(codes.reshape(rows, K // 2), quant.pack_e2m1(c))
        # q * s is exact in float32; q * s * s_g rounds to float32, then to bf16
        want = synth.round_bf16(quant.dequantize_nvfp4(c, s, g).astype(np.float32))
        assert np.array_equal(deq, want)


def test_quantize_refusals(dev):
    import torch
    L = dev.lib()
    W = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    buf = torch.empty(4096, dtype=torch.uint8, device="cuda")
    P = dev._ptr
    assert L.dory_quantize_matrix(3, P(W), 4, 64, P(buf), P(buf), None, None, None) == dev.DORY_EINVAL
    assert L.dory_quantize_matrix(1, P(W), 4, 48, P(buf), P(buf), None, None, None) == dev.DORY_EINVAL
    assert L.dory_quantize_matrix(2, P(W), 4, 64, P(buf), P(buf), None, None, None) == dev.DORY_EINVAL
    assert L.dory_quantize_matrix(1, dev.ctypes.c_void_p(W.data_ptr() + 2), 4, 64, P(buf), P(buf),
                                  None, None, None) == dev.DORY_EINVAL


def _run_model(dev, shape, w, fmt, mode, k, B, T, D, seed, chunk=0, qw=None, swap=False):
    if qw is None:
        qw, _ = quant.quantize_weights(w, fmt)
    o = oracle.Oracle(shape, qw, dtype=np.float64 if shape.d <= 256 else np.float32)
    m = dev.Model(shape, w, max_batch=B, max_ctx=T + D + 24, max_chunk=max(T, 16), k_max=k,
                  cache_mode=mode)
    m.quantize(fmt)
    m.set_quantized_swap(swap)
    prompt = synth.tokens(shape, B, T, seed=seed)
    r = o.prefill(prompt, k, mode, all_logits=True)
    lg = m.prefill(_tok(prompt), k, mode).cpu().numpy()
    check_logits(lg, r["logits"][:, -1])
    check_hidden(m.hidden(B * T).cpu().numpy(), r["hidden"])
    nxt = np.argmax(r["logits"][:, -1], axis=-1).astype(np.int32)
    for _ in range(D):
        r = o.decode(nxt, k, mode)
        lg, g = m.decode(_tok(nxt), k, mode)
        check_logits(lg.cpu().numpy(), r["logits"])
        check_hidden(m.hidden(B).cpu().numpy(), r["hidden"])
        check_greedy(g.cpu().numpy(), r["logits"])
        nxt = np.argmax(r["logits"], axis=-1).astype(np.int32)
    if chunk:
        # a prefill chunk of B * chunk rows: packed codes up to 4 rows, else
        # the dequantised bf16 copy on the GEMV path
        toks = synth.tokens(shape, B, chunk, seed=seed + 1)
        r = o.prefill(toks, k, mode)
        lg = m.prefill(_tok(toks), k, mode).cpu().numpy()
        check_logits(lg, r["logits"][:, -1])
    assert m.device_status() == 0
    m.close()


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
@pytest.mark.parametrize("mode", [oracle.LAST_LOOP, oracle.PER_LOOP], ids=["last", "perloop"])
def test_quantized_model_tiny(dev, fmt, mode):
    shape = synth.TINY_LOOPFULL                      # window 16: the rings wrap
    w = synth.make_weights(shape)
    qw, _ = quant.quantize_weights(w, fmt)
    _run_model(dev, shape, w, fmt, mode, k=2, B=2, T=21, D=4, seed=31, chunk=2, qw=qw)
    _run_model(dev, shape, w, fmt, mode, k=2, B=3, T=9, D=1, seed=32, chunk=5, qw=qw)


SHAPE_3L = synth.DORY4B_SLIM.replace(n_in=1, n_rec=1, n_out=1)


@pytest.fixture(scope="module")
def weights_3l():
    return synth.make_weights(SHAPE_3L, shape_id=103)


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_quantized_model_4b_width(dev, weights_3l, fmt):
    qw, _ = quant.quantize_weights(weights_3l, fmt)
    _run_model(dev, SHAPE_3L, weights_3l, fmt, oracle.LAST_LOOP, k=2, B=3, T=40, D=2, seed=41,
               chunk=5, qw=qw)
    _run_model(dev, SHAPE_3L, weights_3l, fmt, oracle.PER_LOOP, k=2, B=1, T=24, D=3, seed=42,
               chunk=4, qw=qw)


def test_quantized_switch_back(dev):
    """QUANT_NONE returns the few-row projections to the bf16 matrices,
    which then hold the dequantised weights: the same model."""
    shape = synth.TINY
    w = synth.make_weights(shape)
    qw, _ = quant.quantize_weights(w, quant.MXFP8)
    m = dev.Model(shape, w, max_batch=1, max_ctx=32, max_chunk=16, k_max=1)
    m.quantize(quant.MXFP8)
    m.quantize(dev.QUANT_NONE)
    o = oracle.Oracle(shape, qw)
    tok = synth.tokens(shape, 1, 6, seed=2)
    check_logits(m.prefill(_tok(tok), 1).cpu().numpy(), o.prefill(tok, 1, oracle.LAST_LOOP)["logits"][:, -1])
    nxt = np.array([3], np.int32)
    check_logits(m.decode(_tok(nxt), 1)[0].cpu().numpy(), o.decode(nxt, 1, oracle.LAST_LOOP)["logits"])
    m.close()


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_quantized_batched_decode_equals_dequantised_copy(dev, weights_3l, fmt):
    """20 sequences decode through the swapped tensor-core GEMM, which
    expands the packed codes to bf16 in shared memory: bit for bit the
    results of the same GEMM reading the dequantised bf16 matrices."""
    import torch
    B, T, k = 20, 9, 2
    prompt = synth.tokens(SHAPE_3L, B, T, seed=51)
    a = dev.Model(SHAPE_3L, weights_3l, max_batch=B, max_ctx=64, max_chunk=T, k_max=k)
    b = dev.Model(SHAPE_3L, weights_3l, max_batch=B, max_ctx=64, max_chunk=T, k_max=k)
    a.quantize(fmt)
    a.set_quantized_swap(True)
    b.quantize(fmt)
    b.quantize(dev.QUANT_NONE)                       # the same values, as bf16 matrices
    la, lb = a.prefill(_tok(prompt), k), b.prefill(_tok(prompt), k)
    assert torch.equal(la, lb)
    tok = torch.argmax(la, dim=-1).to(torch.int32)
    for _ in range(3):
        la, ga = a.decode(tok, k)
        lb, gb = b.decode(tok, k)
        assert torch.equal(la, lb) and torch.equal(ga, gb)
        tok = ga
    assert a.device_status() == 0
    a.close()
    b.close()


@pytest.mark.parametrize("fmt", FMTS, ids=IDS)
def test_quantized_batched_decode_4b_width(dev, weights_3l, fmt):
    qw, _ = quant.quantize_weights(weights_3l, fmt)
    _run_model(dev, SHAPE_3L, weights_3l, fmt, oracle.LAST_LOOP, k=2, B=20, T=9, D=2, seed=61,
               qw=qw, swap=True)
