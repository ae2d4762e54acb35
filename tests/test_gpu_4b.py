"""Parity at the 4B-class width (d 2048, 16 q / 4 kv heads of 128, SwiGLU
6144, vocab 131072, window 4096) through the C ABI, against the float32
oracle on the same seeded inputs.

The depth is cut to 2 / 4 / 2 layers (the full layers 3 and 7 sit in the
recurrent and output blocks) so that the oracle finishes in seconds; every
projection, head and the whole vocabulary keep their full width, so the
GEMM tiles, attention head groups and LM-head grid are those of the
4B-class workloads:

* prefill of one ragged-length sequence (the 1 x 8192 prefill workload's
  path) at k = 1, 2, 4;
* batched decode of 64 sequences (the 64 x 32768 decode workload's path:
  more rows than the few-row GEMV handles) at k = 1, 2, 3, 4;
* chunked prefill with a ragged last chunk, then decode, in both cache modes
  at k = 4 (the long-context workload's path).

Tolerances as in test_gpu_parity."""
import numpy as np
import pytest

import oracle
import synth
from test_gpu_parity import check_greedy, check_hidden, check_logits, _tok

pytestmark = pytest.mark.gpu

SHAPE = synth.DORY4B_SLIM


@pytest.fixture(scope="module")
def dev(cuda_ok):
    import looped_normalized_transformer_ngpt_b300 as dory
    from looped_normalized_transformer_ngpt_b300 import _build
    _build.build()
    dory.lib()
    return dory


@pytest.fixture(scope="module")
def weights():
    return synth.make_weights(SHAPE)


@pytest.fixture(scope="module")
def model_last(dev, weights):
    # a capacity of a multiple of 64 positions: the decode steps run the TMA-fed
    # decode attention (its inputs here are split-K partial sums)
    return dev.Model(SHAPE, weights, max_batch=64, max_ctx=448, max_chunk=400, k_max=4,
                     cache_mode=dev.LAST_LOOP)


@pytest.mark.parametrize("k", [1, 2, 4])
def test_4b_width_prefill_ragged(dev, weights, model_last, k):
    B, T = 1, 333                     # 2 full 128-row tiles + a ragged tail
    prompt = synth.tokens(SHAPE, B, T, seed=20 + k)
    m = model_last
    m.reset()
    lg = m.prefill(_tok(prompt), k).cpu().numpy()
    hid = m.hidden(B * T).cpu().numpy()
    assert m.device_status() == 0
    ref = oracle.Oracle(SHAPE, weights, dtype=np.float32).prefill(prompt, k, oracle.LAST_LOOP,
                                                                  all_logits=True)
    check_logits(lg, ref["logits"][:, -1])
    check_hidden(hid.reshape(B, T, SHAPE.d), ref["hidden"])


@pytest.mark.parametrize("k", [1, 2, 3, 4])
def test_4b_width_batched_decode_64(dev, weights, model_last, k):
    B, T, D = 64, 16, 2
    prompt = synth.tokens(SHAPE, B, T, seed=30 + k)
    dec = synth.tokens(SHAPE, B, D, seed=40 + k)
    m = model_last
    m.reset()
    o = oracle.Oracle(SHAPE, weights, dtype=np.float32)
    r = o.prefill(prompt, k, oracle.LAST_LOOP)
    lg = m.prefill(_tok(prompt), k)
    check_logits(lg.cpu().numpy(), r["logits"][:, -1])
    for s in range(D):
        r = o.decode(dec[:, s], k, oracle.LAST_LOOP)
        lg, nxt = m.decode(_tok(dec[:, s]), k)
        check_logits(lg.cpu().numpy(), r["logits"])
        check_hidden(m.hidden(B).cpu().numpy(), r["hidden"])
        check_greedy(nxt.cpu().numpy(), r["logits"])
    assert m.device_status() == 0


@pytest.mark.parametrize("mode", [oracle.LAST_LOOP, oracle.PER_LOOP], ids=["last", "perloop"])
def test_4b_width_chunked_prefill_then_decode(dev, weights, mode):
    k, B, T, chunk, D = 4, 2, 300, 128, 3
    prompt = synth.tokens(SHAPE, B, T, seed=50)
    dec = synth.tokens(SHAPE, B, D, seed=51)
    o = oracle.Oracle(SHAPE, weights, dtype=np.float32)
    for c0 in range(0, T, chunk):
        ref = o.prefill(prompt[:, c0:c0 + chunk], k, mode)
    m = dev.Model(SHAPE, weights, max_batch=B, max_ctx=(T + D + 63) // 64 * 64, max_chunk=chunk,
                  k_max=k, cache_mode=mode)
    lg = m.prefill(_tok(prompt), k, mode)
    check_logits(lg.cpu().numpy(), ref["logits"][:, -1])
    for s in range(D):
        r = o.decode(dec[:, s], k, mode)
        lg, nxt = m.decode(_tok(dec[:, s]), k, mode)
        check_logits(lg.cpu().numpy(), r["logits"])
        check_hidden(m.hidden(B).cpu().numpy(), r["hidden"])
        check_greedy(nxt.cpu().numpy(), r["logits"])
    assert m.device_status() == 0
    m.close()


@pytest.mark.parametrize("B", [5, 16])
def test_4b_width_few_row_decode(dev, weights, model_last, B):
    """Decode batches of 5 and 16 sequences: the swapped tensor-core GEMM with
    a part-filled activation operand (rows past B read as zeros): the
    4B-width model at k = 2, two decode steps after a short prefill, against
    the oracle."""
    k, T, D = 2, 24, 2
    prompt = synth.tokens(SHAPE, B, T, seed=60 + B)
    dec = synth.tokens(SHAPE, B, D, seed=70 + B)
    m = model_last
    m.reset()
    o = oracle.Oracle(SHAPE, weights, dtype=np.float32)
    r = o.prefill(prompt, k, oracle.LAST_LOOP)
    lg = m.prefill(_tok(prompt), k)
    check_logits(lg.cpu().numpy(), r["logits"][:, -1])
    for s in range(D):
        r = o.decode(dec[:, s], k, oracle.LAST_LOOP)
        lg, nxt = m.decode(_tok(dec[:, s]), k)
        check_logits(lg.cpu().numpy(), r["logits"])
        check_hidden(m.hidden(B).cpu().numpy(), r["hidden"])
        check_greedy(nxt.cpu().numpy(), r["logits"])
    assert m.device_status() == 0
