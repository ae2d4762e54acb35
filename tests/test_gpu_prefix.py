"""Prefix caching through the C ABI (dory_copy_prefix): a shared prompt is
prefilled once on one sequence, its cached keys and values are copied into
the other sequences, and all of them continue with their own suffixes and
decode steps.  Each sequence must match the oracle run on prompt + its own
suffix, in both cache modes and at k = 1 and 2 (tolerances as in
test_gpu_parity); the window layers' rings wrap on the tiny shape (window
16, prompt 40)."""
import numpy as np
import pytest

import oracle
import synth
from test_gpu_parity import check_greedy, check_hidden, check_logits, _tok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_ok):
    import looped_normalized_transformer_ngpt_b300 as dory
    from looped_normalized_transformer_ngpt_b300 import _build
    _build.build()
    dory.lib()
    return dory


@pytest.mark.parametrize("shape", [synth.TINY_LOOPFULL, synth.DORY4B_SLIM], ids=lambda s: s.name)
@pytest.mark.parametrize("mode", [oracle.LAST_LOOP, oracle.PER_LOOP], ids=["last", "perloop"])
@pytest.mark.parametrize("k", [1, 2])
def test_shared_prefix_then_own_suffixes(dev, shape, mode, k):
    B, P, T2, D = 3, 40, 9, 2
    w = synth.make_weights(shape)
    prompt = synth.tokens(shape, 1, P, seed=11)
    suffix = synth.tokens(shape, B, T2, seed=12)
    dec = synth.tokens(shape, B, D, seed=13)
    m = dev.Model(shape, w, max_batch=B, max_ctx=P + T2 + D + 8, max_chunk=P, k_max=k,
                  cache_mode=mode)
    m.prefill(_tok(prompt), k, mode)                  # the prompt once, on sequence 0
    m.copy_prefix(0, list(range(1, B)), P)
    m.set_length(B, P)
    o = oracle.Oracle(shape, w, dtype=np.float64 if shape.d <= 256 else np.float32)
    o.prefill(np.repeat(prompt, B, axis=0), k, mode)
    r = o.prefill(suffix, k, mode, all_logits=True)
    lg = m.prefill(_tok(suffix), k, mode, all_logits=True)
    check_logits(lg.cpu().numpy(), r["logits"])
    check_hidden(m.hidden(B * T2).cpu().numpy(), r["hidden"])
    for s in range(D):
        r = o.decode(dec[:, s], k, mode)
        lg, nxt = m.decode(_tok(dec[:, s]), k, mode)
        check_logits(lg.cpu().numpy(), r["logits"])
        check_greedy(nxt.cpu().numpy(), r["logits"])
    assert m.device_status() == 0
    m.close()


def test_copy_prefix_refusals(dev):
    shape = synth.TINY
    m = dev.Model(shape, synth.make_weights(shape), max_batch=3, max_ctx=16, max_chunk=8)
    for src, dst, n in ((0, [0], 4), (0, [3], 4), (-1, [1], 4), (0, [1], 17), (0, [1], 0)):
        with pytest.raises(dev.DoryError):
            m.copy_prefix(src, dst, n)
    m.close()
