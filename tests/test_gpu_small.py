"""Parity on the benchmark shape (small looped nGPT: d 1024, 4/10/4 layers,
8 q / 2 kv heads, head_dim 128, SwiGLU 2816, vocab 32000, window 512).

* Full-size prefill in the launch configuration the benchmark times
  (4 x 2048 tokens, one chunk, last-loop cache): the GPU processes the whole
  batch; sequences are independent, so two sampled sequences are checked
  against the float32 oracle run on those sequences alone, at every position.
* Decode steps after a short prefill: few-row GEMVs with split K segments
  and the fused SwiGLU pair, and the split-key decode attention.
Tolerances as in test_gpu_parity."""
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


@pytest.fixture(scope="module")
def weights():
    return synth.make_weights(synth.SMALL)


@pytest.mark.parametrize("k", [1, 2, 4])
def test_full_size_prefill_sampled_sequences(dev, weights, k):
    sh = synth.SMALL
    B, T = 4, 2048
    prompt = synth.tokens(sh, B, T, seed=1000)
    m = dev.Model(sh, weights, max_batch=B, max_ctx=T + 8, max_chunk=T, k_max=4,
                  cache_mode=dev.LAST_LOOP)
    lg = m.prefill(_tok(prompt), k).cpu().numpy()
    hid = m.hidden(B * T).cpu().numpy().reshape(B, T, sh.d)
    assert m.device_status() == 0
    for b in (0, 3):
        o = oracle.Oracle(sh, weights, dtype=np.float32)
        ref = o.prefill(prompt[b:b + 1], k, oracle.LAST_LOOP, all_logits=False)
        check_logits(lg[b:b + 1], ref["logits"][:, -1])
        check_hidden(hid[b:b + 1, -1:], ref["hidden"])
    # every position of one sequence
    o = oracle.Oracle(sh, weights, dtype=np.float32)
    ref = o.prefill(prompt[1:2], k, oracle.LAST_LOOP, all_logits=True)
    check_hidden(hid[1:2], ref["hidden"])


@pytest.mark.parametrize("k,mode", [(2, oracle.LAST_LOOP), (3, oracle.PER_LOOP)])
@pytest.mark.parametrize("max_ctx", [99, 128], ids=["ring99", "ring128"])
def test_decode_steps(dev, weights, k, mode, max_ctx):
    """A cache capacity of 99 positions runs the cp.async decode attention; 128
    (a multiple of 64) the TMA-fed one that the benchmark times."""
    sh = synth.SMALL
    B, T, D = 3, 96, 3
    prompt = synth.tokens(sh, B, T, seed=7)
    dec = synth.tokens(sh, B, D, seed=8)
    o = oracle.Oracle(sh, weights, dtype=np.float32)
    m = dev.Model(sh, weights, max_batch=B, max_ctx=max_ctx, max_chunk=T, k_max=k, cache_mode=mode)
    r = o.prefill(prompt, k, mode)
    lg = m.prefill(_tok(prompt), k, mode)
    check_logits(lg.cpu().numpy(), r["logits"][:, -1])
    for s in range(D):
        r = o.decode(dec[:, s], k, mode)
        lg, nxt = m.decode(_tok(dec[:, s]), k, mode)
        check_logits(lg.cpu().numpy(), r["logits"])
        check_hidden(m.hidden(B).cpu().numpy(), r["hidden"])
        check_greedy(nxt.cpu().numpy(), r["logits"])
    assert m.device_status() == 0
