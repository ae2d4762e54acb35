"""The nGPT step fused into the prefill output / down GEMM epilogues
(thread-block clusters of d / 256 CTAs, row norms summed through distributed
shared memory) against the unfused path (GEMM + row kernel) and the oracle.

* the fused path is the one that runs (no row-kernel launch in the prefill);
* fused and unfused give the same hidden states and logits up to rounding
  order, on the small shape (clusters of 4) and the 4B-class width (clusters
  of 8, slim depth), with a ragged row count (not a multiple of 128);
* the fused prefill matches the float32 oracle within the parity tolerances.
"""
import numpy as np
import pytest

import oracle
import synth
from test_gpu_parity import check_hidden, check_logits, _tok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_ok):
    import looped_normalized_transformer_ngpt_b300 as dory
    from looped_normalized_transformer_ngpt_b300 import _build
    _build.build()
    dory.lib()
    return dory


def _run(dev, sh, weights, prompt, k, fused):
    B, T = prompt.shape
    m = dev.Model(sh, weights, max_batch=B, max_ctx=T + 8, max_chunk=T, k_max=4,
                  cache_mode=dev.LAST_LOOP)
    m.set_fused_ngpt(fused)
    m.profile_begin(1 << 14)
    lg = m.prefill(_tok(prompt), k)
    prof = m.profile_end()
    hid = m.hidden(B * T).cpu().numpy()
    assert m.device_status() == 0
    m.close()
    return lg.cpu().numpy(), hid, prof


@pytest.mark.parametrize("shape_name,B,T", [("small", 2, 300), ("slim4b", 1, 200)])
def test_fused_matches_unfused(dev, shape_name, B, T):
    sh = synth.SMALL if shape_name == "small" else synth.DORY4B_SLIM
    weights = synth.make_weights(sh)
    prompt = synth.tokens(sh, B, T, seed=77)
    lg_f, hid_f, prof_f = _run(dev, sh, weights, prompt, 2, True)
    lg_u, hid_u, prof_u = _run(dev, sh, weights, prompt, 2, False)
    assert prof_f["ngpt_update"][1] == 0, prof_f["ngpt_update"]
    assert prof_u["ngpt_update"][1] > 0
    assert np.abs(hid_f - hid_u).max() < 5e-3
    cos = (hid_f * hid_u).sum(-1) / (np.linalg.norm(hid_f, axis=-1) * np.linalg.norm(hid_u, axis=-1))
    assert cos.min() > 0.9999
    assert np.abs(lg_f - lg_u).max() < 1e-2


@pytest.mark.parametrize("k", [1, 4])
def test_fused_prefill_matches_oracle(dev, k):
    sh = synth.SMALL
    weights = synth.make_weights(sh)
    B, T = 2, 200
    prompt = synth.tokens(sh, B, T, seed=78)
    lg, hid, prof = _run(dev, sh, weights, prompt, k, True)
    assert prof["ngpt_update"][1] == 0
    hid = hid.reshape(B, T, sh.d)
    for b in range(B):
        # a fresh oracle per sequence (its prefill continues the sequence it holds)
        o = oracle.Oracle(sh, weights, dtype=np.float32)
        ref = o.prefill(prompt[b:b + 1], k, oracle.LAST_LOOP, all_logits=False)
        check_logits(lg[b:b + 1], ref["logits"][:, -1])
        check_hidden(hid[b:b + 1, -1:], ref["hidden"])
