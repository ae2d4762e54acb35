"""Temperature sampling and self-speculative rejection sampling through the
C ABI ("Dory1.0-4B: A Looped Normalized-GPT", Self-Speculative Decoding).

A sampled token is an integer decided in floating point, and the GPU's
logits differ from the oracle's by the parity tolerance, so the two parts
are checked separately:
* the decisions: given the GPU's own logits (read back from the step's
  scratch) and the same uniforms, every draw and every acceptance test must
  equal the oracle's rule (oracle/sampling.py), except where the oracle's
  decision margin is below 1e-4 (float32 against float64 rounding);
* the logits: the verifier's rows at the emitted positions against the
  oracle decoding the emitted tokens at k_verify (teacher forcing), the
  drafter's rows of the first step against the oracle drafting the same
  tokens at k_draft, and one plain decode step after the steps (the cache
  state the steps leave), within the parity tolerances."""
import copy

import numpy as np
import pytest

import oracle
import synth
from oracle import sampling
from test_gpu_parity import check_logits

pytestmark = pytest.mark.gpu

MARGIN = 1e-4


@pytest.fixture(scope="module")
def dev(cuda_ok):
    import looped_normalized_transformer_ngpt_b300 as dory
    from looped_normalized_transformer_ngpt_b300 import _build
    _build.build()
    dory.lib()
    return dory


def _dev_f32(x):
    import torch
    return torch.tensor(np.ascontiguousarray(x, np.float32), device="cuda")


def _tok(t):
    import torch
    return torch.tensor(np.ascontiguousarray(t), dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("V", [512, 32000, 131072])
@pytest.mark.parametrize("temperature", [0.6, 1.0, 2.5])
def test_sample_tokens_matches_oracle(dev, V, temperature):
    rng = np.random.default_rng(V + int(10 * temperature))
    rows = 96
    z = (rng.standard_normal((rows, V)) * 3).astype(np.float32)
    z[0, :] = 0.0                                    # uniform distribution
    z[1, 7] = 60.0                                   # one dominant token
    u = rng.random(rows).astype(np.float32)
    u[2], u[3] = 0.0, np.float32(0.99999994)         # the two ends
    got = dev.sample_tokens(_dev_f32(z), temperature, _dev_f32(u)).cpu().numpy()
    p = sampling.softmax_t(z.astype(np.float64), temperature)
    bad = 0
    for r in range(rows):
        marg = []
        want = sampling.sample_weights(p[r], float(u[r]), marg)
        if got[r] != want:
            assert marg[0] < MARGIN, (r, got[r], want, marg)
            bad += 1
    assert bad <= 2
    assert got[1] == 7


def _scratch_views(dev, m, B, gamma, V):
    """The step's verifier logits [B, gamma + 1, V], drafter logits
    [B, gamma, V] and drafts [B, gamma], read from its scratch."""
    import ctypes
    import torch
    offs = (ctypes.c_size_t * 3)()
    assert dev.lib().dory_debug_speculative_layout(m.handle, B, gamma, offs) == 0
    sc = m._spec_scratch
    zp = sc[offs[0]:offs[0] + B * (gamma + 1) * V * 4].view(torch.float32)
    zq = sc[offs[1]:offs[1] + gamma * B * V * 4].view(torch.float32)
    dr = sc[offs[2]:offs[2] + gamma * B * 4].view(torch.int32)
    return (zp.cpu().numpy().reshape(B, gamma + 1, V).astype(np.float64),
            zq.cpu().numpy().reshape(gamma, B, V).transpose(1, 0, 2).astype(np.float64),
            dr.cpu().numpy().reshape(gamma, B).T)


def _check_decisions(p, q, drafts, u, kept, out, n, gamma):
    """Every decision of the GPU's step equals the rule's on the same logits
    and uniforms, or the rule's margin for that decision is below MARGIN
    (and later decisions of that sequence are not compared).  Returns
    whether the whole step matched."""
    B = drafts.shape[0]
    exact = True
    for b in range(B):
        for i in range(gamma):
            marg = []
            want = sampling.sample_weights(q[b, i], u[b, i], marg)
            if drafts[b, i] != want:
                assert marg[0] < MARGIN, ("draft", b, i, marg)
                exact = False
        for i in range(gamma):
            x = drafts[b, i]
            keep = u[b, gamma + i] * q[b, i, x] < p[b, i, x]
            if keep != (i < kept[b]):
                assert abs(u[b, gamma + i] * q[b, i, x] - p[b, i, x]) / p[b, i, x] < MARGIN, \
                    ("keep", b, i)
                exact = False
                break
            if not keep:
                break
    if not exact:
        return False
    want_out, want_n, want_kept = sampling.speculative_accept(p, q, drafts, u[:, gamma:2 * gamma],
                                                              u[:, 2 * gamma])
    assert want_n == n and np.array_equal(want_kept, kept)
    assert np.array_equal(want_out[:, :n - 1], out[:, :n - 1])
    for b in range(B):
        if want_out[b, n - 1] != out[b, n - 1]:
            assert kept[b] <= n - 1, ("a kept draft must be emitted as is", b)
            j = n - 1
            w = np.maximum(p[b, j] - q[b, j], 0.0) if j < gamma else p[b, gamma]
            marg = []
            sampling.sample_weights(w, u[b, 2 * gamma], marg)
            assert marg[0] < MARGIN, ("draw", b, marg)
            exact = False
    return exact


def _run(dev, shape, w, B, T, k_draft, gamma, temperature, steps, seed):
    kv = 4
    prompt = synth.tokens(shape, B, T, seed=seed)
    m = dev.Model(shape, w, max_batch=B, max_ctx=T + steps * (gamma + 1) + 2 * gamma + 8,
                  max_chunk=max(T, gamma + 1), k_max=kv, cache_mode=dev.PER_LOOP)
    o = oracle.Oracle(shape, w, dtype=np.float64 if shape.d <= 256 else np.float32)
    z0 = o.prefill(prompt, kv, oracle.PER_LOOP)["logits"][:, -1]
    lg = m.prefill(_tok(prompt), kv).cpu().numpy()
    check_logits(lg, z0)
    rng = np.random.default_rng(seed)
    cur = np.argmax(lg, axis=-1).astype(np.int32)
    V = shape.vocab
    kept_all, checked, skipped = [], 0, 0
    for step in range(steps):
        u = rng.random((B, 2 * gamma + 1)).astype(np.float32)
        state = copy.deepcopy(o) if step == 0 else None
        out, n, kept = m.speculative_sample_step(_tok(cur), k_draft, kv, gamma, temperature,
                                                 _dev_f32(u))
        out, kept = out.cpu().numpy(), kept.cpu().numpy()
        zp, zq, drafts = _scratch_views(dev, m, B, gamma, V)
        assert out.shape == (B, n) and 1 <= n <= gamma + 1 and n == kept.min() + 1
        # decisions on the GPU's own logits
        q = sampling.softmax_t(zq, temperature)
        p = sampling.softmax_t(zp, temperature)
        if _check_decisions(p, q, drafts, u.astype(np.float64), kept, out, n, gamma):
            checked += 1
        else:
            skipped += 1
        # the drafter's logits of the first step: the oracle drafting the same tokens
        if state is not None:
            tok = cur
            for i in range(gamma):
                h = state.step(tok.reshape(-1, 1), k_draft, oracle.PER_LOOP, draft=True)[:, 0]
                check_logits(zq[:, i], state.logits(h))
                tok = drafts[:, i]
        # the verifier's logits at the emitted positions: the oracle decoding
        # the emitted tokens at k_verify
        prev = cur
        for j in range(n):
            r = o.decode(prev, kv, oracle.PER_LOOP)
            check_logits(zp[:, j], r["logits"])
            prev = out[:, j]
        kept_all.append(kept)
        cur = out[:, -1].astype(np.int32)
    assert m.device_status() == 0
    assert checked >= steps // 2, (checked, skipped)
    lg2, _ = m.decode(_tok(cur), kv)
    check_logits(lg2.cpu().numpy(), o.decode(cur, kv, oracle.PER_LOOP)["logits"])
    m.close()
    return np.array(kept_all)


@pytest.mark.parametrize("k_draft,gamma,temperature", [(1, 4, 1.0), (2, 3, 0.7), (1, 2, 2.0)])
def test_speculative_sampling_tiny(dev, k_draft, gamma, temperature):
    shape = synth.TINY_LOOPFULL                      # window 16: the rings wrap
    _run(dev, shape, synth.make_weights(shape), B=2, T=21, k_draft=k_draft, gamma=gamma,
         temperature=temperature, steps=6, seed=50 + gamma)


def test_speculative_sampling_deep_drafter_keeps_drafts(dev):
    shape = synth.TINY_LOOPFULL
    kept = _run(dev, shape, synth.make_weights(shape), B=2, T=15, k_draft=4, gamma=3,
                temperature=1.0, steps=5, seed=61)
    assert kept.mean() >= 0.9 * 3, kept


def test_speculative_sampling_4b_width(dev):
    shape = synth.DORY4B_SLIM
    _run(dev, shape, synth.make_weights(shape), B=1, T=40, k_draft=1, gamma=4, temperature=0.8,
         steps=3, seed=70)


def test_sampling_refusals(dev):
    import torch
    shape = synth.TINY_LOOPFULL
    m = dev.Model(shape, synth.make_weights(shape), max_batch=1, max_ctx=40, max_chunk=8, k_max=4,
                  cache_mode=dev.PER_LOOP)
    m.prefill(_tok(synth.tokens(shape, 1, 5)), 4)
    u = torch.zeros((1, 9), dtype=torch.float32, device="cuda")
    with pytest.raises(dev.DoryError):
        m.speculative_sample_step(_tok(np.array([1])), 1, 4, 4, 0.0, u)
    L = dev.lib()
    z = torch.zeros((2, 16), dtype=torch.float32, device="cuda")
    o = torch.zeros(2, dtype=torch.int32, device="cuda")
    assert L.dory_sample_tokens(dev._ptr(z), 2, 16, 0.0, dev._ptr(u), dev._ptr(o), None) == dev.DORY_EINVAL
    assert L.dory_sample_tokens(dev._ptr(z), 2, 16, 1.0, None, dev._ptr(o), None) == dev.DORY_EINVAL
    assert m.length() == 5
    m.close()
