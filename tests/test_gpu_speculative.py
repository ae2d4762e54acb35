"""Greedy self-speculative decoding through the C ABI
("Dory1.0-4B: A Looped Normalized-GPT", Self-Speculative Decoding): drafts at
k_draft, one verifying pass at k_verify = 4 under per-loop caching, greedy
acceptance.  Whatever the drafts, the emitted tokens must be those of plain
greedy decoding at k_verify, so the GPU's emitted tokens are compared with
plain greedy decoding at k_verify, teacher-forced on the emitted tokens: on
the GPU's own decode path (a second handle) the tokens must agree wherever
its top-2 logit margin exceeds 1e-3, and against the oracle wherever the
oracle's margin exceeds three times the measured logit error (near-ties may
go either way), with the logits within the parity tolerance at every step.
After the steps a plain decode step must still match the oracle, which
checks the cache state the steps leave behind, including the sliding-window
ring slots that drafting and the rejected positions overwrite and the step
puts back."""
import numpy as np
import pytest

import oracle
import synth
from test_gpu_parity import check_logits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_ok):
    import looped_normalized_transformer_ngpt_b300 as dory
    from looped_normalized_transformer_ngpt_b300 import _build
    _build.build()
    dory.lib()
    return dory


def _tok(t):
    import torch
    return torch.tensor(np.ascontiguousarray(t), dtype=torch.int32, device="cuda")


def _run(dev, shape, w, B, T, k_draft, gamma, n_tokens, seed):
    kv = 4
    prompt = synth.tokens(shape, B, T, seed=seed)
    cap = dict(max_batch=B, max_ctx=T + n_tokens + 2 * gamma + 8, max_chunk=max(T, gamma + 1),
               k_max=kv, cache_mode=dev.PER_LOOP)
    m = dev.Model(shape, w, **cap)
    plain = dev.Model(shape, w, **cap)
    o = oracle.Oracle(shape, w, dtype=np.float64 if shape.d <= 256 else np.float32)
    z = o.prefill(prompt, kv, oracle.PER_LOOP)["logits"][:, -1]
    lg = m.prefill(_tok(prompt), kv).cpu().numpy()
    plain.prefill(_tok(prompt), kv)
    check_logits(lg, z)
    cur = np.argmax(lg, axis=-1).astype(np.int32)
    emitted, counts = [], []
    while sum(e.shape[1] for e in emitted) < n_tokens:
        out, n = m.speculative_step(_tok(cur), k_draft, kv, gamma)
        out = out.cpu().numpy()
        assert out.shape == (B, n) and 1 <= n <= gamma + 1
        emitted.append(out)
        counts.append(n)
        cur = out[:, -1]
    assert m.device_status() == 0
    emitted = np.concatenate(emitted, axis=1)
    # plain greedy decoding at k_verify, fed the speculative tokens (teacher
    # forcing keeps every side on the same history): on the GPU's own decode
    # path the tokens must agree wherever its top-2 margin exceeds 1e-3 (the
    # decode and verifying paths round differently by ~1e-4); against the
    # oracle the logits must agree within the tolerance, and the greedy token
    # wherever the oracle's margin exceeds three times the measured logit
    # error (the verifying path rounds differently from the decode path)
    prev = np.argmax(lg, axis=-1).astype(np.int32)
    n_exact = n_oracle = 0
    for j in range(emitted.shape[1]):
        zg = plain.decode(_tok(prev), kv)[0].cpu().numpy()
        zo = o.decode(prev, kv, oracle.PER_LOOP)["logits"]
        check_logits(zg, zo)
        err = np.max(np.abs(zg - zo))
        for zz, thr in ((zg, 1e-3), (zo, 3 * err)):
            top2 = np.sort(zz, axis=-1)[:, -2:]
            clear = (top2[:, 1] - top2[:, 0]) > thr
            assert np.all((emitted[:, j] == np.argmax(zz, axis=-1)) | ~clear), (j, thr)
            if thr == 1e-3:
                n_exact += int(clear.sum())
            else:
                n_oracle += int(clear.sum())
        prev = emitted[:, j]
    # enough clear positions that the comparison means something (the
    # 131072-entry vocabulary has smaller top-2 gaps than the tiny one's)
    assert n_exact >= 0.6 * emitted.size and n_oracle >= 0.5 * emitted.size, (n_exact, n_oracle)
    # the state continues like plain decoding: one more step on both sides
    lg2, _ = m.decode(_tok(emitted[:, -1]), kv)
    check_logits(lg2.cpu().numpy(), o.decode(emitted[:, -1], kv, oracle.PER_LOOP)["logits"])
    assert m.length() == T + emitted.shape[1] + 1
    plain.close()
    return counts, m


@pytest.mark.parametrize("k_draft,gamma", [(1, 4), (2, 3), (4, 4)])
def test_speculative_matches_plain_greedy_tiny(dev, k_draft, gamma):
    shape = synth.TINY_LOOPFULL                      # window 16: the rings wrap
    w = synth.make_weights(shape)
    counts, m = _run(dev, shape, w, B=2, T=21, k_draft=k_draft, gamma=gamma, n_tokens=24, seed=7)
    if k_draft == 4:
        # a drafter as deep as the verifier: nearly every draft is accepted
        # (a near-tie between the decode and the verifying path may reject one)
        assert np.mean(counts) >= 0.75 * (gamma + 1), counts
    m.close()


def test_speculative_matches_plain_greedy_4b_width(dev):
    shape = synth.DORY4B_SLIM
    w = synth.make_weights(shape)
    counts, m = _run(dev, shape, w, B=1, T=70, k_draft=1, gamma=4, n_tokens=16, seed=8)
    m.close()


def test_speculative_refusals(dev):
    import torch
    shape = synth.TINY_LOOPFULL
    w = synth.make_weights(shape)
    L = dev.lib()
    last = dev.Model(shape, w, max_batch=1, max_ctx=40, max_chunk=8, k_max=4)
    last.prefill(_tok(synth.tokens(shape, 1, 5)), 4)
    with pytest.raises(dev.DoryError) as e:
        last.speculative_step(_tok(np.array([1])), 1, 4, 4)
    assert e.value.code == dev.DORY_EKMISMATCH
    m = dev.Model(shape, w, max_batch=1, max_ctx=12, max_chunk=4, k_max=4,
                  cache_mode=dev.PER_LOOP)
    m.prefill(_tok(synth.tokens(shape, 1, 5)), 4)
    for kd, kv, g in ((5, 4, 2), (0, 4, 2), (1, 4, 0), (1, 4, 17)):
        with pytest.raises(dev.DoryError):
            m.speculative_step(_tok(np.array([1])), kd, kv, g)
    with pytest.raises(dev.DoryError) as e:            # gamma + 1 > max_chunk
        m.speculative_step(_tok(np.array([1])), 1, 4, 4)
    assert e.value.code == dev.DORY_ECAPACITY
    nb = L.dory_speculative_scratch_bytes(m.handle, 1, 2)
    small = torch.empty(nb - 256, dtype=torch.uint8, device="cuda")
    out = torch.empty((1, 3), dtype=torch.int32, device="cuda")
    n = dev.ctypes.c_int()
    rc = L.dory_speculative_step(m.handle, dev._ptr(_tok(np.array([1]))), 1, 1, 4, 2,
                                 dev._ptr(small), nb - 256, dev._ptr(out), dev.ctypes.byref(n),
                                 None)
    assert rc == dev.DORY_ENOMEM
    assert m.length() == 5
    m.close()
    last.close()
