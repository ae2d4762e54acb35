"""Pins of the oracle's temperature sampling and self-speculative rejection
sampling (oracle/sampling.py, Oracle.speculative_sample_step; "Dory1.0-4B: A
Looped Normalized-GPT", Self-Speculative Decoding).  Anchors: closed forms
of the inverse-CDF draw and of softmax at temperature T; the defining
property of rejection sampling (every emitted token is distributed as the
verifier's distribution), checked by Monte Carlo; the batch rule against
each sequence alone; a drafter as deep as the verifier keeps every draft;
near-zero temperature reduces to greedy self-speculative decoding."""
import copy

import numpy as np
import pytest

import oracle
import synth
from oracle import sampling


def test_sample_weights_boundaries():
    p = np.array([0.25, 0.25, 0.5])
    got = [sampling.sample_weights(p, u) for u in (0.0, 0.2499, 0.25, 0.4999, 0.5, 0.9999)]
    assert got == [0, 0, 1, 1, 2, 2]
    w = np.array([0.0, 2.0, 0.0, 2.0, 0.0])                 # zero weights are never drawn
    assert [sampling.sample_weights(w, u) for u in (0.0, 0.49, 0.5, 0.99)] == [1, 1, 3, 3]


def test_softmax_temperature_closed_form():
    p = np.array([0.1, 0.2, 0.3, 0.4])
    z = np.log(p) + 3.0
    np.testing.assert_allclose(sampling.softmax_t(z, 1.0), p, rtol=1e-12)
    np.testing.assert_allclose(sampling.softmax_t(z, 0.5), p ** 2 / np.sum(p ** 2), rtol=1e-12)
    np.testing.assert_allclose(sampling.softmax_t(z, 2.0), np.sqrt(p) / np.sum(np.sqrt(p)),
                               rtol=1e-12)


def test_sample_tokens_frequencies():
    rng = np.random.default_rng(3)
    z = rng.standard_normal(6)
    p = sampling.softmax_t(z, 0.7)
    N = 40000
    toks = sampling.sample_tokens(np.repeat(z[None], N, 0), 0.7, rng.random(N))
    freq = np.bincount(toks, minlength=6) / N
    assert np.all(np.abs(freq - p) <= 5 * np.sqrt(p * (1 - p) / N))


def test_rejection_sampling_keeps_the_verifier_distribution():
    """Monte Carlo over drafts and uniforms: the first emitted token follows
    p_0, the second (when emitted) p_1, the third p_2, whatever q is."""
    rng = np.random.default_rng(11)
    G, V, N = 2, 5, 60000
    p = rng.dirichlet(np.ones(V), G + 1)
    q = rng.dirichlet(np.ones(V) * 0.7, G)
    counts = np.zeros((G + 1, V))
    seen = np.zeros(G + 1)
    for _ in range(N):
        u = rng.random(2 * G + 1)
        drafts = np.array([[sampling.sample_weights(q[i], u[i]) for i in range(G)]])
        out, n, _ = sampling.speculative_accept(p[None], q[None], drafts, u[None, G:2 * G],
                                                u[None, 2 * G:])
        for j in range(n):
            counts[j, out[0, j]] += 1
            seen[j] += 1
    for j in range(G + 1):
        freq = counts[j] / seen[j]
        assert np.all(np.abs(freq - p[j]) <= 5 * np.sqrt(p[j] * (1 - p[j]) / seen[j])), (j, freq, p[j])
    # the acceptance rate of the first draft is sum_x min(p, q)
    assert abs(seen[1] / N - np.minimum(p[0], q[0]).sum()) <= 5 * np.sqrt(0.25 / N)


def test_batch_rule_against_each_sequence_alone():
    rng = np.random.default_rng(5)
    G, V = 4, 7
    for _ in range(200):
        B = 3
        p = rng.dirichlet(np.ones(V), (B, G + 1))
        q = rng.dirichlet(np.ones(V), (B, G))
        u = rng.random((B, 2 * G + 1))
        drafts = np.array([[sampling.sample_weights(q[b, i], u[b, i]) for i in range(G)]
                           for b in range(B)])
        out, n, kept = sampling.speculative_accept(p, q, drafts, u[:, G:2 * G], u[:, 2 * G])
        assert n == kept.min() + 1
        for b in range(B):
            alone, na, ka = sampling.speculative_accept(p[b:b + 1], q[b:b + 1], drafts[b:b + 1],
                                                        u[b:b + 1, G:2 * G], u[b:b + 1, 2 * G])
            assert ka[0] == kept[b] and na == kept[b] + 1 and na >= n
            # the batch emits a prefix of what the sequence alone emits
            assert np.array_equal(out[b], alone[0, :n])


def _prefilled(shape, w, B, T, k, seed):
    o = oracle.Oracle(shape, w)
    o.prefill(synth.tokens(shape, B, T, seed=seed), k, oracle.PER_LOOP)
    return o


def test_draft_as_deep_as_verifier_keeps_every_draft():
    shape = synth.TINY_LOOPFULL
    w = synth.make_weights(shape)
    o = _prefilled(shape, w, 2, 11, 4, seed=3)
    rng = np.random.default_rng(0)
    cur = np.array([5, 9])
    for _ in range(3):
        out, n, kept = o.speculative_sample_step(cur, 4, 4, 3, 0.8, rng.random((2, 7)))
        assert n == 4 and np.all(kept == 3)
        cur = out[:, -1]


def test_low_temperature_is_greedy_speculative():
    """At T = 1e-4 every distribution is one-hot on its greedy token (the
    tiny model's top-2 logit gaps are far above T), so sampling with any
    uniforms emits what greedy self-speculative decoding emits."""
    shape = synth.TINY_LOOPFULL
    w = synth.make_weights(shape)
    a = _prefilled(shape, w, 2, 13, 4, seed=4)
    b = copy.deepcopy(a)
    rng = np.random.default_rng(1)
    cur_a = cur_b = np.array([3, 17])
    for _ in range(4):
        ga, na = a.speculative_step(cur_a, 1, 4, 3)
        gb, nb, _ = b.speculative_sample_step(cur_b, 1, 4, 3, 1e-4, rng.random((2, 7)))
        assert na == nb and np.array_equal(ga, gb)
        cur_a, cur_b = ga[:, -1], gb[:, -1]


def test_sample_step_refusals():
    shape = synth.TINY_LOOPFULL
    w = synth.make_weights(shape)
    o = _prefilled(shape, w, 1, 5, 4, seed=2)
    for args in ((1, 4, 2, 0.0), (5, 4, 2, 1.0), (1, 3, 2, 1.0), (1, 4, 0, 1.0)):
        with pytest.raises(ValueError):
            o.speculative_sample_step(np.array([1]), *args, np.zeros((1, 5)))
