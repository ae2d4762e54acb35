"""Pins for the CPU oracle: closed forms, special cases and invariants that
the model description fixes, each checked against something other than the
oracle's own formula.  No GPU.

Sources ("Dory1.0-4B: A Looped Normalized-GPT"): Architecture (nGPT update,
normalisations, gate, GQA, 3:1 interleave), Training with Loops (schedule,
32 + 40k layer applications), Last-Loop KV Caching (cache policies, their
coincidence at k = 1, memory growth), Long-Context Extension (RoPE bases).
"""
import copy
import math

import numpy as np
import pytest

import oracle
import synth
from oracle import LAST_LOOP, PER_LOOP


def _model(shape=synth.TINY, **kw):
    w = synth.make_weights(shape)
    return oracle.Oracle(shape, w, **kw), w


# ---------------------------------------------------------------- primitives
def test_l2n_closed_form():
    np.testing.assert_allclose(oracle.l2n(np.array([3.0, 4.0])), [0.6, 0.8], rtol=0, atol=1e-15)
    assert np.all(oracle.l2n(np.zeros(5)) == 0.0)
    # batched: normalises the last axis only
    x = np.array([[[1.0, 0.0], [0.0, -2.0]]])
    np.testing.assert_allclose(oracle.l2n(x), [[[1.0, 0.0], [0.0, -1.0]]], atol=1e-15)


def test_ngpt_update_closed_form():
    e0, e1 = np.array([1.0, 0.0, 0.0]), np.array([0.0, 1.0, 0.0])
    half = np.full(3, 0.5)
    # halfway between two orthogonal unit vectors; y's scale is irrelevant
    np.testing.assert_allclose(oracle.ngpt_update(e0, 7.0 * e1, half),
                               [1 / math.sqrt(2), 1 / math.sqrt(2), 0.0], atol=1e-15)
    np.testing.assert_allclose(oracle.ngpt_update(e0, e1, np.zeros(3)), e0, atol=1e-15)
    np.testing.assert_allclose(oracle.ngpt_update(e0, -3.0 * e1, np.ones(3)), -e1, atol=1e-15)
    # per-coordinate rate: only coordinate 1 moves, (1, 0, 0) + (0, 1, 0)
    a = np.array([0.0, 1.0, 0.0])
    np.testing.assert_allclose(oracle.ngpt_update(e0, e1, a),
                               [1 / math.sqrt(2), 1 / math.sqrt(2), 0.0], atol=1e-15)


def test_sigmoid_silu_closed_form():
    assert oracle.sigmoid(0.0) == 0.5
    assert abs(oracle.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert abs(oracle.silu(-2.0) + 2.0 / (1.0 + math.exp(2.0))) < 1e-15


def test_rope_closed_form():
    base = 100.0
    p = 3
    eye = np.eye(4)
    r = oracle.rope(eye[:, None, :], np.array([p]), base)[:, 0, :]   # rows: images of e_i
    t0, t1 = p * 1.0, p * base ** (-0.5)
    np.testing.assert_allclose(r[0], [math.cos(t0), 0, math.sin(t0), 0], atol=1e-15)
    np.testing.assert_allclose(r[1], [0, math.cos(t1), 0, math.sin(t1)], atol=1e-15)
    np.testing.assert_allclose(r[2], [-math.sin(t0), 0, math.cos(t0), 0], atol=1e-15)
    np.testing.assert_allclose(r[3], [0, -math.sin(t1), 0, math.cos(t1)], atol=1e-15)


def test_rope_properties():
    rng = np.random.default_rng(5)
    q, k = rng.standard_normal((2, 1, 32))
    pos = np.array([0])
    np.testing.assert_allclose(oracle.rope(q, pos, 1e4), q, atol=0)           # identity at 0
    for base in (1e4, 1e7):
        a = oracle.rope(q, np.array([17]), base) @ oracle.rope(k, np.array([5]), base).T
        b = oracle.rope(q, np.array([112]), base) @ oracle.rope(k, np.array([100]), base).T
        np.testing.assert_allclose(a, b, rtol=1e-12)                          # relative only
        np.testing.assert_allclose(np.linalg.norm(oracle.rope(q, np.array([999]), base)),
                                   np.linalg.norm(q), rtol=1e-14)            # a rotation


def test_attention_two_keys_closed_form():
    # unit q aligned with key 0 and orthogonal to key 1: weights e^s / (e^s + 1)
    s = math.sqrt(32.0)
    q = np.zeros((1, 4)); q[0, 0] = 1
    kk = np.zeros((2, 4)); kk[0, 0] = 1; kk[1, 1] = 1
    v = np.zeros((2, 4)); v[0, 2] = 1; v[1, 3] = 1
    o = oracle.attention(q, kk, v, np.array([1]), np.array([0, 1]), 16, True, s)
    p0 = math.exp(s) / (math.exp(s) + 1.0)
    np.testing.assert_allclose(o[0], [0, 0, p0, 1 - p0], rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("window,full", [(16, False), (5, False), (1, False), (10**6, True)])
@pytest.mark.parametrize("P0,C", [(0, 40), (23, 17), (39, 1)])
def test_attention_uniform_probe_counts(window, full, P0, C):
    """Equal scores: the output averages the values of the visible keys.
    With one-hot values the visible set of query t is the interval
    [max(0, t - W + 1), t] (sliding window) or [0, t] (full)."""
    L = P0 + C
    q = np.ones((C, L)) / math.sqrt(L)
    kk = np.ones((L, L)) / math.sqrt(L)
    v = np.eye(L)
    qpos = np.arange(P0, L)
    o = oracle.attention(q, kk, v, qpos, np.arange(L), window, full, 11.3)
    for i, t in enumerate(qpos):
        lo = 0 if full else max(0, t - window + 1)
        want = np.zeros(L)
        want[lo:t + 1] = 1.0 / (t + 1 - lo)
        np.testing.assert_allclose(o[i], want, atol=1e-15)


# ------------------------------------------------------------ model pieces
def test_mlp_closed_form_silu_side():
    """d = F = 2, h = e0, W_down = I, alpha = 1: output = N(m) with
    m = (W_up h) * SiLU(W_sl h) = (1*SiLU(1), 1*SiLU(-1))."""
    sh = synth.TINY.replace(d=2, ffn=2)
    o = oracle.Oracle.__new__(oracle.Oracle)
    o.shape, o.dtype, o.trace = sh, np.float64, None
    lw = {"w_up": np.array([[1.0, 0.0], [1.0, 0.0]]), "w_sl": np.array([[1.0, 0.0], [-1.0, 0.0]]),
          "w_down": np.eye(2), "alpha_mlp": np.ones(2)}
    o.w = {"layers": [lw]}
    s1 = 1.0 / (1.0 + math.exp(-1.0))
    m = np.array([s1, -(1.0 - s1)])          # SiLU(-1) = -sigmoid(-1) = -(1 - sigmoid(1))
    out = o.mlp_sublayer(0, np.array([[[1.0, 0.0]]]))
    np.testing.assert_allclose(out[0, 0], m / np.linalg.norm(m), atol=1e-15)


def test_gqa_group_mapping_equals_duplicated_mha():
    """GQA with G = n_q / n_kv query heads per kv head equals MHA whose
    k/v heads are copies: q head h reads kv head h // G."""
    sh = synth.TINY.replace(n_in=1, n_rec=0, n_out=0)
    w = synth.make_weights(sh)
    mha_sh = sh.replace(n_kv=sh.n_q)
    w2 = {k: v for k, v in w.items() if k != "layers"}
    lw = dict(w["layers"][0])
    G, dh = sh.n_q // sh.n_kv, sh.head_dim
    for name in ("w_k", "w_v"):
        heads = lw[name].reshape(sh.n_kv, dh, sh.d)
        lw[name] = np.concatenate([heads[h // G] for h in range(sh.n_q)], axis=0)
    w2["layers"] = [lw]
    tok = synth.tokens(sh, 2, 24)
    a = oracle.Oracle(sh, w).prefill(tok, 1, LAST_LOOP, all_logits=True)["hidden"]
    b = oracle.Oracle(mha_sh, w2).prefill(tok, 1, LAST_LOOP, all_logits=True)["hidden"]
    np.testing.assert_allclose(a, b, atol=1e-13)


def test_window_one_returns_own_value():
    """W = 1: each query sees only itself, so the attention output is its own
    value vector, whatever q and k are."""
    rng = np.random.default_rng(2)
    q, kk, v = rng.standard_normal((3, 9, 8))
    o = oracle.attention(q, kk, v, np.arange(9), np.arange(9), 1, False, 3.0)
    np.testing.assert_allclose(o, v, atol=1e-15)


def test_window_covering_sequence_equals_full():
    sh = synth.TINY.replace(window=10**6, rope_base_full=1e4)
    sh_full = sh.replace(full_every=1, full_offset=0)
    w = synth.make_weights(synth.TINY)
    tok = synth.tokens(sh, 2, 40)
    a = oracle.Oracle(sh, w).prefill(tok, 2, LAST_LOOP, all_logits=True)["logits"]
    b = oracle.Oracle(sh_full, w).prefill(tok, 2, LAST_LOOP, all_logits=True)["logits"]
    np.testing.assert_allclose(a, b, atol=1e-13)


def test_value_scale_invariance():
    """Scaling W_v scales o, which the sublayer normalisations remove; a
    missing N(y) in the residual step would break this."""
    sh = synth.TINY
    w = synth.make_weights(sh)
    w2 = dict(w)
    w2["layers"] = [dict(lw, w_v=lw["w_v"] * 3.0, w_up=lw["w_up"] * 0.25) for lw in w["layers"]]
    tok = synth.tokens(sh, 1, 20)
    a = oracle.Oracle(sh, w).prefill(tok, 2, LAST_LOOP, all_logits=True)["logits"]
    b = oracle.Oracle(sh, w2).prefill(tok, 2, LAST_LOOP, all_logits=True)["logits"]
    np.testing.assert_allclose(a, b, atol=1e-13)


def test_alpha_zero_reduces_to_embedding_dot_products():
    """alpha = 0: every residual step and every loop boundary returns its
    input, so logits = s_z * E_out . N(E_in[tok]) at any k."""
    sh = synth.TINY.replace(alpha_attn=0.0, alpha_mlp=0.0)
    w = synth.make_weights(sh)
    tok = synth.tokens(sh, 2, 12)
    e = w["embed_in"][tok].astype(np.float64)
    want = (e / np.linalg.norm(e, axis=-1, keepdims=True)) @ w["embed_out"].astype(np.float64).T
    for k in (1, 3):
        got = oracle.Oracle(sh, w).prefill(tok, k, PER_LOOP, all_logits=True)["logits"]
        np.testing.assert_allclose(got, want, atol=1e-13)


def test_loop_schedule_closed_form():
    """2-D geometry: x = e0 and a block that adds e1 then normalises.  With
    s_{i-1} at angle phi, N(s + x) sits at phi/2 and the block output at
    45deg + phi/4, so phi_i = 45 + phi_{i-1}/4 (degrees), phi_0 = 0."""
    x = np.array([1.0, 0.0])
    block = lambda u, i: oracle.l2n(u + np.array([0.0, 1.0]))
    phi = 0.0
    for k in range(1, 6):
        phi = 45.0 + phi / 4.0
        s = oracle.loop_schedule(x, k, block)
        r = math.radians(phi)
        np.testing.assert_allclose(s, [math.cos(r), math.sin(r)], atol=1e-15)
    # the loop index reaches the block as 1..k
    seen = []
    oracle.loop_schedule(x, 3, lambda u, i: (seen.append(i), u)[1])
    assert seen == [1, 2, 3]


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("k", [1, 2, 4])
def test_unit_norm_everywhere_and_layer_applications(k):
    o, _ = _model()
    o.trace = oracle.Trace()
    o.prefill(synth.tokens(o.shape, 2, 30), k, LAST_LOOP)
    allnorms = np.concatenate([n.ravel() for n in o.trace.norms])
    assert np.max(np.abs(allnorms - 1.0)) < 1e-12
    sh = o.shape
    assert o.trace.layer_apps == sh.n_in + sh.n_out + k * sh.n_rec


def test_layer_application_counts_4b():
    """32 + 40k physical-layer applications: 72, 112, 192 at k = 1, 2, 4."""
    sh = synth.DORY4B
    assert [sh.n_in + sh.n_out + k * sh.n_rec for k in (1, 2, 4)] == [72, 112, 192]
    assert sum(sh.is_full(l) for l in range(sh.n_layers)) == 18
    assert sum(sh.is_full(l) for l in range(sh.n_in, sh.n_in + sh.n_rec)) == 10


@pytest.mark.parametrize("shape", [synth.TINY, synth.TINY_LOOPFULL])
def test_k1_equals_plain_stack(shape):
    o, _ = _model(shape)
    tok = synth.tokens(shape, 2, 40)
    h_loop = o.prefill(tok, 1, LAST_LOOP, all_logits=True)["hidden"]
    h_stack = oracle.Oracle(shape, synth.make_weights(shape)).stack_forward(tok)
    np.testing.assert_allclose(h_loop, h_stack, atol=1e-12)


def _run(shape, w, k, mode, prompt, dec, chunks=None):
    o = oracle.Oracle(shape, w)
    outs = []
    if chunks is None:
        outs.append(o.prefill(prompt, k, mode)["logits"][:, -1])
    else:
        for c0, c1 in chunks:
            r = o.prefill(prompt[:, c0:c1], k, mode)
        outs.append(r["logits"][:, -1])
    for t in dec.T:
        outs.append(o.decode(t, k, mode)["logits"])
    return np.stack(outs), o


@pytest.mark.parametrize("shape", [synth.TINY, synth.TINY_LOOPFULL])
def test_cache_policies_coincide_at_k1(shape):
    w = synth.make_weights(shape)
    prompt = synth.tokens(shape, 2, 40)
    dec = synth.tokens(shape, 2, 8, seed=1)
    a, _ = _run(shape, w, 1, LAST_LOOP, prompt, dec)
    b, _ = _run(shape, w, 1, PER_LOOP, prompt, dec)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("k", [2, 4])
def test_single_chunk_prefill_same_in_both_policies(k):
    sh = synth.TINY_LOOPFULL
    w = synth.make_weights(sh)
    tok = synth.tokens(sh, 2, 40)
    a = oracle.Oracle(sh, w).prefill(tok, k, LAST_LOOP, all_logits=True)["logits"]
    b = oracle.Oracle(sh, w).prefill(tok, k, PER_LOOP, all_logits=True)["logits"]
    assert np.array_equal(a, b)


@pytest.mark.parametrize("shape", [synth.TINY, synth.TINY_LOOPFULL])
@pytest.mark.parametrize("k", [1, 2, 4])
def test_per_loop_decode_equals_recompute(shape, k):
    """Per-loop caching attends loop i to loop i, exactly as a fresh
    prefill of the whole prefix does."""
    w = synth.make_weights(shape)
    prompt = synth.tokens(shape, 2, 40)
    dec = synth.tokens(shape, 2, 8, seed=1)
    inc, _ = _run(shape, w, k, PER_LOOP, prompt, dec)
    full = np.concatenate([prompt, dec], axis=1)
    ref = oracle.Oracle(shape, w).prefill(full, k, PER_LOOP, all_logits=True)["logits"]
    for s in range(dec.shape[1] + 1):
        np.testing.assert_allclose(inc[s], ref[:, 39 + s], atol=1e-12)


def test_last_loop_decode_differs_from_recompute_beyond_k1():
    """Last-loop caching shows earlier-loop queries final-loop keys of past
    tokens, so it is not a recompute once k > 1 (and is one at k = 1)."""
    sh = synth.TINY_LOOPFULL
    w = synth.make_weights(sh)
    prompt = synth.tokens(sh, 2, 40)
    dec = synth.tokens(sh, 2, 4, seed=1)
    full = np.concatenate([prompt, dec], axis=1)
    for k, differs in ((1, False), (2, True)):
        inc, _ = _run(sh, w, k, LAST_LOOP, prompt, dec)
        ref = oracle.Oracle(sh, w).prefill(full, k, LAST_LOOP, all_logits=True)["logits"]
        diff = max(np.max(np.abs(inc[s] - ref[:, 39 + s])) for s in range(1, 5))
        assert (diff > 1e-6) == differs, diff


def test_chunked_prefill_equals_unchunked_per_loop():
    sh = synth.TINY_LOOPFULL
    w = synth.make_weights(sh)
    prompt = synth.tokens(sh, 2, 48)
    dec = synth.tokens(sh, 2, 3, seed=1)
    a, _ = _run(sh, w, 2, PER_LOOP, prompt, dec)
    b, _ = _run(sh, w, 2, PER_LOOP, prompt, dec, chunks=[(0, 7), (7, 30), (30, 48)])
    np.testing.assert_allclose(a, b, atol=1e-12)


def test_per_loop_rejects_k_change():
    o, _ = _model()
    o.prefill(synth.tokens(o.shape, 1, 8), 2, PER_LOOP)
    with pytest.raises(ValueError):
        o.decode(np.array([1]), 3, PER_LOOP)
    o2, _ = _model()
    o2.prefill(synth.tokens(o2.shape, 1, 8), 2, LAST_LOOP)
    o2.decode(np.array([1]), 3, LAST_LOOP)        # last-loop cache is k-independent


def test_greedy_ties_lowest_index():
    """Greedy decoding picks the lowest index among equal maxima.  Two rows of
    E_out are set to the decode step's own final hidden state (a unit vector,
    and the LM head does not feed back into it), so those two logits are
    exactly 1, the maximum over unit rows; the next token must be the lower
    of the two indices whichever order they are planted in."""
    sh = synth.TINY
    w = synth.make_weights(sh)
    prompt = synth.tokens(sh, 2, 10)
    tok = synth.tokens(sh, 2, 1, seed=1)[:, 0]
    o = oracle.Oracle(sh, w)
    o.prefill(prompt, 2, LAST_LOOP)
    h = o.decode(tok, 2, LAST_LOOP)["hidden"]
    for lo, hi in ((37, 411), (5, 6)):
        for b in range(2):
            w2 = dict(w)
            e = w["embed_out"].astype(np.float64).copy()
            e[lo] = e[hi] = h[b]
            w2["embed_out"] = e
            o2 = oracle.Oracle(sh, w2)
            o2.prefill(prompt, 2, LAST_LOOP)
            r = o2.decode(tok, 2, LAST_LOOP)
            assert r["logits"][b, lo] == r["logits"][b, hi]
            assert r["logits"][b, lo] == np.max(r["logits"][b])
            assert int(r["next"][b]) == lo


def _final_loop_everywhere(o, sh, k):
    """Cache surgery on a per-loop oracle: every loop's slice of every
    recurrent layer is replaced by the final loop's keys and values."""
    for l in range(sh.n_in, sh.n_in + sh.n_rec):
        fin = o.cache[(l, k)]
        for i in range(1, k):
            o.cache[(l, i)] = type(fin)(fin.k.copy(), fin.v.copy(), fin.first)


@pytest.mark.parametrize("k", [2, 4])
def test_last_loop_decode_equals_recompute_with_final_loop_keys(k):
    """Last-Loop KV Caching: past positions are seen through the final
    loop's keys and values whichever loop the query is in, while the current
    token uses its own current-loop values.  Built by hand from the per-loop
    cache (pinned against full recompute above): after the prompt and after
    each decode step, every loop's slice is overwritten with loop k's, and
    the per-loop step that follows must then reproduce the last-loop step
    exactly.  A last-loop rule that kept any other loop's entries fails."""
    sh = synth.TINY_LOOPFULL
    w = synth.make_weights(sh)
    prompt = synth.tokens(sh, 2, 40)
    dec = synth.tokens(sh, 2, 4, seed=1)
    a = oracle.Oracle(sh, w)
    b = oracle.Oracle(sh, w)
    a.prefill(prompt, k, LAST_LOOP)
    b.prefill(prompt, k, PER_LOOP)
    for s in range(dec.shape[1]):
        _final_loop_everywhere(b, sh, k)
        ra = a.decode(dec[:, s], k, LAST_LOOP)
        rb = b.decode(dec[:, s], k, PER_LOOP)
        assert np.array_equal(ra["logits"], rb["logits"])
        assert np.array_equal(ra["hidden"], rb["hidden"])


def test_last_loop_chunked_prefill_equals_final_loop_surgery():
    """The same rule across prefill chunks: a later chunk sees the earlier
    chunks through their final-loop entries."""
    sh = synth.TINY_LOOPFULL
    k = 3
    w = synth.make_weights(sh)
    prompt = synth.tokens(sh, 2, 45)
    a = oracle.Oracle(sh, w)
    b = oracle.Oracle(sh, w)
    for c0, c1 in ((0, 9), (9, 30), (30, 45)):
        if c0:
            _final_loop_everywhere(b, sh, k)
        ra = a.prefill(prompt[:, c0:c1], k, LAST_LOOP, all_logits=True)
        rb = b.prefill(prompt[:, c0:c1], k, PER_LOOP, all_logits=True)
        assert np.array_equal(ra["logits"], rb["logits"])


def test_rope_base_follows_layer_type():
    """Long-Context Extension: sliding-window layers rotate with base 1e4,
    full-attention layers with base 1e7.  One head of width 4 (pairs (0, 2)
    at frequency 1 and (1, 3) at base^-1/2), two tokens whose query/key
    parts are both e1 at positions 0 and p, so their rotated dot product is
    cos(p * base^-1/2) while each token's own score is 1.  Their values are
    orthogonal and W_o, the gate and alpha = 1 pass the attention output
    through, so the second token's new state is N(w0 e0 + w1 e1) with
    w0 / w1 = exp(scale * (cos(p base^-1/2) - 1)), scale = sqrt(4) = 2."""
    sh = synth.TINY.replace(d=6, n_q=1, n_kv=1, head_dim=4, n_in=2, n_rec=0, n_out=0,
                            full_every=2, full_offset=1, window=10**6)
    assert not sh.is_full(0) and sh.is_full(1)
    o = oracle.Oracle.__new__(oracle.Oracle)
    o.shape, o.dtype, o.trace = sh, np.float64, None
    qk = np.zeros((4, 6)); qk[:4, :4] = np.eye(4)
    wv = np.zeros((4, 6)); wv[0, 4] = 1.0; wv[1, 5] = 1.0
    wo = np.zeros((6, 4)); wo[:4, :4] = np.eye(4)
    lw = {"w_q": qk, "w_k": qk, "w_v": wv, "w_g": np.zeros((4, 6)), "w_o": wo,
          "alpha_attn": np.ones(6), "s_qk": np.ones(4)}
    o.w = {"layers": [lw, lw]}
    h = np.zeros((1, 2, 6))
    h[0, 0, [1, 4]] = 1 / math.sqrt(2)
    h[0, 1, [1, 5]] = 1 / math.sqrt(2)
    for p in (100, 3000):
        for layer, base in ((0, 1.0e4), (1, 1.0e7)):
            o.reset()
            out = o.attn_sublayer(layer, h, np.array([0, p]), None, LAST_LOOP, 1)
            ratio = out[0, 1, 0] / out[0, 1, 1]
            want = math.exp(2.0 * (math.cos(p * base ** -0.5) - 1.0))
            np.testing.assert_allclose(ratio, want, rtol=1e-12)
            np.testing.assert_allclose(np.linalg.norm(out[0, 1]), 1.0, atol=1e-15)


# ------------------------------------------------------------- KV footprint
def test_kv_bytes_closed_forms():
    # tiny, batch 2, 72 positions: per position 2 (K,V) * 2 kv heads * 32 * 2 B = 256 B;
    # layers 0-2 window 16, layer 3 full: (3*16 + 72) * 256 * 2 sequences
    assert oracle.kv_bytes(synth.TINY, 2, 72, 4, LAST_LOOP) == (3 * 16 + 72) * 256 * 2 == 61440
    # per-loop: the two recurrent (window) layers hold 4 slices each
    assert oracle.kv_bytes(synth.TINY, 2, 72, 4, PER_LOOP) == (16 + 8 * 16 + 72) * 256 * 2 == 110592
    sh = synth.DORY4B
    full_only = 18 * 262144 * (2 * 4 * 128 * 2)
    assert full_only == 9_663_676_416
    swa = 54 * 4096 * (2 * 4 * 128 * 2)
    assert oracle.kv_bytes(sh, 1, 262144, 1, LAST_LOOP) == full_only + swa


@pytest.mark.parametrize("shape", [synth.TINY, synth.SMALL, synth.DORY4B])
def test_kv_bytes_scaling_in_k(shape):
    last = [oracle.kv_bytes(shape, 4, 5000, k, LAST_LOOP) for k in (1, 2, 3, 4)]
    per = [oracle.kv_bytes(shape, 4, 5000, k, PER_LOOP) for k in (1, 2, 3, 4)]
    assert len(set(last)) == 1 and per[0] == last[0]
    per_pos = 2 * shape.n_kv * shape.head_dim * 2
    rec = sum((5000 if shape.is_full(l) else min(5000, shape.window)) * per_pos
              for l in range(shape.n_in, shape.n_in + shape.n_rec)) * 4
    assert [b - a for a, b in zip(per, per[1:])] == [rec] * 3


def test_slot_positions_closed_form():
    S = 16
    for n in (0, 5, 16, 17, 40, 71):
        got = oracle.slot_positions(range(n), S)
        want = [s + S * ((n - 1 - s) // S) if s < n else -1 for s in range(S)]
        assert list(got) == want


def test_round_bf16():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 0.0], np.float32)
    assert list(synth.round_bf16(x)) == [1.0, 1.0, 1.0 + 2**-6, -2.5, 0.0]


def test_qk_scale_invariance():
    """Per-head q/k normalisation: scaling W_q and W_k leaves every output
    unchanged (it would not without the normalisation)."""
    sh = synth.TINY_LOOPFULL
    w = synth.make_weights(sh)
    w2 = dict(w)
    w2["layers"] = [dict(lw, w_q=lw["w_q"] * 4.0, w_k=lw["w_k"] * 0.125) for lw in w["layers"]]
    tok = synth.tokens(sh, 1, 24)
    a = oracle.Oracle(sh, w).prefill(tok, 2, LAST_LOOP, all_logits=True)["logits"]
    b = oracle.Oracle(sh, w2).prefill(tok, 2, LAST_LOOP, all_logits=True)["logits"]
    np.testing.assert_allclose(a, b, atol=1e-13)
    # and the per-head normalisation is not a whole-row one: scaling one
    # head's W_q rows changes nothing either
    w3 = dict(w)
    dh = sh.head_dim
    w3["layers"] = [dict(lw, w_q=np.concatenate([lw["w_q"][:dh] * 8.0, lw["w_q"][dh:]]))
                    for lw in w["layers"]]
    c = oracle.Oracle(sh, w3).prefill(tok, 2, LAST_LOOP, all_logits=True)["logits"]
    np.testing.assert_allclose(a, c, atol=1e-13)


def test_gate_closed_form_single_token():
    """One token, one head, d = head_dim = 2, no RoPE: its only visible key
    is itself, so o = v.  With h = e0, W_v h = (1, 1), W_g h = (2, -1),
    W_o = I and alpha = 1 the sublayer returns N(sigmoid(2), sigmoid(-1))."""
    sh = synth.TINY.replace(d=2, n_q=1, n_kv=1, head_dim=2, rope=False, n_in=1, n_rec=0,
                            n_out=0, full_offset=0)
    o = oracle.Oracle.__new__(oracle.Oracle)
    o.shape, o.dtype, o.trace = sh, np.float64, None
    lw = {"w_q": np.eye(2), "w_k": np.eye(2), "w_v": np.array([[1.0, 0.0], [1.0, 0.0]]),
          "w_g": np.array([[2.0, 0.0], [-1.0, 0.0]]), "w_o": np.eye(2),
          "alpha_attn": np.ones(2), "s_qk": np.ones(2)}
    o.w = {"layers": [lw]}
    o.reset()
    out = o.attn_sublayer(0, np.array([[[1.0, 0.0]]]), np.array([0]), None, LAST_LOOP, 1)
    g = np.array([1 / (1 + math.exp(-2.0)), 1 / (1 + math.exp(1.0))])
    np.testing.assert_allclose(out[0, 0], g / np.linalg.norm(g), atol=1e-15)


def test_qk_scale_parameter_scales_logits_quadratically():
    """s_qk multiplies both unit q and unit k, so s_qk = c is the same as
    a softmax scale multiplied by c^2."""
    rng = np.random.default_rng(3)
    q, kk, v = rng.standard_normal((3, 12, 8))
    qh, kh = oracle.l2n(q), oracle.l2n(kk)
    pos = np.arange(12)
    c = 1.7
    a = oracle.attention(c * qh, c * kh, v, pos, pos, 5, False, 2.0)
    b = oracle.attention(qh, kh, v, pos, pos, 5, False, 2.0 * c * c)
    np.testing.assert_allclose(a, b, atol=1e-13)
    sh = synth.TINY
    w = synth.make_weights(sh)
    w2 = dict(w)
    w2["layers"] = [dict(lw, s_qk=lw["s_qk"] * 1.3) for lw in w["layers"]]
    tok = synth.tokens(sh, 1, 20)
    x = oracle.Oracle(sh, w).prefill(tok, 1, LAST_LOOP)["logits"]
    y = oracle.Oracle(sh, w2).prefill(tok, 1, LAST_LOOP)["logits"]
    assert np.max(np.abs(x - y)) > 1e-6          # s_qk reaches the scores


def test_logit_scale_is_per_vocabulary_entry():
    """logits = s_z * (E_out h): a per-entry scale multiplies each vocabulary
    column of the logits and leaves the hidden state alone."""
    sh = synth.TINY
    w = synth.make_weights(sh)
    tok = synth.tokens(sh, 2, 12)
    a = oracle.Oracle(sh, w).prefill(tok, 2, LAST_LOOP)
    s = np.linspace(0.5, 3.0, sh.vocab)
    b = oracle.Oracle(sh, dict(w, s_z=s)).prefill(tok, 2, LAST_LOOP)
    assert np.array_equal(a["hidden"], b["hidden"])
    np.testing.assert_allclose(b["logits"], a["logits"] * s, rtol=1e-14, atol=1e-16)
    np.testing.assert_allclose(a["logits"], a["hidden"] @ w["embed_out"].astype(np.float64).T,
                               rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("mode", [LAST_LOOP, PER_LOOP], ids=["last", "perloop"])
def test_restore_replays_the_next_step(mode):
    """A step replayed from a copy of the cache state (what the GPU tests
    export at long contexts) equals the step taken by the oracle that built
    that state."""
    sh, k = synth.TINY_LOOPFULL, 3
    w = synth.make_weights(sh)
    a = oracle.Oracle(sh, w)
    a.prefill(synth.tokens(sh, 2, 37), k, mode)
    a.decode(synth.tokens(sh, 2, 1, seed=1)[:, 0], k, mode)
    saved = {key: (c.k.copy(), c.v.copy(), c.first) for key, c in a.cache.items()}
    b = oracle.Oracle(sh, w)
    b.restore(a.length, mode, k, saved)
    tok = synth.tokens(sh, 2, 1, seed=2)[:, 0]
    ra, rb = a.decode(tok, k, mode), b.decode(tok, k, mode)
    assert np.array_equal(ra["logits"], rb["logits"])
    chunk = synth.tokens(sh, 2, 9, seed=3)
    assert np.array_equal(a.prefill(chunk, k, mode)["logits"], b.prefill(chunk, k, mode)["logits"])
    with pytest.raises(ValueError):
        b.restore(a.length + 1, mode, k, saved)


def _greedy_decode(o, first, k, n, mode, draft=False):
    out, cur = [], np.asarray(first)
    for _ in range(n):
        h = o.step(cur.reshape(-1, 1), k, mode, draft=draft)[:, 0]
        cur = np.argmax(o.logits(h), axis=-1)
        out.append(cur)
    return np.stack(out, axis=1)


@pytest.mark.parametrize("k_draft,gamma", [(1, 4), (2, 3), (1, 1)])
def test_speculative_greedy_equals_plain_greedy_at_k_verify(k_draft, gamma):
    """Self-Speculative Decoding: whatever the drafts, the emitted tokens are
    those of plain greedy decoding at the verifier's loop count (the
    verifier decides every emitted token), and the caches the step leaves
    behind are those plain decoding of the emitted tokens leaves."""
    sh, kv = synth.TINY_LOOPFULL, 4
    w = synth.make_weights(sh)
    prompt = synth.tokens(sh, 2, 21)
    ref = oracle.Oracle(sh, w)
    first = np.argmax(ref.prefill(prompt, kv, PER_LOOP)["logits"][:, -1], axis=-1)
    spec = oracle.Oracle(sh, w)
    spec.prefill(prompt, kv, PER_LOOP)
    emitted, cur, counts = [], first, []
    while sum(e.shape[1] for e in emitted) < 12:
        # the count by brute force from copies of the state: greedy drafts at
        # k_draft against greedy tokens at the verifier's depth
        d = _greedy_decode(copy.deepcopy(spec), cur, k_draft, gamma, PER_LOOP, draft=True)
        v = _greedy_decode(copy.deepcopy(spec), cur, kv, gamma + 1, PER_LOOP)
        lead = np.cumprod(d == v[:, :gamma], axis=1).sum(axis=1)
        out, n = spec.speculative_step(cur, k_draft, kv, gamma)
        assert n == int(lead.min()) + 1 and out.shape == (2, n)
        assert np.array_equal(out, v[:, :n])
        emitted.append(out)
        counts.append(n)
        cur = out[:, -1]
    assert max(counts) > 1                     # some drafts were accepted
    emitted = np.concatenate(emitted, axis=1)
    plain = _greedy_decode(ref, first, kv, emitted.shape[1], PER_LOOP)
    assert np.array_equal(emitted, plain)
    # the state after the steps continues exactly like plain decoding
    assert spec.length == ref.length
    np.testing.assert_allclose(spec.decode(emitted[:, -1], kv, PER_LOOP)["logits"],
                               ref.decode(plain[:, -1], kv, PER_LOOP)["logits"], atol=1e-12)


def test_speculative_draft_at_verify_depth_accepts_everything():
    """With the drafter as deep as the verifier every draft is the verifier's
    own greedy token, so all gamma drafts are accepted."""
    sh = synth.TINY_LOOPFULL
    w = synth.make_weights(sh)
    o = oracle.Oracle(sh, w)
    first = np.argmax(o.prefill(synth.tokens(sh, 2, 17), 2, PER_LOOP)["logits"][:, -1], axis=-1)
    out, n = o.speculative_step(first, 2, 2, 5)
    assert n == 6
    assert len(set(out[1].tolist())) == 6     # six different tokens: no fixed point


def test_speculative_step_needs_per_loop_caching():
    sh = synth.TINY_LOOPFULL
    o = oracle.Oracle(sh, synth.make_weights(sh))
    o.prefill(synth.tokens(sh, 1, 5), 4, LAST_LOOP)
    with pytest.raises(ValueError):
        o.speculative_step(np.array([1]), 1, 4, 4)
