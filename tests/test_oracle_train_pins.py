"""Pins of the truncated-backpropagation training-step oracle (oracle/train.py;
"Dory1.0-4B: A Looped Normalized-GPT", Truncated Backpropagation).

Anchors, all against the numpy oracle (oracle/model.py, a separate
implementation of the forward pass that is pinned on its own):
  * the step's loss equals the next-token cross-entropy of the numpy
    oracle's logits;
  * sampled gradient entries of every kind of parameter equal central
    finite differences of the numpy objective: the plain objective at
    k = 1, and at k >= 2 the objective with the state before the final
    invocation held at its value (the definition of the truncation);
  * at k >= 2 the truncated gradient of the recurrent weights is not the
    full-backpropagation difference quotient (the truncation is real),
    while the input block still receives a gradient (through the
    re-injected input of the final invocation)."""
import numpy as np
import pytest

import oracle
import synth
from oracle import train

SHAPE = synth.TINY
EPS = 1e-5


def _weights64():
    w = synth.make_weights(SHAPE)
    out = {k: np.asarray(v, np.float64).copy() for k, v in w.items() if k != "layers"}
    out["layers"] = [{k: np.asarray(v, np.float64).copy() for k, v in lw.items()}
                     for lw in w["layers"]]
    return out


def _tokens(B=2, T=20, seed=7):
    return synth.tokens(SHAPE, B, T, seed=seed)


def _objective(w, tokens, k, frozen=None):
    """Mean next-token cross-entropy of the numpy oracle's forward pass.
    frozen: the state before the final invocation, held fixed (k >= 2)."""
    o = oracle.Oracle(SHAPE, w)
    T = tokens.shape[1]
    pos = np.arange(T)
    h = oracle.l2n(o.w["embed_in"][tokens])
    for l in range(SHAPE.n_in):
        h = o.layer(l, h, pos, None, oracle.LAST_LOOP, k)
    x = h

    def block(u, i):
        for l in range(SHAPE.n_in, SHAPE.n_in + SHAPE.n_rec):
            u = o.layer(l, u, pos, i, oracle.LAST_LOOP, k)
        return u

    if frozen is None:
        s = oracle.loop_schedule(x, k, block)
    else:
        s = oracle.l2n(block(oracle.l2n(frozen + x), k))
    h = s
    for l in range(SHAPE.n_in + SHAPE.n_rec, SHAPE.n_layers):
        h = o.layer(l, h, pos, None, oracle.LAST_LOOP, k)
    z = o.logits(h)[:, :-1]
    m = z.max(axis=-1, keepdims=True)
    lse = m[..., 0] + np.log(np.exp(z - m).sum(axis=-1))
    picked = np.take_along_axis(z, tokens[:, 1:, None], axis=-1)[..., 0]
    return float(np.mean(lse - picked))


def _state_before_final(w, tokens, k):
    """s_{k-1}: the state after invocations 1 .. k-1 (numpy oracle)."""
    o = oracle.Oracle(SHAPE, w)
    pos = np.arange(tokens.shape[1])
    h = oracle.l2n(o.w["embed_in"][tokens])
    for l in range(SHAPE.n_in):
        h = o.layer(l, h, pos, None, oracle.LAST_LOOP, k)

    def block(u, i):
        for l in range(SHAPE.n_in, SHAPE.n_in + SHAPE.n_rec):
            u = o.layer(l, u, pos, i, oracle.LAST_LOOP, k)
        return u

    return oracle.loop_schedule(h, k - 1, block)


def _array(tree, where):
    """where: ("top", name) or ("layer", l, name)."""
    return tree[where[1]] if where[0] == "top" else tree["layers"][where[1]][where[2]]


def _perturbed(w, where, idx, delta):
    w2 = dict(w)
    w2["layers"] = [dict(lw) for lw in w["layers"]]
    a = _array(w, where).copy()
    a[idx] += delta
    if where[0] == "top":
        w2[where[1]] = a
    else:
        w2["layers"][where[1]][where[2]] = a
    return w2


def _fd(w, where, idx, tokens, k, frozen):
    fp = _objective(_perturbed(w, where, idx, EPS), tokens, k, frozen)
    fm = _objective(_perturbed(w, where, idx, -EPS), tokens, k, frozen)
    return (fp - fm) / (2 * EPS)


NAMES = ("w_q", "w_k", "w_v", "w_g", "w_o", "w_up", "w_sl", "w_down",
         "alpha_attn", "alpha_mlp", "s_qk")


def _entries(tokens):
    """(where, index) pairs covering every kind of parameter: embeddings of
    used tokens, the LM head and s_z, and each matrix and vector kind in the
    input layer, both recurrent layers and the output layer."""
    t0, t1 = int(tokens[0, 3]), int(tokens[1, 5])
    e = [(("top", "embed_in"), (t0, 11)), (("top", "embed_out"), (t1, 40)),
         (("top", "s_z"), (t1,)), (("top", "s_z"), (int(tokens[0, 9]),))]
    rng = np.random.default_rng(3)
    for l in range(SHAPE.n_layers):
        lw = synth.layer_weights(SHAPE, l)
        for j, name in enumerate(NAMES):
            if (l + j) % 2:                             # half per layer, every kind overall
                continue
            e.append((("layer", l, name), tuple(int(rng.integers(0, n)) for n in lw[name].shape)))
    return e


def _check_fd(k):
    w = _weights64()
    tokens = _tokens()
    loss, grads = train.tbptl_step(SHAPE, w, tokens, k)
    frozen = None if k == 1 else _state_before_final(w, tokens, k)
    assert abs(loss - _objective(w, tokens, k)) <= 1e-12 * max(1.0, abs(loss))
    kinds = set()
    for where, idx in _entries(tokens):
        fd = _fd(w, where, idx, tokens, k, frozen)
        g = _array(grads, where)[idx]
        assert abs(g - fd) <= 1e-7 + 1e-5 * abs(fd), (where, idx, g, fd)
        kinds.add(where[-1])
    return kinds


def test_loss_and_gradients_k1_match_finite_differences():
    kinds = _check_fd(1)
    assert {"embed_in", "embed_out", "s_z", *NAMES} <= kinds


@pytest.mark.parametrize("k", [2, 3])
def test_truncated_gradients_match_frozen_state_differences(k):
    _check_fd(k)


def test_truncation_drops_the_earlier_invocations():
    """k = 3: the recurrent weights' truncated gradient differs from the
    difference quotient of the untruncated objective; the input block's
    gradient is not zero (it flows through the final re-injection)."""
    k = 3
    w = _weights64()
    tokens = _tokens()
    _, grads = train.tbptl_step(SHAPE, w, tokens, k)
    gaps = []
    for l in range(SHAPE.n_in, SHAPE.n_in + SHAPE.n_rec):
        for name, idx in (("w_up", (5, 17)), ("w_q", (9, 30)), ("w_down", (60, 7))):
            fd_full = _fd(w, ("layer", l, name), idx, tokens, k, None)
            gaps.append(abs(grads["layers"][l][name][idx] - fd_full) / (abs(fd_full) + 1e-12))
    assert max(gaps) > 1e-3, gaps
    assert np.max(np.abs(grads["layers"][0]["w_q"])) > 0
    assert np.max(np.abs(grads["layers"][0]["w_up"])) > 0


def test_unused_embedding_rows_get_no_gradient():
    w = _weights64()
    tokens = _tokens()
    _, grads = train.tbptl_step(SHAPE, w, tokens, 2)
    unused = np.setdiff1d(np.arange(SHAPE.vocab), np.unique(tokens))
    assert np.all(grads["embed_in"][unused] == 0)
    # the LM head row of a token never predicted still gets the softmax term
    assert np.any(grads["embed_out"][unused] != 0)


def test_refusals():
    w = _weights64()
    with pytest.raises(ValueError):
        train.tbptl_step(SHAPE, w, _tokens(), 0)
    with pytest.raises(ValueError):
        train.tbptl_step(SHAPE, w, _tokens(T=1), 2)
