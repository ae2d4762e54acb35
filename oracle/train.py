"""The truncated-backpropagation training step (TBPTL, depth one): loss and
parameter gradients of one batch.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module;
only the tests do.

"Dory1.0-4B: A Looped Normalized-GPT", Truncated Backpropagation: the
recurrent block's earlier invocations run without gradient tracking; the
final invocation and the input and output blocks are trained, the input
block receiving its gradient through the final invocation's re-injected
input; the next-token cross-entropy is taken only after the final
invocation (no intermediate-exit or early-loop losses).  The forward pass is
the one of oracle/model.py (Training with Loops, Architecture), written
again with torch tensors in float64 so that torch's reverse-mode
differentiation gives the gradient of that definition; the pins check it
against the numpy oracle's forward and against central finite differences
of the numpy oracle (tests/test_oracle_train_pins.py).

Readings (listed in the design notes):
  * every weight is a parameter: embeddings, LM head and s_z, the per-layer
    alpha and s_qk vectors as well as the matrices;
  * at k = 1 no invocation precedes the final one: the state s_0 is the
    input block's output x itself, so N(s_0 + x) = N(2 x) carries gradient
    through both terms (plain backpropagation);
  * at k >= 2 the state s_{k-1} after the earlier invocations is a constant
    of the step; x (the re-injected input) is not;
  * loss = mean over the B (T - 1) positions t < T - 1 of
    -log softmax(z_t)[token_{t+1}] with z = s_z * (E_out h).
"""
from __future__ import annotations

import math

import numpy as np
import torch

_MATS = ("w_q", "w_k", "w_v", "w_g", "w_o", "w_up", "w_sl", "w_down")
_VECS = ("alpha_attn", "alpha_mlp", "s_qk")


def _l2n(v):
    return v / torch.sqrt(torch.clamp((v * v).sum(-1, keepdim=True), min=1e-12))


def _rope(x, pos, base):
    """Rotate-half RoPE over the whole head (as oracle.model.rope)."""
    dh = x.shape[-1]
    half = dh // 2
    inv = torch.tensor([base ** (-2.0 * i / dh) for i in range(half)], dtype=torch.float64)
    ang = torch.tensor(pos, dtype=torch.float64)[:, None] * inv[None, :]
    c, s = torch.cos(ang), torch.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return torch.cat([x1 * c - x2 * s, x2 * c + x1 * s], dim=-1)


def _ngpt(h, y, alpha):
    return _l2n(h + alpha * (_l2n(y) - h))


def _layer(shape, w, l, h, pos):
    """One layer (attention then SwiGLU sublayer) over full sequences
    h [B, T, d], no cache: every query sees the causal (windowed) keys of
    the same pass."""
    B, T, _ = h.shape
    dh, nq, nkv = shape.head_dim, shape.n_q, shape.n_kv
    G = nq // nkv
    full = shape.is_full(l)
    base = shape.rope_base_full if full else shape.rope_base_swa
    q = (h @ w["w_q"].T).reshape(B, T, nq, dh).transpose(1, 2)
    k = (h @ w["w_k"].T).reshape(B, T, nkv, dh).transpose(1, 2)
    v = (h @ w["w_v"].T).reshape(B, T, nkv, dh).transpose(1, 2)
    g = h @ w["w_g"].T
    if shape.rope:
        q = _rope(q, pos, base)
        k = _rope(k, pos, base)
    qh = w["s_qk"] * _l2n(q)
    kh = w["s_qk"] * _l2n(k)
    rel = torch.tensor(pos)[:, None] - torch.tensor(pos)[None, :]
    allowed = rel >= 0
    if not full:
        allowed &= rel < shape.window
    kh = kh.repeat_interleave(G, dim=1)                  # query head hq reads group hq // G
    vv = v.repeat_interleave(G, dim=1)
    s = shape.softmax_scale * (qh @ kh.transpose(-1, -2))
    s = s.masked_fill(~allowed, -math.inf)
    o = torch.softmax(s, dim=-1) @ vv                    # [B, nq, T, dh]
    o = o.transpose(1, 2).reshape(B, T, nq * dh)
    a = _l2n(o * torch.sigmoid(g))
    h = _ngpt(h, a @ w["w_o"].T, w["alpha_attn"])
    m = (h @ w["w_up"].T) * torch.nn.functional.silu(h @ w["w_sl"].T)
    return _ngpt(h, _l2n(m) @ w["w_down"].T, w["alpha_mlp"])


def _params(weights):
    p = {n: torch.tensor(np.asarray(weights[n], np.float64), requires_grad=True)
         for n in ("embed_in", "embed_out", "s_z")}
    p["layers"] = [{n: torch.tensor(np.asarray(lw[n], np.float64), requires_grad=True)
                    for n in _MATS + _VECS} for lw in weights["layers"]]
    return p


def forward_loss(shape, p, tokens, k: int):
    """TBPTL-1 objective as a torch scalar (p: parameters as from _params)."""
    tokens = np.asarray(tokens)
    B, T = tokens.shape
    pos = np.arange(T)
    lay = p["layers"]
    h = _l2n(p["embed_in"][torch.tensor(tokens)])
    for l in range(shape.n_in):
        h = _layer(shape, lay[l], l, h, pos)
    x = h

    def block(u):
        for l in range(shape.n_in, shape.n_in + shape.n_rec):
            u = _layer(shape, lay[l], l, u, pos)
        return u

    if k == 1:
        s = x                                            # s_0 = x, tracked
    else:
        with torch.no_grad():                            # invocations 1 .. k-1
            s = x.detach()
            for _ in range(k - 1):
                s = _l2n(block(_l2n(s + x.detach())))
    h = _l2n(block(_l2n(s + x)))                         # the final invocation
    for l in range(shape.n_in + shape.n_rec, shape.n_layers):
        h = _layer(shape, lay[l], l, h, pos)
    z = p["s_z"] * (h @ p["embed_out"].T)                # [B, T, V]
    logp = torch.log_softmax(z[:, :-1], dim=-1)
    nxt = torch.tensor(tokens[:, 1:])
    return -logp.gather(-1, nxt[..., None]).mean()


def tbptl_step(shape, weights: dict, tokens, k: int):
    """Loss and gradients of one TBPTL-1 step.  weights: the oracle's weight
    dict; tokens [B, T] (T >= 2).  Returns (loss, grads) with grads in the
    weights' structure (float64 arrays)."""
    if k < 1:
        raise ValueError("k must be >= 1")
    if np.asarray(tokens).shape[1] < 2:
        raise ValueError("need at least two positions for a next-token loss")
    p = _params(weights)
    loss = forward_loss(shape, p, tokens, k)
    loss.backward()
    grads = {n: p[n].grad.numpy() for n in ("embed_in", "embed_out", "s_z")}
    grads["layers"] = [{n: lw[n].grad.numpy() if lw[n].grad is not None
                        else np.zeros(tuple(lw[n].shape)) for n in _MATS + _VECS}
                       for lw in p["layers"]]
    return float(loss.detach()), grads
