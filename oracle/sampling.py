"""Temperature sampling and the acceptance rule of self-speculative sampling.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module;
only the tests do.

"Dory1.0-4B: A Looped Normalized-GPT", Self-Speculative Decoding: a shallow
loop count drafts tokens, the full loop count verifies them in one pass, and
rejection sampling keeps the verifier's output distribution.  The pages name
the method without writing it out; this is the standard speculative-sampling
rule it refers to: draft token x at a position is kept with probability
min(1, p(x) / q(x)) (p the verifier's distribution there, q the drafter's);
at the first rejected position a token is drawn from the residual
max(0, p - q) (renormalised); if every draft is kept, one more token is drawn
from the verifier's distribution after the last draft.

Random numbers are inputs (uniforms in [0, 1)), so that the GPU path and this
one can be compared draw by draw.  Readings (listed in the design notes):
  * p = softmax(z / T) for temperature T > 0 (no top-k / top-p);
  * a draw from non-negative weights w with uniform u is the smallest index
    x whose running sum w_0 + ... + w_x exceeds u * sum(w) (indices in
    vocabulary order; if rounding leaves none, the last index with w > 0);
  * draft x is kept iff u * q(x) < p(x), i.e. u < p(x) / q(x);
  * a batch advances by its smallest count of leading kept drafts plus one:
    a sequence that kept more emits its kept draft at that last position
    (whether a position is emitted depends only on earlier positions, so
    every emitted token keeps the verifier's conditional distribution).
"""
from __future__ import annotations

import numpy as np


def softmax_t(z: np.ndarray, temperature: float) -> np.ndarray:
    """softmax(z / T) over the last axis, float64."""
    z = np.asarray(z, np.float64) / float(temperature)
    e = np.exp(z - z.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def sample_weights(w: np.ndarray, u: float, margins=None) -> int:
    """Inverse-CDF draw from non-negative weights w [V] with uniform u.
    margins (a list, optional) receives the distance of u * sum(w) to the
    nearest edge of the chosen interval, relative to sum(w): a draw whose
    margin is below another implementation's rounding may go either way."""
    w = np.asarray(w, np.float64)
    c = np.cumsum(w)
    t = u * c[-1]
    hit = np.nonzero(c > t)[0]
    x = int(hit[0]) if len(hit) else int(np.nonzero(w > 0)[0][-1])
    if margins is not None:
        lo = c[x - 1] if x > 0 else 0.0
        margins.append(min(abs(t - lo), abs(c[x] - t)) / c[-1])
    return x


def sample_tokens(z: np.ndarray, temperature: float, u: np.ndarray) -> np.ndarray:
    """One token per row of logits z [B, V] at temperature T with uniforms u [B]."""
    p = softmax_t(z, temperature)
    return np.array([sample_weights(p[b], u[b]) for b in range(p.shape[0])], np.int32)


def speculative_accept(p: np.ndarray, q: np.ndarray, drafts: np.ndarray, u_acc: np.ndarray,
                       u_res: np.ndarray, margins=None):
    """The acceptance step for a batch.

    p [B, gamma + 1, V]: verifier probabilities at the positions of the last
    emitted token and of each draft; q [B, gamma, V]: drafter probabilities
    the drafts were drawn from; drafts [B, gamma]; u_acc [B, gamma]; u_res
    [B].  Returns (tokens [B, n], n, kept [B] = leading kept drafts).
    margins (optional list) receives |u q - p| / p of every acceptance test
    and the margins of the draws (see sample_weights)."""
    B, G = drafts.shape
    kept = np.zeros(B, np.int64)
    for b in range(B):
        while kept[b] < G:
            i = kept[b]
            x = drafts[b, i]
            if margins is not None:
                margins.append(abs(u_acc[b, i] * q[b, i, x] - p[b, i, x]) / p[b, i, x])
            if u_acc[b, i] * q[b, i, x] < p[b, i, x]:
                kept[b] += 1
            else:
                break
    n = int(kept.min()) + 1
    out = np.zeros((B, n), np.int32)
    for b in range(B):
        out[b, :n - 1] = drafts[b, :n - 1]
        j = n - 1                                    # position of the last emitted token
        if kept[b] > j:
            out[b, j] = drafts[b, j]                 # a kept draft
        elif j < G:
            out[b, j] = sample_weights(np.maximum(p[b, j] - q[b, j], 0.0), u_res[b], margins)
        else:
            out[b, j] = sample_weights(p[b, G], u_res[b], margins)
    return out, n, kept
