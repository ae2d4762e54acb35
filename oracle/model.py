"""Plain CPU definition of the looped normalized-GPT forward pass.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module;
only the tests, the smoke check and the benchmark's CPU-baseline leg do.

Written from "Dory1.0-4B: A Looped Normalized-GPT":
  * Architecture: nGPT backbone (hidden states on the unit sphere, residual
    update rule), L2 normalisation of the concatenated gated attention output
    before the output projection and of the SwiGLU activation before the down
    projection, an input-dependent sigmoid attention-output gate, grouped-query
    attention, a 3:1 sliding-window : full interleave.
  * Training with Loops: input block once, shared recurrent block k times,
    output block once; the state starts as a copy of the input block's output x,
    x is added before every invocation, normalisation at both boundaries, no
    adapter weights and no outer residual.
  * Long-Context Extension: RoPE bases 1e4 (sliding window) and 1e7 (full).
  * Last-Loop KV Caching: per-loop caches (loop-i queries see loop-i keys of
    earlier tokens) versus one cache per recurrent layer that keeps the final
    loop's entries; current-step tokens are always seen as current-loop values.

Readings where the pages are silent (each is listed in the design notes):
  * recurrence: s_0 = x;  s_i = N(F(N(s_{i-1} + x)));  output block gets s_k.
  * nGPT update: h <- N(h + alpha * (N(y) - h)), alpha = effective rate.
  * gate: elementwise sigmoid(W_g h) over the n_q*head_dim attention output,
    applied before the concatenation norm.
  * SwiGLU: m = (W_up h) * SiLU(W_sl h), all SwiGLU scales 1.
  * RoPE: rotate-half over the whole head, absolute positions from 0, applied
    before the per-head q/k normalisation, then scaled by s_qk.
  * window W counts the query itself: key j is visible from t iff
    j <= t and t - j < W.
  * softmax scale sqrt(head_dim) (unit q, k); logits = s_z * (E_out h).
  * N(v) = v / sqrt(max(sum(v^2), 1e-12)).

Parity pins live in tests/test_oracle_pins.py.  Precision: float64 by
default; float32 for large shapes (BLAS speed).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from .sampling import sample_weights, softmax_t, speculative_accept

LAST_LOOP = 0
PER_LOOP = 1


def l2n(v: np.ndarray) -> np.ndarray:
    """Per-token L2 normalisation along the last axis (nGPT's N)."""
    s = np.sum(v * v, axis=-1, keepdims=True)
    return v / np.sqrt(np.maximum(s, 1e-12))


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def silu(x):
    return x * sigmoid(x)


def rope(x: np.ndarray, pos: np.ndarray, base: float) -> np.ndarray:
    """Rotary position embedding, rotate-half convention over the full head.

    x: [..., T, dh], pos: [T] integer positions.  Pair (i, i + dh/2) is rotated
    by the angle pos * base^(-2i/dh)."""
    dh = x.shape[-1]
    half = dh // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = base ** (-2.0 * i / dh)
    ang = pos.astype(np.float64)[:, None] * inv_freq[None, :]          # [T, half]
    c = np.cos(ang).astype(x.dtype)
    s = np.sin(ang).astype(x.dtype)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def ngpt_update(h: np.ndarray, y: np.ndarray, alpha: np.ndarray) -> np.ndarray:
    """nGPT residual step: move h towards the normalised sublayer output."""
    return l2n(h + alpha * (l2n(y) - h))


def attention(qh, kh, vh, q_pos, k_pos, window, full, scale):
    """Masked softmax attention for one sequence and one query head.

    qh [C, dh], kh/vh [L, dh] with key positions k_pos [L].  Key j is visible
    from query t iff k_pos[j] <= q_pos[t] and, for a sliding-window layer,
    q_pos[t] - k_pos[j] < window.  Softmax in the array's precision."""
    s = scale * (qh @ kh.T)                                            # [C, L]
    rel = q_pos[:, None] - k_pos[None, :]
    allowed = rel >= 0
    if not full:
        allowed &= rel < window
    s = np.where(allowed, s, -np.inf)
    s = s - np.max(s, axis=1, keepdims=True)
    p = np.exp(s)
    p = p / np.sum(p, axis=1, keepdims=True)
    return p @ vh


def loop_schedule(x: np.ndarray, k: int, block):
    """Boundary transforms around the shared block: s_0 = x; for i = 1..k the
    block sees N(s_{i-1} + x) (tagged with loop index i) and s_i is the
    normalised block output.  Returns s_k."""
    s = x
    for i in range(1, k + 1):
        s = l2n(block(l2n(s + x), i))
    return s


def kv_bytes(shape, max_batch: int, max_ctx: int, k: int, cache_mode: int,
             elem_bytes: int = 2) -> int:
    """Bytes of K and V held for `max_batch` sequences of `max_ctx` positions.

    Sliding-window layers keep only the last `window` positions.  Recurrent
    layers keep k slices in per-loop mode, one otherwise; input and output
    layers keep one."""
    per_pos = 2 * shape.n_kv * shape.head_dim * elem_bytes
    total = 0
    for l in range(shape.n_layers):
        slots = max_ctx if shape.is_full(l) else min(max_ctx, shape.window)
        mult = k if (cache_mode == PER_LOOP and shape.is_recurrent(l)) else 1
        total += mult * slots * per_pos
    return total * max_batch


def slot_positions(written_positions, n_slots: int) -> np.ndarray:
    """Ring-slot map: slot s holds the latest written position p with
    p mod n_slots == s, or -1 if none was written."""
    out = np.full(n_slots, -1, np.int64)
    for p in sorted(written_positions):
        out[p % n_slots] = p
    return out


@dataclass
class _Cache:
    k: np.ndarray       # [B, n_kv, L, dh]: keys of positions first .. first + L - 1
    v: np.ndarray
    first: int = 0      # sliding-window layers drop keys no later query can see


@dataclass
class Trace:
    """Optional record of intermediate states for pins."""
    norms: list = field(default_factory=list)
    layer_apps: int = 0


class Oracle:
    """Stateful looped-nGPT model over a batch of equal-length sequences."""

    def __init__(self, shape, weights: dict, dtype=np.float64):
        self.shape = shape
        self.dtype = dtype
        self.w = self._cast(weights, dtype)
        self.trace = None
        self.reset()

    @staticmethod
    def _cast(weights, dtype):
        out = {k: np.asarray(v, dtype) for k, v in weights.items() if k != "layers"}
        out["layers"] = [{k: np.asarray(v, dtype) for k, v in lw.items()}
                         for lw in weights["layers"]]
        return out

    # ------------------------------------------------------------------ state
    def reset(self):
        self.length = 0
        self.batch = None
        self.k_bound = None
        self.mode_bound = None
        self.cache = {}            # (layer, slice) -> _Cache
        self.written = {}          # (layer, slice) -> list of positions
        self.window_slack = 0      # extra window positions kept (speculative verification)

    def _slice(self, layer, loop, mode):
        if loop is not None and mode == PER_LOOP:
            return loop
        return 0

    # ------------------------------------------------------------- sublayers
    def attn_sublayer(self, l, h, pos, loop, mode, k):
        sh, w = self.shape, self.w["layers"][l]
        B, C, _ = h.shape
        dh, nq, nkv = sh.head_dim, sh.n_q, sh.n_kv
        G = nq // nkv
        full = sh.is_full(l)
        base = sh.rope_base_full if full else sh.rope_base_swa
        q = (h @ w["w_q"].T).reshape(B, C, nq, dh).transpose(0, 2, 1, 3)    # [B,nq,C,dh]
        kk = (h @ w["w_k"].T).reshape(B, C, nkv, dh).transpose(0, 2, 1, 3)
        v = (h @ w["w_v"].T).reshape(B, C, nkv, dh).transpose(0, 2, 1, 3)
        g = h @ w["w_g"].T                                                  # [B,C,nq*dh]
        if sh.rope:
            q = rope(q, pos, base)
            kk = rope(kk, pos, base)
        qh = w["s_qk"] * l2n(q)
        kh = w["s_qk"] * l2n(kk)
        sl = self._slice(l, loop, mode)
        past = self.cache.get((l, sl))
        P0 = pos[0]
        if past is not None and P0 > past.first:
            n_old = P0 - past.first
            k_all = np.concatenate([past.k[:, :, :n_old], kh], axis=2)
            v_all = np.concatenate([past.v[:, :, :n_old], v], axis=2)
            k_pos = np.arange(past.first, P0 + C)
        else:
            k_all, v_all, k_pos = kh, v, pos
        o = np.empty((B, nq, C, dh), self.dtype)
        for b in range(B):
            for hq in range(nq):
                grp = hq // G
                o[b, hq] = attention(qh[b, hq], k_all[b, grp], v_all[b, grp], pos, k_pos,
                                     sh.window, full, sh.softmax_scale)
        o = o.transpose(0, 2, 1, 3).reshape(B, C, nq * dh)
        a = l2n(o * sigmoid(g))
        y = a @ w["w_o"].T
        h = ngpt_update(h, y, w["alpha_attn"])
        # cache store: last-loop keeps only the final loop, per-loop every loop
        store = (loop is None) or (mode == PER_LOOP) or (loop == k)
        if store:
            self._store(l, sl, kh, v, P0)
        return h

    def mlp_sublayer(self, l, h):
        w = self.w["layers"][l]
        m = (h @ w["w_up"].T) * silu(h @ w["w_sl"].T)
        y = l2n(m) @ w["w_down"].T
        return ngpt_update(h, y, w["alpha_mlp"])

    def layer(self, l, h, pos, loop, mode, k):
        h = self.attn_sublayer(l, h, pos, loop, mode, k)
        self._note(h)
        h = self.mlp_sublayer(l, h)
        self._note(h)
        if self.trace is not None:
            self.trace.layer_apps += 1
        return h

    def _note(self, h):
        if self.trace is not None:
            self.trace.norms.append(np.sqrt(np.sum(h * h, axis=-1)))

    def _store(self, l, sl, kh, v, P0):
        B, nkv, C, dh = kh.shape
        c = self.cache.get((l, sl))
        if c is None:
            c = _Cache(np.zeros((B, nkv, 0, dh), self.dtype), np.zeros((B, nkv, 0, dh), self.dtype),
                       P0)
        # positions >= P0 are (re)written; earlier ones are kept
        n_old = P0 - c.first
        k = np.concatenate([c.k[:, :, :n_old], kh], axis=2)
        v = np.concatenate([c.v[:, :, :n_old], v], axis=2)
        first = c.first
        if not self.shape.is_full(l):
            # keep the last W positions: a query at position t >= P0 + C sees
            # keys j > t - W only, so older keys are never read again (unless
            # the length is rolled back, for which window_slack keeps more)
            drop = max(0, P0 + C - self.shape.window - self.window_slack - first)
            k, v, first = k[:, :, drop:], v[:, :, drop:], first + drop
        self.cache[(l, sl)] = _Cache(k, v, first)
        self.written.setdefault((l, sl), set()).update(range(P0, P0 + C))

    def restore(self, length: int, mode: int, k: int, caches: dict):
        """Start from a saved cache state, to replay single steps at contexts
        too long to prefill here.  caches maps (layer, slice) to (K, V, first):
        arrays [B, n_kv, L, dh] holding positions first .. first + L - 1 of
        every sequence, L = length - first.  Slices are numbered as in step():
        loop index 1..k for recurrent layers under per-loop caching, else 0.
        Last-Loop KV Caching fixes what each slice holds; the caller supplies
        the values."""
        self.reset()
        self.length = length
        self.mode_bound = mode
        if mode == PER_LOOP:
            self.k_bound = k
        for (l, sl), (kk, vv, first) in caches.items():
            kk, vv = np.asarray(kk, self.dtype), np.asarray(vv, self.dtype)
            if kk.shape != vv.shape or first + kk.shape[2] != length:
                raise ValueError("cache slice does not end at the current length")
            self.batch = kk.shape[0]
            self.cache[(l, sl)] = _Cache(kk, vv, first)
            self.written[(l, sl)] = set(range(first, length))

    # --------------------------------------------------------------- forward
    def step(self, tokens: np.ndarray, k: int, mode: int, draft: bool = False):
        """Process tokens [B, C] at positions length .. length+C-1.
        Returns the final hidden states [B, C, d] (input to the LM head).
        draft=True: a shallower drafting pass of self-speculative decoding
        under per-loop caching (k at most the bound k; it reads and writes
        the slices of loops 1..k only)."""
        sh = self.shape
        tokens = np.asarray(tokens)
        B, C = tokens.shape
        if k < 1:
            raise ValueError("k must be >= 1")
        if self.batch is None:
            self.batch = B
        elif B != self.batch:
            raise ValueError("batch size changed")
        if mode == PER_LOOP and self.k_bound is not None and self.k_bound != k and not (
                draft and k < self.k_bound):
            raise ValueError("per-loop caching needs the same k for every step")
        if self.mode_bound is not None and self.mode_bound != mode:
            raise ValueError("cache mode changed")
        self.mode_bound = mode
        if mode == PER_LOOP and not draft:
            self.k_bound = k
        pos = np.arange(self.length, self.length + C)
        h = l2n(self.w["embed_in"][tokens])
        self._note(h)
        for l in range(sh.n_in):
            h = self.layer(l, h, pos, None, mode, k)
        x = h

        def block(u, i):
            for l in range(sh.n_in, sh.n_in + sh.n_rec):
                u = self.layer(l, u, pos, i, mode, k)
            return u

        h = loop_schedule(x, k, block)
        self._note(h)
        for l in range(sh.n_in + sh.n_rec, sh.n_layers):
            h = self.layer(l, h, pos, None, mode, k)
        self.length += C
        return h

    def logits(self, h: np.ndarray) -> np.ndarray:
        return self.w["s_z"] * (h @ self.w["embed_out"].T)

    def prefill(self, tokens, k, mode, all_logits=False):
        h = self.step(tokens, k, mode)
        hs = h if all_logits else h[:, -1:, :]
        return {"hidden": hs, "logits": self.logits(hs)}

    def decode(self, tokens, k, mode):
        """One decode step for tokens [B].  Returns hidden [B, d], logits
        [B, V] and the greedy next token (lowest index among equal maxima)."""
        h = self.step(np.asarray(tokens).reshape(-1, 1), k, mode)[:, 0, :]
        z = self.logits(h)
        return {"hidden": h, "logits": z, "next": np.argmax(z, axis=-1).astype(np.int32)}

    def speculative_step(self, token, k_draft: int, k_verify: int, gamma: int):
        """One step of greedy self-speculative decoding (Self-Speculative
        Decoding): the same weights draft gamma tokens autoregressively at
        k_draft, then verify them in one forward pass at k_verify over the
        last emitted token and the drafts; drafts are accepted while each
        equals the verifier's greedy token at the position before it, and the
        verifier's token at the first mismatch (or after the last draft) is
        emitted too.  Per-loop caching: drafting reads and writes only the
        slices of loops 1..k_draft, which the verifier shares; the verifier
        rewrites every slice of the positions it processes.  The batch
        advances by the smallest accepted count over its sequences plus one
        (a sequence that accepted more would emit the same token there).
        token: [B] the last emitted tokens (not yet in the cache).  Returns
        emitted tokens [B, n] and n."""
        if self.mode_bound != PER_LOOP or self.k_bound != k_verify or not (
                1 <= k_draft <= k_verify) or gamma < 1:
            raise ValueError("self-speculative decoding needs per-loop caching bound at k_verify")
        token = np.asarray(token).reshape(-1)
        L = self.length
        # drafting may not change what the verifier sees at positions < L:
        # keep the cache state and return to it before verifying (the
        # verifier recomputes and stores every slice of the positions it
        # processes; cached arrays are never modified in place)
        saved = (dict(self.cache), {key: set(v) for key, v in self.written.items()})
        drafts, cur = [], token
        for _ in range(gamma):
            h = self.step(cur.reshape(-1, 1), k_draft, PER_LOOP, draft=True)[:, 0]
            cur = np.argmax(self.logits(h), axis=-1)
            drafts.append(cur)
        drafts = np.stack(drafts, axis=1)                                  # [B, gamma]
        self.cache, self.written = saved
        self.length = L
        # the verifier stores positions L .. L + gamma; only L .. L + n - 1
        # stay, so window layers must keep gamma + 1 more positions than a
        # query at L + gamma + 1 would need
        self.window_slack = gamma + 1
        h = self.step(np.concatenate([token[:, None], drafts], axis=1), k_verify, PER_LOOP)
        self.window_slack = 0
        g = np.argmax(self.logits(h), axis=-1)                             # [B, gamma + 1]
        match = drafts == g[:, :gamma]
        accepted = np.where(match.all(axis=1), gamma, np.argmin(match, axis=1))
        n = int(accepted.min()) + 1
        out = np.concatenate([drafts[:, :n - 1], g[:, n - 1:n]], axis=1)
        self.length = L + n
        return out, n

    def speculative_sample_step(self, token, k_draft: int, k_verify: int, gamma: int,
                                temperature: float, u, margins=None):
        """One step of self-speculative decoding with rejection sampling
        (Self-Speculative Decoding; the rule is written out in
        oracle/sampling.py): gamma drafts drawn at k_draft from softmax(z / T),
        one verifying pass at k_verify, each draft kept with probability
        min(1, p / q), the first rejected position redrawn from the residual
        max(0, p - q), a last token from the verifier when every draft is kept.
        Cache handling as in speculative_step.  u [B, 2 gamma + 1]: uniforms,
        columns 0 .. gamma - 1 draw the drafts, gamma .. 2 gamma - 1 decide
        acceptance, 2 gamma draws the residual or last token.  Returns
        (tokens [B, n], n, kept drafts per sequence [B]); margins (optional
        list) collects the decision margins of oracle/sampling.py."""
        if self.mode_bound != PER_LOOP or self.k_bound != k_verify or not (
                1 <= k_draft <= k_verify) or gamma < 1 or temperature <= 0:
            raise ValueError("self-speculative sampling needs per-loop caching bound at k_verify")
        token = np.asarray(token).reshape(-1)
        u = np.asarray(u, np.float64)
        B, L = token.shape[0], self.length
        saved = (dict(self.cache), {key: set(v) for key, v in self.written.items()})
        drafts, qs, cur = [], [], token
        for i in range(gamma):
            h = self.step(cur.reshape(-1, 1), k_draft, PER_LOOP, draft=True)[:, 0]
            q = softmax_t(self.logits(h), temperature)
            cur = np.array([sample_weights(q[b], u[b, i], margins) for b in range(B)], np.int64)
            drafts.append(cur)
            qs.append(q)
        drafts, q = np.stack(drafts, axis=1), np.stack(qs, axis=1)
        self.cache, self.written = saved
        self.length = L
        self.window_slack = gamma + 1
        h = self.step(np.concatenate([token[:, None], drafts], axis=1), k_verify, PER_LOOP)
        self.window_slack = 0
        p = softmax_t(self.logits(h), temperature)                         # [B, gamma + 1, V]
        out, n, kept = speculative_accept(p, q, drafts, u[:, gamma:2 * gamma], u[:, 2 * gamma],
                                          margins)
        self.length = L + n
        return out, n, kept

    def stack_forward(self, tokens):
        """The same layers run once each as a plain (non-looped) stack,
        with no cache.  For the k = 1 equivalence pin."""
        sh = self.shape
        tokens = np.asarray(tokens)
        pos = np.arange(tokens.shape[1])
        saved = (self.cache, self.written)
        self.cache, self.written = {}, {}
        h = l2n(self.w["embed_in"][tokens])
        for l in range(sh.n_layers):
            h = self.layer(l, h, pos, None, LAST_LOOP, 1)
        self.cache, self.written = saved
        return h

    def kv_slot_positions(self, layer: int, sl: int = 0) -> np.ndarray:
        """Which position each ring slot of (layer, slice) holds; full layers
        have one slot per position of the context capacity."""
        sh = self.shape
        n = self.length if sh.is_full(layer) else min(self.length, sh.window)
        slots = max(n, 1) if sh.is_full(layer) else sh.window
        return slot_positions(self.written.get((layer, sl), ()), slots)
