"""Seeded synthetic inputs for the looped normalized-GPT forward pass.

This module is the one piece shared by the CPU oracle and the CUDA path: it
holds the model shapes, draws the random weights and token streams, and
rounds weights to bfloat16.  It contains none of the forward arithmetic
(no attention, no residual update, no loop schedule).

Shapes follow the model description in "Dory1.0-4B: A Looped Normalized-GPT"
(Architecture; Training with Loops; Long-Context Extension): an input block,
a shared recurrent block run k times, an output block; grouped-query
attention with a sliding window on three of every four layers.  Weight init
follows the nGPT convention used there (Architecture, and the re-normalisation
of matrices in Quantization-Aware Distillation): every matrix is Gaussian
N(0, 0.02^2) and then each vector along the model dimension d is scaled to
unit L2 norm.  The effective residual rate is 0.05 (Architecture).
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Shape:
    """Model dimensions.  Layer i (global index) uses full causal attention
    iff i % full_every == full_offset, else a sliding window of `window`
    keys (self included)."""
    name: str
    d: int
    n_in: int
    n_rec: int
    n_out: int
    n_q: int
    n_kv: int
    head_dim: int
    ffn: int
    vocab: int
    window: int
    full_every: int = 4
    full_offset: int = 3
    rope: bool = True
    rope_base_swa: float = 1.0e4
    rope_base_full: float = 1.0e7
    alpha_attn: float = 0.05
    alpha_mlp: float = 0.05
    s_qk: float = 1.0

    @property
    def n_layers(self) -> int:
        return self.n_in + self.n_rec + self.n_out

    @property
    def softmax_scale(self) -> float:
        return math.sqrt(self.head_dim)

    def is_full(self, layer: int) -> bool:
        return layer % self.full_every == self.full_offset

    def is_recurrent(self, layer: int) -> bool:
        return self.n_in <= layer < self.n_in + self.n_rec

    def replace(self, **kw) -> "Shape":
        return dataclasses.replace(self, **kw)


# The five workloads.  Sizes are fixed by the problem statement; the 4B-class
# dims match the paper's 72 = 16 + 40 + 16 layer split and 16 q / 4 kv heads.
TINY = Shape("tiny", d=128, n_in=1, n_rec=2, n_out=1, n_q=4, n_kv=2, head_dim=32,
             ffn=256, vocab=512, window=16)
# Test-only variant of TINY with a full-attention layer inside the loop.
TINY_LOOPFULL = Shape("tiny_loopfull", d=128, n_in=2, n_rec=4, n_out=2, n_q=4, n_kv=2,
                      head_dim=32, ffn=256, vocab=512, window=16)
SMALL = Shape("small", d=1024, n_in=4, n_rec=10, n_out=4, n_q=8, n_kv=2, head_dim=128,
              ffn=2816, vocab=32000, window=512)
DORY4B = Shape("dory4b", d=2048, n_in=16, n_rec=40, n_out=16, n_q=16, n_kv=4, head_dim=128,
               ffn=6144, vocab=131072, window=4096)

# Test-only variant of the 4B-class shape with 2 / 4 / 2 layers: every matrix
# and head has its full width (so every tile and the full vocabulary are
# exercised) while the CPU oracle stays fast.  Layers 3 and 7 are full.
DORY4B_SLIM = DORY4B.replace(name="dory4b_slim", n_in=2, n_rec=4, n_out=2)

SHAPES = {s.name: s for s in (TINY, TINY_LOOPFULL, SMALL, DORY4B, DORY4B_SLIM)}
SHAPE_ID = {"tiny": 0, "small": 1, "dory4b": 2, "tiny_loopfull": 100, "dory4b_slim": 102}

# Tensor ids used to derive one independent seed per weight tensor.
_TID = {"embed_in": 0, "embed_out": 1, "w_q": 2, "w_k": 3, "w_v": 4, "w_g": 5,
        "w_o": 6, "w_up": 7, "w_sl": 8, "w_down": 9}


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even), returned
    as float32 arrays whose values are exactly representable in bfloat16."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
         & np.uint32(0xFFFF0000))
    return r.view(np.float32)


def _gauss(shape_id: int, layer: int, tid: int, size) -> np.ndarray:
    rng = np.random.default_rng(np.random.SeedSequence([shape_id, layer + 1, tid]))
    return rng.standard_normal(size, dtype=np.float32) * np.float32(0.02)


def _unit_rows(w: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(w.astype(np.float64) ** 2, axis=1, keepdims=True))
    return (w / n).astype(np.float32)


def layer_weights(shape: Shape, layer: int, shape_id: int | None = None) -> dict:
    """Weights of one layer, bf16-exact float32.  Matrices are [out, in].

    Rows of W_q, W_k, W_v, W_g, W_up, W_sl (vectors along d) and columns of
    W_o, W_down (also vectors along d) have unit L2 norm."""
    sid = SHAPE_ID[shape.name] if shape_id is None else shape_id
    d, hq, hk, F = shape.d, shape.n_q * shape.head_dim, shape.n_kv * shape.head_dim, shape.ffn
    out = {}
    for name, rows in (("w_q", hq), ("w_k", hk), ("w_v", hk), ("w_g", hq),
                       ("w_up", F), ("w_sl", F)):
        out[name] = round_bf16(_unit_rows(_gauss(sid, layer, _TID[name], (rows, d))))
    for name, cols in (("w_o", hq), ("w_down", F)):
        # draw the transpose so the unit vectors along d are contiguous
        out[name] = np.ascontiguousarray(
            round_bf16(_unit_rows(_gauss(sid, layer, _TID[name], (cols, d)))).T)
    out["alpha_attn"] = np.full(d, shape.alpha_attn, np.float32)
    out["alpha_mlp"] = np.full(d, shape.alpha_mlp, np.float32)
    out["s_qk"] = np.full(shape.head_dim, shape.s_qk, np.float32)
    return out


def embeddings(shape: Shape, shape_id: int | None = None) -> dict:
    sid = SHAPE_ID[shape.name] if shape_id is None else shape_id
    V, d = shape.vocab, shape.d
    return {
        "embed_in": round_bf16(_unit_rows(_gauss(sid, -1, _TID["embed_in"], (V, d)))),
        "embed_out": round_bf16(_unit_rows(_gauss(sid, -1, _TID["embed_out"], (V, d)))),
        "s_z": np.ones(V, np.float32),
    }


_CACHE = {}


def make_weights(shape: Shape, shape_id: int | None = None, workers: int = 1) -> dict:
    """All weights of a model: {'embed_in', 'embed_out', 's_z', 'layers': [...]}.

    workers > 1 draws the tensors on that many threads (each tensor has its
    own seed, so the values do not depend on the thread count).  Shallow
    models of 1024 or more wide (the test-sized cuts of the wide shapes,
    seconds to draw) are drawn once per process: each call returns new dicts
    around the same arrays, which callers must not modify in place."""
    key = (repr(shape), shape_id)
    if shape.d >= 1024 and shape.n_layers <= 8:
        if key not in _CACHE:
            _CACHE[key] = _draw(shape, shape_id, workers)
        base = _CACHE[key]
        w = {k: v for k, v in base.items() if k != "layers"}
        w["layers"] = [dict(lw) for lw in base["layers"]]
        return w
    return _draw(shape, shape_id, workers)


def _draw(shape: Shape, shape_id: int | None, workers: int) -> dict:
    if workers <= 1:
        w = embeddings(shape, shape_id)
        w["layers"] = [layer_weights(shape, l, shape_id) for l in range(shape.n_layers)]
        return w
    from concurrent.futures import ThreadPoolExecutor
    sid = SHAPE_ID[shape.name] if shape_id is None else shape_id
    V, d = shape.vocab, shape.d
    emb = lambda name: round_bf16(_unit_rows(_gauss(sid, -1, _TID[name], (V, d))))
    with ThreadPoolExecutor(workers) as ex:
        e_in, e_out = ex.submit(emb, "embed_in"), ex.submit(emb, "embed_out")
        layers = list(ex.map(lambda l: layer_weights(shape, l, shape_id), range(shape.n_layers)))
        w = {"embed_in": e_in.result(), "embed_out": e_out.result(), "s_z": np.ones(V, np.float32),
             "layers": layers}
    return w


def make_weights_lazy(shape: Shape, shape_id: int | None = None) -> dict:
    """Like make_weights, but 'layers' is a generator that draws one layer at
    a time (for shapes whose weights do not fit in host memory at once)."""
    w = embeddings(shape, shape_id)
    w["layers"] = (layer_weights(shape, l, shape_id) for l in range(shape.n_layers))
    return w


def make_weights_torch(shape: Shape, device="cuda", seed: int = 0) -> dict:
    """Weights with the same distribution as make_weights (Gaussian
    N(0, 0.02^2), unit vectors along d, bf16), drawn on the GPU by torch's
    seeded generator: a fast stand-in for timing shapes too large to draw on
    the host.  Values differ from make_weights'; no parity check uses them."""
    import torch
    g = torch.Generator(device=device).manual_seed(seed)
    d, hq, hk, F = shape.d, shape.n_q * shape.head_dim, shape.n_kv * shape.head_dim, shape.ffn

    def unit_rows(rows, cols):
        w = torch.randn(rows, cols, device=device, generator=g, dtype=torch.float32) * 0.02
        return (w / w.norm(dim=1, keepdim=True)).to(torch.bfloat16)

    out = {"embed_in": unit_rows(shape.vocab, d), "embed_out": unit_rows(shape.vocab, d),
           "s_z": torch.ones(shape.vocab, device=device)}

    def layer(l):
        lw = {n: unit_rows(r, d) for n, r in (("w_q", hq), ("w_k", hk), ("w_v", hk), ("w_g", hq),
                                                ("w_up", F), ("w_sl", F))}
        lw["w_o"] = unit_rows(hq, d).t().contiguous()
        lw["w_down"] = unit_rows(F, d).t().contiguous()
        lw["alpha_attn"] = torch.full((d,), shape.alpha_attn, device=device)
        lw["alpha_mlp"] = torch.full((d,), shape.alpha_mlp, device=device)
        lw["s_qk"] = torch.full((shape.head_dim,), shape.s_qk, device=device)
        return lw

    out["layers"] = (layer(l) for l in range(shape.n_layers))
    return out


def tokens(shape: Shape, batch: int, length: int, seed: int = 0) -> np.ndarray:
    """Token ids uniform over the vocabulary, int32 [batch, length]."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, shape.vocab, size=(batch, length), dtype=np.int64).astype(np.int32)
