"""Python binding of libdory, the CUDA library behind include/dory.h.

Argument marshalling only: every step of the forward pass runs in the
library's kernels.  PyTorch is used for device memory and streams.  If the
library is not built, or no CUDA device is present, the compute calls raise;
there is no fallback path.

Low-level: the C functions under the same names (dory_create, dory_bind,
dory_prefill, dory_decode_step, dory_kv_bytes, ...), taking ctypes
structures and raw device pointers.  High-level: `Model`, which uploads a
weight dictionary, allocates the KV cache and workspace with torch and binds
them.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB

DORY_OK = 0
DORY_EINVAL = -1
DORY_ENOMEM = -2
DORY_ECUDA = -3
DORY_ECAPACITY = -4
DORY_EKMISMATCH = -5
DORY_EUNBOUND = -6
DORY_EDEVICE = -7
DORY_EUNSUPPORTED = -8

LAST_LOOP = 0
PER_LOOP = 1

QUANT_NONE = 0
QUANT_MXFP8 = 1
QUANT_NVFP4 = 2

KERNEL_CLASSES = ("embed", "rope", "qkvg_gemm", "attention", "kv_write", "o_gemm", "ngpt_update",
                  "upgate_gemm", "down_gemm", "boundary", "lm_head", "argmax")


class DoryConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("d", "n_in", "n_rec", "n_out", "n_q", "n_kv", "head_dim", "ffn", "vocab",
                 "window", "full_every", "full_offset", "rope")] + [
        ("rope_base_swa", ctypes.c_float), ("rope_base_full", ctypes.c_float),
        ("softmax_scale", ctypes.c_float)]


class DoryLayerWeights(ctypes.Structure):
    _fields_ = [("w_qkvg", ctypes.c_void_p), ("w_o", ctypes.c_void_p),
                ("w_upgate", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
                ("alpha_attn", ctypes.c_void_p), ("alpha_mlp", ctypes.c_void_p),
                ("s_qk", ctypes.c_void_p)]


class DoryWeights(ctypes.Structure):
    _fields_ = [("embed_in", ctypes.c_void_p), ("embed_out", ctypes.c_void_p),
                ("s_z", ctypes.c_void_p), ("layers", ctypes.POINTER(DoryLayerWeights))]


class DoryQMatrix(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("row_scale", ctypes.c_void_p)]


class DoryQLayer(ctypes.Structure):
    _fields_ = [("qkvg", DoryQMatrix), ("o", DoryQMatrix), ("upgate", DoryQMatrix),
                ("down", DoryQMatrix)]


class DoryError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} failed: {code} ({strerror(code)})")
        self.code = code


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGS = {
    "dory_create": (_I, [ctypes.POINTER(DoryConfig), ctypes.POINTER(DoryWeights), ctypes.POINTER(_P)]),
    "dory_kv_bytes": (ctypes.c_size_t, [ctypes.POINTER(DoryConfig), _I, _I, _I, _I]),
    "dory_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(DoryConfig), _I, _I]),
    "dory_bind": (_I, [_P, _P, ctypes.c_size_t, _P, ctypes.c_size_t, _I, _I, _I, _I, _I]),
    "dory_prefill": (_I, [_P, _P, _I, _I, _I, _I, _P, _I, _P]),
    "dory_decode_step": (_I, [_P, _P, _I, _I, _I, _P, _P, _P]),
    "dory_length": (_I, [_P, ctypes.POINTER(_I)]),
    "dory_reset": (_I, [_P]),
    "dory_set_length": (_I, [_P, _I, _I]),
    "dory_destroy": (_I, [_P]),
    "dory_strerror": (ctypes.c_char_p, [_I]),
    "dory_device_status": (_I, [_P, ctypes.POINTER(_I), _P]),
    "dory_last_launch_count": (_I, [_P, ctypes.POINTER(_I)]),
    "dory_set_tc_attention": (_I, [_P, _I]),
    "dory_set_fused_ngpt": (_I, [_P, _I]),
    "dory_debug_hidden": (_I, [_P, _P, _I, _P]),
    "dory_debug_kv_offset": (_I, [_P, _I, _I, _I, ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(_I)]),
    "dory_debug_gemm": (_I, [_P, _P, _P, _I, _I, _I, _I, _P]),
    "dory_debug_expire_wait": (_I, [_P, _I, _P]),
    "dory_speculative_step": (_I, [_P, _P, _I, _I, _I, _I, _P, ctypes.c_size_t, _P,
                                   ctypes.POINTER(_I), _P]),
    "dory_speculative_scratch_bytes": (ctypes.c_size_t, [_P, _I, _I]),
    "dory_speculative_sample_step": (_I, [_P, _P, _I, _I, _I, _I, ctypes.c_float, _P, _P,
                                          ctypes.c_size_t, _P, ctypes.POINTER(_I), _P, _P]),
    "dory_sample_tokens": (_I, [_P, _I, _I, ctypes.c_float, _P, _P, _P]),
    "dory_debug_speculative_layout": (_I, [_P, _I, _I, ctypes.POINTER(ctypes.c_size_t)]),
    "dory_copy_prefix": (_I, [_P, _I, ctypes.POINTER(_I), _I, _I, _P]),
    "dory_set_lengths": (_I, [_P, _I, ctypes.POINTER(_I)]),
    "dory_get_lengths": (_I, [_P, _I, ctypes.POINTER(_I)]),
    "dory_prefill_slot": (_I, [_P, _I, _P, _I, _I, _I, _P, _I, _P]),
    "dory_decode_step_ragged": (_I, [_P, _P, _I, _I, _I, _P, _P, _P]),
    "dory_decode_step_multi": (_I, [_P, _P, _I, ctypes.POINTER(_I), _I, _P, _P, _P]),
    "dory_step_mixed": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "dory_quant_bytes": (_I, [_I, _I, _I, ctypes.POINTER(ctypes.c_size_t),
                              ctypes.POINTER(ctypes.c_size_t)]),
    "dory_quantize_matrix": (_I, [_I, _P, _I, _I, _P, _P, _P, _P, _P]),
    "dory_set_quantized_weights": (_I, [_P, _I, ctypes.POINTER(DoryQLayer)]),
    "dory_set_quantized_swap": (_I, [_P, _I]),
    "dory_profile_begin": (_I, [_P, _I]),
    "dory_profile_end": (_I, [_P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(_I)]),
    "dory_debug_attention": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                  ctypes.c_float, _P, ctypes.c_size_t, _P]),
    "dory_debug_attention_scratch_bytes": (ctypes.c_size_t, [_I, _I, _I]),
    "dory_decode_attention_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                           _I, ctypes.c_float, _P]),
}


def lib():
    """The loaded libdory.so (built in-tree by __graft_entry__.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is not built; run __graft_entry__.build()")
        h = ctypes.CDLL(LIB)
        for name, (res, args) in _SIGS.items():
            f = getattr(h, name)
            f.restype = res
            f.argtypes = args
        _lib = h
    return _lib


def strerror(code: int) -> str:
    return lib().dory_strerror(code).decode()


def _check(fn, rc):
    if rc != DORY_OK:
        raise DoryError(fn, rc)


def config_from_shape(shape) -> DoryConfig:
    """DoryConfig from an object with the fields of synth.Shape."""
    return DoryConfig(d=shape.d, n_in=shape.n_in, n_rec=shape.n_rec, n_out=shape.n_out,
                      n_q=shape.n_q, n_kv=shape.n_kv, head_dim=shape.head_dim, ffn=shape.ffn,
                      vocab=shape.vocab, window=shape.window, full_every=shape.full_every,
                      full_offset=shape.full_offset, rope=1 if shape.rope else 0,
                      rope_base_swa=shape.rope_base_swa, rope_base_full=shape.rope_base_full,
                      softmax_scale=0.0)


def kv_bytes(cfg: DoryConfig, max_batch: int, max_ctx: int, k: int, cache_mode: int) -> int:
    return int(lib().dory_kv_bytes(ctypes.byref(cfg), max_batch, max_ctx, k, cache_mode))


def workspace_bytes(cfg: DoryConfig, max_batch: int, max_chunk: int) -> int:
    return int(lib().dory_workspace_bytes(ctypes.byref(cfg), max_batch, max_chunk))


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def quant_bytes(fmt: int, rows: int, K: int):
    """(codes bytes, block-scale bytes) of a rows x K matrix in format fmt."""
    cb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    _check("dory_quant_bytes", lib().dory_quant_bytes(fmt, rows, K, ctypes.byref(cb),
                                                      ctypes.byref(sb)))
    return cb.value, sb.value


def quantize_matrix(fmt: int, W, codes=None, scales=None, row_scale=None, deq=None, stream=None):
    """Quantises the bf16 device matrix W [rows, K] as one tensor
    (dory_quantize_matrix); allocates the outputs that are not given.
    Returns (codes uint8, scales uint8, row_scale fp32 [rows])."""
    import torch
    rows, K = W.shape
    cb, sb = quant_bytes(fmt, rows, K)
    dev = W.device
    codes = torch.empty(cb, dtype=torch.uint8, device=dev) if codes is None else codes
    scales = torch.empty(sb, dtype=torch.uint8, device=dev) if scales is None else scales
    row_scale = torch.empty(rows, dtype=torch.float32, device=dev) if row_scale is None else row_scale
    _check("dory_quantize_matrix",
           lib().dory_quantize_matrix(fmt, _ptr(W), rows, K, _ptr(codes), _ptr(scales),
                                      _ptr(row_scale), _ptr(deq), _stream_ptr(stream)))
    return codes, scales, row_scale


def sample_tokens(logits, temperature, u, out=None, stream=None):
    """One token per row of fp32 device logits [rows, V] drawn from
    softmax(logits / T) with the uniforms u (fp32 device [rows])."""
    import torch
    rows, V = logits.shape
    out = torch.empty((rows,), dtype=torch.int32, device=logits.device) if out is None else out
    _check("dory_sample_tokens", lib().dory_sample_tokens(_ptr(logits), rows, V, float(temperature),
                                                          _ptr(u), _ptr(out), _stream_ptr(stream)))
    return out


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


class Model:
    """Device-resident looped nGPT: weights, KV cache and workspace held as
    torch tensors, compute through libdory.

    weights: dict like synth.make_weights() returns (numpy or torch, values
    bf16-exact); matrices are uploaded as bf16, vectors as fp32."""

    def __init__(self, shape, weights, max_batch, max_ctx, max_chunk, k_max=1,
                 cache_mode=LAST_LOOP, device="cuda"):
        import torch
        if not torch.cuda.is_available():
            raise RuntimeError("libdory needs a CUDA device")
        self.shape = shape
        self.cfg = config_from_shape(shape)
        self.device = torch.device(device)
        L = lib()

        def bf(x):
            # always the model's own copy (quantize() rewrites it in place)
            t = torch.as_tensor(x)
            y = t.to(self.device, torch.bfloat16).contiguous()
            return y.clone() if y.data_ptr() == t.data_ptr() else y

        def f32(x):
            return torch.as_tensor(x).to(self.device, torch.float32).contiguous()

        self._keep = []
        self.embed_in = bf(weights["embed_in"])
        self.embed_out = bf(weights["embed_out"])
        self.s_z = f32(weights["s_z"]) if weights.get("s_z") is not None else None
        n = shape.n_layers
        self._layers = (DoryLayerWeights * n)()
        for l, lw in enumerate(weights["layers"]):
            qkvg = torch.cat([bf(lw["w_q"]), bf(lw["w_k"]), bf(lw["w_v"]), bf(lw["w_g"])], 0)
            upg = torch.cat([bf(lw["w_up"]), bf(lw["w_sl"])], 0)
            t = dict(qkvg=qkvg, o=bf(lw["w_o"]), upg=upg.contiguous(), down=bf(lw["w_down"]),
                     aa=f32(lw["alpha_attn"]), am=f32(lw["alpha_mlp"]), sqk=f32(lw["s_qk"]))
            self._keep.append(t)
            self._layers[l] = DoryLayerWeights(t["qkvg"].data_ptr(), t["o"].data_ptr(),
                                               t["upg"].data_ptr(), t["down"].data_ptr(),
                                               t["aa"].data_ptr(), t["am"].data_ptr(),
                                               t["sqk"].data_ptr())
        w = DoryWeights(self.embed_in.data_ptr(), self.embed_out.data_ptr(),
                        self.s_z.data_ptr() if self.s_z is not None else 0, self._layers)
        h = ctypes.c_void_p()
        _check("dory_create", L.dory_create(ctypes.byref(self.cfg), ctypes.byref(w), ctypes.byref(h)))
        self.handle = h
        self.bind(max_batch, max_ctx, max_chunk, k_max, cache_mode)

    def bind(self, max_batch, max_ctx, max_chunk, k_max=1, cache_mode=LAST_LOOP):
        import torch
        kvb = kv_bytes(self.cfg, max_batch, max_ctx, k_max, cache_mode)
        wsb = workspace_bytes(self.cfg, max_batch, max_chunk)
        if kvb == 0 or wsb == 0:
            raise DoryError("dory_kv_bytes/dory_workspace_bytes", DORY_EINVAL)
        self.kv = torch.zeros(kvb, dtype=torch.uint8, device=self.device)
        self.ws = torch.zeros(wsb, dtype=torch.uint8, device=self.device)
        _check("dory_bind", lib().dory_bind(self.handle, _ptr(self.kv), kvb, _ptr(self.ws), wsb,
                                            max_batch, max_ctx, max_chunk, k_max, cache_mode))
        self.max_batch, self.max_ctx, self.max_chunk = max_batch, max_ctx, max_chunk
        self.k_max, self.cache_mode = k_max, cache_mode

    # ------------------------------------------------------------- calls
    def prefill(self, tokens, k, cache_mode=None, all_logits=False, logits=None, stream=None):
        """tokens: int32 device tensor [B, T].  Returns fp32 logits
        [B, V] (last position) or [B, T, V]."""
        import torch
        B, T = tokens.shape
        mode = self.cache_mode if cache_mode is None else cache_mode
        if logits is None:
            shp = (B, T, self.shape.vocab) if all_logits else (B, self.shape.vocab)
            logits = torch.empty(shp, dtype=torch.float32, device=self.device)
        _check("dory_prefill", lib().dory_prefill(self.handle, _ptr(tokens), B, T, k, mode,
                                                  _ptr(logits), 1 if all_logits else 0,
                                                  _stream_ptr(stream)))
        return logits

    def decode(self, tokens, k, cache_mode=None, logits=None, next_tokens=None, stream=None):
        """tokens: int32 device tensor [B].  Returns (logits [B, V], next [B])."""
        import torch
        B = tokens.shape[0]
        mode = self.cache_mode if cache_mode is None else cache_mode
        if logits is None:
            logits = torch.empty((B, self.shape.vocab), dtype=torch.float32, device=self.device)
        if next_tokens is None:
            next_tokens = torch.empty((B,), dtype=torch.int32, device=self.device)
        _check("dory_decode_step", lib().dory_decode_step(self.handle, _ptr(tokens), B, k, mode,
                                                          _ptr(logits), _ptr(next_tokens),
                                                          _stream_ptr(stream)))
        return logits, next_tokens

    def quantize(self, fmt, stream=None):
        """Weight-only quantisation of every projection matrix (not the
        embeddings or the LM head), on the GPU: the few-row projections
        (decode) then stream the packed codes and block scales, and the
        model's bf16 matrices are overwritten with the dequantised values so
        that the larger projections compute with the same weights.  Each of
        W_q, W_k, W_v, W_g, W_o, W_up, W_sl, W_down is its own tensor (its
        own NVFP4 scale).  fmt QUANT_NONE switches the decode projections
        back to the bf16 matrices (which keep the dequantised values)."""
        import torch
        L = lib()
        if fmt == QUANT_NONE:
            _check("dory_set_quantized_weights", L.dory_set_quantized_weights(self.handle, 0, None))
            self._q = None
            return
        sh = self.shape
        hq, hk = sh.n_q * sh.head_dim, sh.n_kv * sh.head_dim
        parts = {"qkvg": (hq, hk, hk, hq), "o": (sh.d,), "upg": (sh.ffn, sh.ffn), "down": (sh.d,)}
        table = (DoryQLayer * sh.n_layers)()
        keep = []
        for l, t in enumerate(self._keep):
            mats = {}
            for name in ("qkvg", "o", "upg", "down"):
                W = t[name]
                rows, K = W.shape
                cb, sb = quant_bytes(fmt, rows, K)
                codes = torch.empty(cb, dtype=torch.uint8, device=self.device)
                scales = torch.empty(sb, dtype=torch.uint8, device=self.device)
                rs = torch.empty(rows, dtype=torch.float32, device=self.device)
                r0 = 0
                for nr in parts[name]:
                    quantize_matrix(fmt, W[r0:r0 + nr], codes[r0 * cb // rows:(r0 + nr) * cb // rows],
                                    scales[r0 * sb // rows:(r0 + nr) * sb // rows], rs[r0:r0 + nr],
                                    deq=W[r0:r0 + nr], stream=stream)
                    r0 += nr
                mats[name] = DoryQMatrix(codes.data_ptr(), scales.data_ptr(), rs.data_ptr())
                keep.append((codes, scales, rs))
            table[l] = DoryQLayer(mats["qkvg"], mats["o"], mats["upg"], mats["down"])
        _check("dory_set_quantized_weights", L.dory_set_quantized_weights(self.handle, fmt, table))
        self._q = keep

    def set_quantized_swap(self, stream_codes):
        """Whether decode steps of 2-128 sequences expand the quantised
        codes inside the swapped GEMM (True) or read the dequantised bf16
        matrices (False, the default); the results are bit-identical."""
        _check("dory_set_quantized_swap",
               lib().dory_set_quantized_swap(self.handle, 1 if stream_codes else 0))

    def set_lengths(self, lengths):
        """Per-sequence lengths of batch slots 0 .. len(lengths) - 1."""
        arr = (ctypes.c_int * len(lengths))(*[int(x) for x in lengths])
        _check("dory_set_lengths", lib().dory_set_lengths(self.handle, len(lengths), arr))

    def lengths(self, B):
        arr = (ctypes.c_int * B)()
        _check("dory_get_lengths", lib().dory_get_lengths(self.handle, B, arr))
        return list(arr)

    def prefill_slot(self, slot, tokens, k, cache_mode=None, all_logits=False, logits=None,
                     stream=None):
        """Prefill of one sequence (tokens int32 device [T]) in batch slot
        `slot`, from that slot's own length.  Returns fp32 logits [V] (last
        position) or [T, V]."""
        import torch
        T = tokens.shape[-1]
        mode = self.cache_mode if cache_mode is None else cache_mode
        if logits is None:
            shp = (T, self.shape.vocab) if all_logits else (self.shape.vocab,)
            logits = torch.empty(shp, dtype=torch.float32, device=self.device)
        _check("dory_prefill_slot", lib().dory_prefill_slot(
            self.handle, slot, _ptr(tokens), T, k, mode, _ptr(logits), 1 if all_logits else 0,
            _stream_ptr(stream)))
        return logits

    def decode_ragged(self, tokens, k, cache_mode=None, logits=None, next_tokens=None,
                      stream=None):
        """One decode step of slots 0 .. B-1 at their own lengths.  Returns
        (logits [B, V], next [B])."""
        import torch
        B = tokens.shape[0]
        mode = self.cache_mode if cache_mode is None else cache_mode
        if logits is None:
            logits = torch.empty((B, self.shape.vocab), dtype=torch.float32, device=self.device)
        if next_tokens is None:
            next_tokens = torch.empty((B,), dtype=torch.int32, device=self.device)
        _check("dory_decode_step_ragged", lib().dory_decode_step_ragged(
            self.handle, _ptr(tokens), B, k, mode, _ptr(logits), _ptr(next_tokens),
            _stream_ptr(stream)))
        return logits, next_tokens

    def decode_multi(self, tokens, ks, cache_mode=None, logits=None, next_tokens=None,
                     stream=None):
        """One decode step of slots 0 .. B-1 at their own lengths and their
        own loop counts ks (last-loop cache).  Returns (logits, next)."""
        import torch
        B = tokens.shape[0]
        mode = self.cache_mode if cache_mode is None else cache_mode
        if logits is None:
            logits = torch.empty((B, self.shape.vocab), dtype=torch.float32, device=self.device)
        if next_tokens is None:
            next_tokens = torch.empty((B,), dtype=torch.int32, device=self.device)
        arr = (ctypes.c_int * B)(*[int(x) for x in ks])
        _check("dory_decode_step_multi", lib().dory_decode_step_multi(
            self.handle, _ptr(tokens), B, arr, mode, _ptr(logits), _ptr(next_tokens),
            _stream_ptr(stream)))
        return logits, next_tokens

    def step_mixed(self, dec_tokens, slot, chunk, k, cache_mode=None, stream=None):
        """One forward pass over decode tokens of slots 0 .. Bd-1 (int32
        device [Bd]) and a chunk (int32 device [C]) of the sequence in slot
        `slot`.  Returns (logits [Bd + 1, V]: decode rows then the chunk's
        last position, greedy next tokens [Bd] or None)."""
        import torch
        Bd, C = dec_tokens.shape[0], chunk.shape[0]
        mode = self.cache_mode if cache_mode is None else cache_mode
        toks = torch.cat([dec_tokens, chunk]).to(torch.int32).contiguous()
        logits = torch.empty((Bd + 1, self.shape.vocab), dtype=torch.float32, device=self.device)
        nxt = torch.empty((max(Bd, 1),), dtype=torch.int32, device=self.device)
        _check("dory_step_mixed", lib().dory_step_mixed(
            self.handle, _ptr(toks), Bd, slot, C, k, mode, _ptr(logits),
            _ptr(nxt) if Bd > 0 else None, _stream_ptr(stream)))
        return logits, (nxt[:Bd] if Bd > 0 else None)

    def copy_prefix(self, src, dst, length, stream=None):
        """Copy the cached positions 0 .. length-1 of sequence src into the
        sequences listed in dst (prefix caching); then set_length()."""
        arr = (ctypes.c_int * len(dst))(*dst)
        _check("dory_copy_prefix", lib().dory_copy_prefix(self.handle, src, arr, len(dst), length,
                                                          _stream_ptr(stream)))

    def speculative_step(self, tokens, k_draft, k_verify, gamma, stream=None):
        """One greedy self-speculative step: tokens int32 device [B] (the last
        emitted tokens).  Returns (emitted int32 device [B, n], n)."""
        import torch
        B = tokens.shape[0]
        nb = int(lib().dory_speculative_scratch_bytes(self.handle, B, gamma))
        if nb == 0:
            raise DoryError("dory_speculative_scratch_bytes", DORY_EINVAL)
        if getattr(self, "_spec_scratch", None) is None or self._spec_scratch.numel() < nb:
            self._spec_scratch = torch.empty(nb, dtype=torch.uint8, device=self.device)
        out = torch.empty((B, gamma + 1), dtype=torch.int32, device=self.device)
        n = ctypes.c_int()
        _check("dory_speculative_step", lib().dory_speculative_step(
            self.handle, _ptr(tokens), B, k_draft, k_verify, gamma, _ptr(self._spec_scratch), nb,
            _ptr(out), ctypes.byref(n), _stream_ptr(stream)))
        return out[:, :n.value], n.value

    def speculative_sample_step(self, tokens, k_draft, k_verify, gamma, temperature, u,
                                stream=None):
        """One self-speculative step with rejection sampling: tokens int32
        device [B]; u fp32 device [B, 2 gamma + 1] uniforms.  Returns
        (emitted int32 device [B, n], n, kept drafts int32 device [B])."""
        import torch
        B = tokens.shape[0]
        nb = int(lib().dory_speculative_scratch_bytes(self.handle, B, gamma))
        if nb == 0:
            raise DoryError("dory_speculative_scratch_bytes", DORY_EINVAL)
        if getattr(self, "_spec_scratch", None) is None or self._spec_scratch.numel() < nb:
            self._spec_scratch = torch.empty(nb, dtype=torch.uint8, device=self.device)
        out = torch.empty((B, gamma + 1), dtype=torch.int32, device=self.device)
        kept = torch.empty((B,), dtype=torch.int32, device=self.device)
        n = ctypes.c_int()
        _check("dory_speculative_sample_step", lib().dory_speculative_sample_step(
            self.handle, _ptr(tokens), B, k_draft, k_verify, gamma, float(temperature), _ptr(u),
            _ptr(self._spec_scratch), nb, _ptr(out), ctypes.byref(n), _ptr(kept),
            _stream_ptr(stream)))
        return out[:, :n.value], n.value, kept

    def hidden(self, rows, stream=None):
        """Final hidden states (LM-head input) of the last chunk, [rows, d] fp32."""
        import torch
        out = torch.empty((rows, self.shape.d), dtype=torch.float32, device=self.device)
        _check("dory_debug_hidden", lib().dory_debug_hidden(self.handle, _ptr(out), rows,
                                                            _stream_ptr(stream)))
        return out

    def kv_block(self, layer, slc, which):
        """View of the K (which=0) or V (which=1) block of (layer, slice):
        bf16 [max_batch, n_kv, slots, head_dim]."""
        import torch
        off = ctypes.c_size_t()
        slots = ctypes.c_int()
        _check("dory_debug_kv_offset", lib().dory_debug_kv_offset(
            self.handle, layer, slc, which, ctypes.byref(off), ctypes.byref(slots)))
        sh = self.shape
        n = self.max_batch * sh.n_kv * slots.value * sh.head_dim
        raw = self.kv[off.value: off.value + 2 * n]
        return raw.view(torch.bfloat16).view(self.max_batch, sh.n_kv, slots.value, sh.head_dim)

    def length(self):
        v = ctypes.c_int()
        _check("dory_length", lib().dory_length(self.handle, ctypes.byref(v)))
        return v.value

    def set_length(self, batch, length):
        """Declare that the KV cache already holds `length` positions of
        `batch` sequences (contents are the caller's)."""
        _check("dory_set_length", lib().dory_set_length(self.handle, batch, length))

    def reset(self):
        _check("dory_reset", lib().dory_reset(self.handle))

    def device_status(self, stream=None):
        v = ctypes.c_int()
        _check("dory_device_status", lib().dory_device_status(self.handle, ctypes.byref(v),
                                                              _stream_ptr(stream)))
        return v.value

    def expire_wait(self, limit_us=1000, stream=None):
        """Test-only: one kernel whose bounded wait is never completed gives up
        after limit_us and sets the device status word (code 0x71)."""
        _check("dory_debug_expire_wait", lib().dory_debug_expire_wait(self.handle, limit_us,
                                                                      _stream_ptr(stream)))

    def set_tc_attention(self, enable: bool):
        """Prefill attention on tcgen05 where its tile rules hold (default)
        or always on the mma.sync kernel."""
        _check("dory_set_tc_attention", lib().dory_set_tc_attention(self.handle, 1 if enable else 0))

    def set_fused_ngpt(self, enable: bool):
        """nGPT step fused into the prefill output / down GEMM epilogues
        (default, when d is a multiple of 256 with d / 256 <= 8) or a
        separate row kernel."""
        _check("dory_set_fused_ngpt", lib().dory_set_fused_ngpt(self.handle, 1 if enable else 0))

    def launch_count(self):
        v = ctypes.c_int()
        _check("dory_last_launch_count", lib().dory_last_launch_count(self.handle, ctypes.byref(v)))
        return v.value

    def profile_begin(self, max_launches=65536):
        _check("dory_profile_begin", lib().dory_profile_begin(self.handle, max_launches))

    def profile_end(self):
        """{kernel class: (total ms, launches)} for the launches since
        profile_begin."""
        n = len(KERNEL_CLASSES)
        ms = (ctypes.c_double * n)()
        cnt = (ctypes.c_int * n)()
        _check("dory_profile_end", lib().dory_profile_end(self.handle, ms, cnt))
        return {KERNEL_CLASSES[i]: (ms[i], cnt[i]) for i in range(n)}

    def close(self):
        if getattr(self, "handle", None):
            lib().dory_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def set_debug_tc_attention(enable: bool):
    """dory_debug_attention: tensor-core prefill kernel where it applies
    (default) or always the mma.sync kernel."""
    _check("dory_set_tc_attention", lib().dory_set_tc_attention(None, 1 if enable else 0))


def debug_gemm(A, B, C=None, stream=None):
    """C = A @ B^T through the library's tensor-core GEMM (A [M,K], B [N,K]
    bf16 device tensors; C fp32 [M, N])."""
    import torch
    M, K = A.shape
    N = B.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _check("dory_debug_gemm", lib().dory_debug_gemm(_ptr(A), _ptr(B), _ptr(C), M, N, K,
                                                    C.stride(0), _stream_ptr(stream)))
    return C


def debug_attention(q, k_cur, v_cur, k_cache, v_cache, gate, out, B, C, P0, S, n_q, n_kv,
                    head_dim, window, scale=0.0, stream=None):
    """The library's attention step alone (all tensors bf16 on the device);
    one-token calls run the split-key decode kernels on a torch scratch buffer."""
    import torch
    if C == 1:
        nbytes = int(lib().dory_debug_attention_scratch_bytes(B, n_q, head_dim))
    else:                               # room for 64 key-range splits
        nbytes = 64 * (B * C * n_q * (head_dim + 2) * 4 + 512)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=out.device)
    _check("dory_debug_attention", lib().dory_debug_attention(
        _ptr(q), _ptr(k_cur), _ptr(v_cur), _ptr(k_cache), _ptr(v_cache), _ptr(gate), _ptr(out),
        B, C, P0, S, n_q, n_kv, head_dim, window, scale, _ptr(scratch), nbytes,
        _stream_ptr(stream)))
    return out
