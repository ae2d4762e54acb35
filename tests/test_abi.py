"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/dory.h declares, and its host-only functions (size queries,
validation, state errors) behave as documented.  No call here reaches CUDA."""
import ctypes
import os
import re

import pytest

import oracle
import synth
import looped_normalized_transformer_ngpt_b300 as dory
from looped_normalized_transformer_ngpt_b300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    _build.build()
    return dory.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "dory.h")).read()
    return sorted(set(re.findall(r"DORY_API\s+[\w\s\*]+?\b(dory_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("dory_create", "dory_bind", "dory_prefill", "dory_decode_step", "dory_kv_bytes",
              "dory_workspace_bytes", "dory_destroy", "dory_strerror"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for name in _declared():
        assert hasattr(L, name), name
        assert name in dory._SIGS, name


@pytest.mark.parametrize("shape", [synth.TINY, synth.TINY_LOOPFULL, synth.SMALL, synth.DORY4B])
@pytest.mark.parametrize("mode", [oracle.LAST_LOOP, oracle.PER_LOOP])
def test_kv_bytes_matches_oracle(L, shape, mode):
    cfg = dory.config_from_shape(shape)
    for mb, ctx, k in ((1, 1, 1), (2, 72, 4), (4, 5000, 3), (64, 32768, 2), (1, 262144, 4)):
        assert dory.kv_bytes(cfg, mb, ctx, k, mode) == oracle.kv_bytes(shape, mb, ctx, k, mode)


def test_kv_bytes_published_figure(L):
    cfg = dory.config_from_shape(synth.DORY4B)
    last = dory.kv_bytes(cfg, 1, 262144, 4, dory.LAST_LOOP)
    assert last == 9_663_676_416 + 54 * 4096 * 2048
    assert all(dory.kv_bytes(cfg, 1, 262144, k, dory.LAST_LOOP) == last for k in (1, 2, 3))


def test_size_queries_reject_bad_args(L):
    cfg = dory.config_from_shape(synth.TINY)
    assert dory.kv_bytes(cfg, 0, 10, 1, 0) == 0
    assert dory.kv_bytes(cfg, 1, 10, 0, 0) == 0
    assert dory.kv_bytes(cfg, 1, 10, 1, 7) == 0
    assert dory.workspace_bytes(cfg, 1, 0) == 0
    assert dory.workspace_bytes(cfg, 2, 64) > 0
    bad = dory.config_from_shape(synth.TINY.replace(head_dim=48))
    assert dory.kv_bytes(bad, 1, 10, 1, 0) == 0


def _fake_weights(shape):
    n = shape.n_layers
    layers = (dory.DoryLayerWeights * n)()
    for l in range(n):
        layers[l] = dory.DoryLayerWeights(*([0x1000 * (l + 1)] * 7))
    return dory.DoryWeights(0x100, 0x200, 0, layers), layers


def test_create_validates_config(L):
    w, keep = _fake_weights(synth.TINY)
    h = ctypes.c_void_p()
    for bad, code in ((synth.TINY.replace(head_dim=48), dory.DORY_EUNSUPPORTED),
                      (synth.TINY.replace(n_kv=3), dory.DORY_EINVAL),
                      (synth.TINY.replace(d=100), dory.DORY_EUNSUPPORTED),
                      (synth.TINY.replace(ffn=200), dory.DORY_EUNSUPPORTED),
                      (synth.TINY.replace(window=0), dory.DORY_EINVAL)):
        cfg = dory.config_from_shape(bad)
        assert L.dory_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == code
    cfg = dory.config_from_shape(synth.TINY)
    assert L.dory_create(ctypes.byref(cfg), None, ctypes.byref(h)) == dory.DORY_EINVAL
    keep[1] = dory.DoryLayerWeights(0, 1, 1, 1, 1, 1, 1)
    assert L.dory_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == dory.DORY_EINVAL


def test_state_errors_before_any_launch(L):
    shape = synth.TINY
    w, keep = _fake_weights(shape)
    cfg = dory.config_from_shape(shape)
    h = ctypes.c_void_p()
    assert L.dory_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == dory.DORY_OK
    try:
        assert L.dory_prefill(h, ctypes.c_void_p(0x10), 1, 4, 1, 0, None, 0, None) == dory.DORY_EUNBOUND
        assert L.dory_decode_step(h, ctypes.c_void_p(0x10), 1, 1, 0, None, None, None) == dory.DORY_EUNBOUND
        n = ctypes.c_int(-1)
        assert L.dory_length(h, ctypes.byref(n)) == dory.DORY_OK and n.value == 0
        kvb = dory.kv_bytes(cfg, 2, 72, 1, 0)
        wsb = dory.workspace_bytes(cfg, 2, 64)
        # misaligned and undersized buffers are rejected before any CUDA call
        assert L.dory_bind(h, ctypes.c_void_p(0x1008), kvb, ctypes.c_void_p(0x2000), wsb,
                           2, 72, 64, 1, 0) == dory.DORY_EINVAL
        assert L.dory_bind(h, ctypes.c_void_p(0x1000), kvb - 1, ctypes.c_void_p(0x2000), wsb,
                           2, 72, 64, 1, 0) == dory.DORY_ENOMEM
        assert L.dory_bind(h, ctypes.c_void_p(0x1000), kvb, ctypes.c_void_p(0x2000), wsb - 1,
                           2, 72, 64, 1, 0) == dory.DORY_ENOMEM
        assert L.dory_bind(h, ctypes.c_void_p(0x1000), kvb, ctypes.c_void_p(0x2000), wsb,
                           2, 72, 64, 1, 5) == dory.DORY_EINVAL
        off, slots = ctypes.c_size_t(), ctypes.c_int()
        assert L.dory_debug_kv_offset(h, 0, 0, 0, ctypes.byref(off), ctypes.byref(slots)) == dory.DORY_EUNBOUND
    finally:
        assert L.dory_destroy(h) == dory.DORY_OK


def test_strerror(L):
    for code in range(0, -9, -1):
        s = dory.strerror(code)
        assert s and s != "unknown status"
    assert dory.strerror(-99) == "unknown status"


def test_debug_gemm_rejects_bad_shapes(L):
    assert L.dory_debug_gemm(None, None, None, 1, 1, 8, 1, None) == dory.DORY_EINVAL
    assert L.dory_debug_gemm(ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                             4, 4, 12, 4, None) == dory.DORY_EINVAL


def test_bench_visible_key_count_matches_brute_force():
    """bench.py's algorithmic work model: the closed-form count of visible
    (query, key) pairs equals direct counting."""
    import bench
    import synth
    for sh in (synth.SMALL, synth.TINY):
        for l in range(4):
            for P0, C in ((0, 2048), (300, 700), (1000, 5), (0, 1), (511, 2), (512, 1), (15, 40)):
                brute = sum(t + 1 if sh.is_full(l) else min(t + 1, sh.window)
                            for t in range(P0, P0 + C))
                assert bench.visible_keys(sh, l, P0, C) == brute


def test_path_switches_validate_arguments(L):
    """The comparison switches are host state: argument errors come back
    without any CUDA call, on a created (unbound) handle."""
    shape = synth.TINY
    w, keep = _fake_weights(shape)
    cfg = dory.config_from_shape(shape)
    h = ctypes.c_void_p()
    assert L.dory_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h)) == dory.DORY_OK
    try:
        assert L.dory_set_fused_ngpt(None, 1) == dory.DORY_EINVAL
        assert L.dory_set_fused_ngpt(h, 2) == dory.DORY_EINVAL
        assert L.dory_set_fused_ngpt(h, 0) == dory.DORY_OK
        assert L.dory_set_fused_ngpt(h, 1) == dory.DORY_OK
        assert L.dory_set_tc_attention(h, 3) == dory.DORY_EINVAL
        assert L.dory_set_tc_attention(h, 0) == dory.DORY_OK
        assert L.dory_set_quantized_swap(None, 1) == dory.DORY_EINVAL
        assert L.dory_set_quantized_swap(h, 2) == dory.DORY_EINVAL
        assert L.dory_set_quantized_swap(h, 1) == dory.DORY_OK
        assert L.dory_set_quantized_swap(h, 0) == dory.DORY_OK
    finally:
        assert L.dory_destroy(h) == dory.DORY_OK


def test_bench_work_models_match_the_closed_forms():
    """bench.py's algorithmic work per step (the numerators of every
    roofline fraction) against the closed-form figures of the workloads:
    prefill FLOP per token (layer applications 32 + 40k at 2 x parameters,
    attention over visible pairs, the LM head on one row per sequence) and
    decode bytes per step (every weight once, the LM head, the visible
    cached K/V)."""
    import bench
    import synth

    def close(a, b, rel=5e-3):
        return abs(a - b) <= rel * b

    for sh, B, C, want in ((synth.DORY4B, 1, 8192, (9.51, 14.80, 25.37)),
                           (synth.SMALL, 4, 2048, (0.486, 0.756, 1.295))):
        for k, w in zip((1, 2, 4), want):
            f = bench.step_flops(sh, B, C, k)
            assert close(sum(f.values()) / (B * C) / 1e9, w), (sh.name, k)
    for k, w in zip((1, 2, 3, 4), (114.4, 177.6, 240.9, 304.1)):
        d = bench.decode_step_bytes(synth.DORY4B, 64, k, 32768)
        assert close((d["weights"] + d["kv"]) / 1e9, w), k
    for k, w in ((1, 18.2), (4, 47.6)):
        d = bench.decode_step_bytes(synth.DORY4B, 1, k, 262144)
        assert close((d["weights"] + d["kv"]) / 1e9, w), k
    # the per-class split the roofline uses adds up to the same bytes
    for B, k, P0 in ((64, 1, 32768), (64, 4, 32775), (1, 3, 100), (4, 2, 5000)):
        d = bench.decode_step_bytes(synth.DORY4B, B, k, P0)
        c = bench.decode_class_bytes(synth.DORY4B, B, k, P0)
        assert sum(c.values()) == d["weights"] + d["kv"] and c["attention"] == d["kv"]
    assert [bench.layer_apps(synth.DORY4B, k).count(20) for k in (1, 2, 4)] == [1, 2, 4]
    assert len(bench.layer_apps(synth.DORY4B, 4)) == 192
