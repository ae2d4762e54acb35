"""The allocation-free decode attention entry point.

Some callers cannot give the library any scratch memory: a plug-in inside a
host program that owns all device allocations and offers its extensions no
allocator or workspace, or a serving loop that forbids cudaMalloc after
start-up because it can block and synchronise the device.
dory_decode_attention_noalloc serves them with partial results kept in a
fixed array inside the library.  These tests call it through the C ABI and
compare it with the entry point that takes caller scratch, twice in a row, so
results left in the shared array by one call cannot leak into the next, and
with the CPU oracle's attention (the masked softmax of "Dory1.0-4B: A Looped
Normalized-GPT", Architecture and Last-Loop KV Caching) on small GQA and
sliding-window shapes.

This file is named so that pytest collects it after every other test file."""
import ctypes
import math

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_ok):
    import looped_normalized_transformer_ngpt_b300 as dory
    from looped_normalized_transformer_ngpt_b300 import _build
    _build.build()
    dory.lib()
    return dory


def _inputs(B, P0, W, nq, nkv, dh, seed):
    import torch
    g = torch.Generator(device="cuda").manual_seed(seed)
    L = P0 + 1
    S = L if W <= 0 else min(W, L)
    rnd = lambda *s: torch.randn(*s, device="cuda", generator=g)
    unit = lambda t: (t / t.norm(dim=-1, keepdim=True)).to(torch.bfloat16).contiguous()
    return dict(
        q=unit(rnd(B, nq, dh)), k_cur=unit(rnd(B, nkv, dh)),
        v_cur=(0.3 * rnd(B, nkv, dh)).to(torch.bfloat16),
        k_cache=unit(rnd(B, nkv, S, dh)), v_cache=(0.3 * rnd(B, nkv, S, dh)).to(torch.bfloat16),
        gate=torch.sigmoid(rnd(B, nq * dh)).to(torch.bfloat16), S=S)


def _noalloc(dev, x, out, B, P0, W, nq, nkv, dh):
    import torch
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = dev.lib().dory_decode_attention_noalloc(
        p(x["q"]), p(x["k_cur"]), p(x["v_cur"]), p(x["k_cache"]), p(x["v_cache"]), p(x["gate"]),
        p(out), B, P0, x["S"], nq, nkv, dh, W, 0.0,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc


@pytest.mark.parametrize("B,P0,W,nq,nkv,dh", [(4, 2055, 0, 8, 2, 128), (4, 2055, 512, 8, 2, 128),
                                              (2, 70, 16, 4, 2, 32)])
def test_noalloc_matches_scratch_entry_point_twice(dev, B, P0, W, nq, nkv, dh):
    import torch
    for call in range(2):
        # the second call uses other inputs and, for the long case, fewer keys
        p0 = P0 if call == 0 else max(1, P0 // 3)
        x = _inputs(B, p0, W, nq, nkv, dh, seed=100 * call + dh)
        ref = torch.zeros((B, nq * dh), dtype=torch.bfloat16, device="cuda")
        dev.debug_attention(x["q"], x["k_cur"], x["v_cur"], x["k_cache"], x["v_cache"], x["gate"],
                            ref, B, 1, p0, x["S"], nq, nkv, dh, W)
        out = torch.full((B, nq * dh), 7.0, dtype=torch.bfloat16, device="cuda")
        assert _noalloc(dev, x, out, B, p0, W, nq, nkv, dh) == dev.DORY_OK
        torch.cuda.synchronize()
        np.testing.assert_allclose(out.float().cpu().numpy(), ref.float().cpu().numpy(),
                                   atol=2e-2, rtol=2e-2)


def _oracle_attention(x, B, P0, W, nq, nkv, dh):
    """The oracle's masked softmax over the keys the ring holds plus the new
    token's own key, times the gate; float64 on the same bf16 inputs."""
    f = lambda t: t.float().cpu().numpy().astype(np.float64)
    q, kc, vc, kcur, vcur, gate = (f(x[n]) for n in ("q", "k_cache", "v_cache", "k_cur", "v_cur",
                                                     "gate"))
    S, G = x["S"], nq // nkv
    lo = 0 if W <= 0 else max(0, P0 - W + 1)
    pos = np.arange(lo, P0 + 1)
    want = np.zeros((B, nq, dh))
    for b in range(B):
        for h in range(nq):
            g = h // G
            keys = np.concatenate([kc[b, g, pos[:-1] % S], kcur[b, g][None]])
            vals = np.concatenate([vc[b, g, pos[:-1] % S], vcur[b, g][None]])
            want[b, h] = oracle.attention(q[b, h][None], keys, vals, np.array([P0]), pos,
                                          W if W > 0 else 1, W <= 0, math.sqrt(dh))[0]
    return want.reshape(B, nq * dh) * gate


@pytest.mark.parametrize("B,P0,W,nq,nkv,dh", [(2, 300, 0, 8, 2, 128), (3, 200, 64, 4, 1, 64),
                                              (2, 70, 16, 4, 2, 32), (1, 0, 0, 8, 2, 128)])
def test_noalloc_matches_oracle(dev, B, P0, W, nq, nkv, dh):
    """Error per (sequence, head) row relative to that row's norm: the outputs
    are O(0.3 / sqrt(visible keys)), so a plain absolute tolerance of the
    bf16 scale would not see a wrong key set."""
    import torch
    x = _inputs(B, P0, W, nq, nkv, dh, seed=7 + dh)
    out = torch.full((B, nq * dh), 7.0, dtype=torch.bfloat16, device="cuda")
    assert _noalloc(dev, x, out, B, P0, W, nq, nkv, dh) == dev.DORY_OK
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().reshape(B, nq, dh)
    want = _oracle_attention(x, B, P0, W, nq, nkv, dh).reshape(B, nq, dh)
    rel = np.linalg.norm(got - want, axis=-1) / np.linalg.norm(want, axis=-1)
    assert rel.max() < 1e-2, rel.max()


def test_noalloc_refuses_sizes_beyond_its_array(dev):
    import torch
    x = _inputs(1, 4, 0, 8, 2, 128, seed=1)
    out = torch.empty((1, 8 * 128), dtype=torch.bfloat16, device="cuda")
    # B * n_q = 256 * 8 partial rows of 128 splits need more than 16 MiB
    assert _noalloc(dev, x, out, 256, 4, 0, 8, 2, 128) == dev.DORY_ECAPACITY
    assert _noalloc(dev, x, out, 1, 4, 0, 8, 3, 128) == dev.DORY_EINVAL


def test_noalloc_refuses_misaligned_pointers_and_short_rings(dev):
    """Both refusals happen on the host before any launch."""
    import torch
    p = lambda t, off=0: ctypes.c_void_p(t.data_ptr() + off)
    lib = dev.lib()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    B, P0, nq, nkv, dh = 1, 40, 8, 2, 128
    x = _inputs(B, P0, 0, nq, nkv, dh, seed=3)
    out = torch.empty((B, nq * dh), dtype=torch.bfloat16, device="cuda")
    args = [p(x[n]) for n in ("q", "k_cur", "v_cur", "k_cache", "v_cache", "gate")] + [p(out)]
    for i in (1, 2, 3, 4):              # k_cur, v_cur, k_cache, v_cache off by 8 bytes
        bad = list(args)
        bad[i] = ctypes.c_void_p(args[i].value + 8)
        assert lib.dory_decode_attention_noalloc(*bad, B, P0, x["S"], nq, nkv, dh, 0, 0.0,
                                                 st) == dev.DORY_EINVAL
    # a ring shorter than the keys the mask shows
    assert lib.dory_decode_attention_noalloc(*args, B, P0, P0 - 1, nq, nkv, dh, 0, 0.0,
                                             st) == dev.DORY_EINVAL
    assert lib.dory_decode_attention_noalloc(*args, B, P0, 15, nq, nkv, dh, 17, 0.0,
                                             st) == dev.DORY_EINVAL
    assert lib.dory_decode_attention_noalloc(*args, B, P0, 16, nq, nkv, dh, 17, 0.0,
                                             st) == dev.DORY_OK
    torch.cuda.synchronize()
