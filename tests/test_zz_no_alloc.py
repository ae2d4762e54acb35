"""The allocation-free decode attention entry point.

Some callers cannot give the library any scratch memory: a plug-in inside a
host program that owns all device allocations and offers its extensions no
allocator or workspace, or a serving loop that forbids cudaMalloc after
start-up because it can block and synchronise the device.
dory_decode_attention_noalloc serves them with partial results kept in a
fixed array inside the library.  These tests call it through the C ABI and
compare it with the entry point that takes caller scratch, twice in a row, so
results left in the shared array by one call cannot leak into the next.

This file is named so that pytest collects it after every other test file."""
import ctypes

import numpy as np
import pytest

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


def test_noalloc_refuses_sizes_beyond_its_array(dev):
    import torch
    x = _inputs(1, 4, 0, 8, 2, 128, seed=1)
    out = torch.empty((1, 8 * 128), dtype=torch.bfloat16, device="cuda")
    # B * n_q = 256 * 8 partial rows of 128 splits need more than 16 MiB
    assert _noalloc(dev, x, out, 256, 4, 0, 8, 2, 128) == dev.DORY_ECAPACITY
    assert _noalloc(dev, x, out, 1, 4, 0, 8, 3, 128) == dev.DORY_EINVAL
