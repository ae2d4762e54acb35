"""Ragged batches through the C ABI: sequences of different lengths prefilled
slot by slot (dory_prefill_slot) and decoded together at their own
positions (dory_decode_step_ragged).  Every sequence must compute exactly
what it computes alone, so each is compared with its own oracle run
(prompt + decode steps, one sequence), in both cache modes, with window
rings that wrap, on the tiny shape (cp.async decode attention) and at the
4B-class width (TMA decode attention, ring sizes of 64-multiples).  Equal
lengths through the ragged path must give the uniform path's results bit
for bit.  Tolerances as in test_gpu_parity."""
import numpy as np
import pytest

import oracle
import synth
from test_gpu_parity import check_greedy, check_hidden, check_logits, _tok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev(cuda_ok):
    import looped_normalized_transformer_ngpt_b300 as dory
    from looped_normalized_transformer_ngpt_b300 import _build
    _build.build()
    dory.lib()
    return dory


def _run(dev, shape, w, lens, mode, k, steps, max_ctx, extend=None, seed=0, ks=None):
    """ks: one loop count per sequence (last-loop cache), else k for all."""
    B = len(lens)
    ks = list(ks) if ks is not None else [k] * B
    dt = np.float64 if shape.d <= 256 else np.float32
    m = dev.Model(shape, w, max_batch=B + 1, max_ctx=max_ctx, max_chunk=max(lens),
                  k_max=max(ks), cache_mode=mode)
    oracles, nxt = [], []
    for b, T in enumerate(lens):
        prompt = synth.tokens(shape, 1, T, seed=seed + b)
        o = oracle.Oracle(shape, w, dtype=dt)
        z = o.prefill(prompt, ks[b], mode)["logits"][0, -1]
        lg = m.prefill_slot(b, _tok(prompt[0]), ks[b], mode).cpu().numpy()
        check_logits(lg, z)
        oracles.append(o)
        nxt.append(int(np.argmax(z)))
    assert m.lengths(B) == list(lens)
    cur = np.array(nxt, np.int32)
    for s in range(steps):
        if extend is not None and s == extend[0]:
            # continuous batching: one slot takes more prompt tokens mid-stream
            b, n = extend[1], extend[2]
            more = synth.tokens(shape, 1, n, seed=seed + 100)
            z = oracles[b].prefill(more, ks[b], mode)["logits"][0, -1]
            lg = m.prefill_slot(b, _tok(more[0]), ks[b], mode).cpu().numpy()
            check_logits(lg, z)
            cur[b] = int(np.argmax(z))
        if len(set(ks)) == 1:
            lg, g = m.decode_ragged(_tok(cur), k, mode)
        else:
            lg, g = m.decode_multi(_tok(cur), ks, mode)
        lg, g, hid = lg.cpu().numpy(), g.cpu().numpy(), m.hidden(B).cpu().numpy()
        for b, o in enumerate(oracles):
            r = o.decode(cur[b:b + 1], ks[b], mode)
            check_logits(lg[b:b + 1], r["logits"])
            check_hidden(hid[b:b + 1], r["hidden"])
            check_greedy(g[b:b + 1], r["logits"])
        cur = np.array([int(np.argmax(o_lg)) for o_lg in lg], np.int32)
    assert m.lengths(B) == [o.length for o in oracles]
    assert m.device_status() == 0
    m.close()


@pytest.mark.parametrize("mode", [oracle.LAST_LOOP, oracle.PER_LOOP], ids=["last", "perloop"])
@pytest.mark.parametrize("k", [1, 2])
def test_ragged_tiny(dev, mode, k):
    shape = synth.TINY_LOOPFULL                      # window 16: the rings wrap
    _run(dev, shape, synth.make_weights(shape), [5, 23, 12], mode, k, steps=4, max_ctx=64,
         extend=(2, 0, 7), seed=10 * k + mode)


@pytest.mark.parametrize("mode", [oracle.LAST_LOOP, oracle.PER_LOOP], ids=["last", "perloop"])
def test_ragged_4b_width_windowed(dev, mode):
    """4B-class width with a 128-position window so that the window rings
    (128 slots) wrap for the longer sequences and not for the shorter."""
    shape = synth.DORY4B_SLIM.replace(window=128)
    _run(dev, shape, synth.make_weights(shape), [70, 200, 131], mode, 2, steps=3, max_ctx=384,
         extend=(1, 2, 9), seed=30 + mode)


def test_per_sequence_loop_counts_tiny(dev):
    """Each sequence at its own loop count in one decode step (last-loop
    cache): as the same sequence decoded alone at that count."""
    shape = synth.TINY_LOOPFULL
    _run(dev, shape, synth.make_weights(shape), [5, 23, 12, 9], oracle.LAST_LOOP, 0, steps=4,
         max_ctx=64, extend=(2, 1, 6), seed=77, ks=[1, 3, 2, 4])


def test_per_sequence_loop_counts_4b_width(dev):
    shape = synth.DORY4B_SLIM.replace(window=128)
    _run(dev, shape, synth.make_weights(shape), [70, 200, 131], oracle.LAST_LOOP, 0, steps=3,
         max_ctx=384, seed=88, ks=[2, 4, 1])


def test_equal_loop_counts_match_ragged_bitwise(dev):
    import torch
    shape = synth.DORY4B_SLIM
    w = synth.make_weights(shape)
    B, k = 3, 2
    ms = [dev.Model(shape, w, max_batch=B, max_ctx=192, max_chunk=64, k_max=k) for _ in range(2)]
    for m in ms:
        for b, T in enumerate([20, 64, 41]):
            m.prefill_slot(b, _tok(synth.tokens(shape, 1, T, seed=b)[0]), k)
    tok = _tok(np.array([3, 1000, 77], np.int32))
    for _ in range(2):
        la, ga = ms[0].decode_ragged(tok, k)
        lb, gb = ms[1].decode_multi(tok, [k] * B)
        assert torch.equal(la, lb) and torch.equal(ga, gb)
        tok = ga
    for m in ms:
        m.close()


def test_ragged_equal_lengths_match_uniform_bitwise(dev):
    import torch
    shape = synth.DORY4B_SLIM
    w = synth.make_weights(shape)
    B, T, k = 3, 70, 2
    prompt = synth.tokens(shape, B, T, seed=5)
    a = dev.Model(shape, w, max_batch=B, max_ctx=128, max_chunk=T, k_max=k)
    b = dev.Model(shape, w, max_batch=B, max_ctx=128, max_chunk=T, k_max=k)
    a.prefill(_tok(prompt), k)
    b.prefill(_tok(prompt), k)
    tok = _tok(np.array([3, 1000, 77], np.int32))
    for _ in range(3):
        la, ga = a.decode(tok, k)
        lb, gb = b.decode_ragged(tok, k)
        assert torch.equal(la, lb) and torch.equal(ga, gb)
        tok = ga
    assert b.lengths(B) == [T + 3] * B
    a.close()
    b.close()


def test_ragged_refusals(dev):
    shape = synth.TINY
    m = dev.Model(shape, synth.make_weights(shape), max_batch=2, max_ctx=16, max_chunk=8)
    L = dev.lib()
    m.prefill_slot(1, _tok(synth.tokens(shape, 1, 4)[0]), 1)
    assert m.lengths(2) == [0, 4]
    with pytest.raises(dev.DoryError):                 # uniform calls in the ragged state
        m.decode(_tok(np.array([1, 2], np.int32)), 1)
    with pytest.raises(dev.DoryError):
        m.prefill(_tok(synth.tokens(shape, 2, 3)), 1)
    with pytest.raises(dev.DoryError):                 # slot out of range
        m.prefill_slot(2, _tok(np.array([1], np.int32)), 1)
    with pytest.raises(dev.DoryError) as e:            # too long for the ring capacity
        m.prefill_slot(1, _tok(synth.tokens(shape, 1, 13)[0]), 1)
    assert e.value.code == dev.DORY_ECAPACITY
    with pytest.raises(dev.DoryError):
        m.set_lengths([3, 17])
    with pytest.raises(dev.DoryError):                 # a loop count below 1
        m.decode_multi(_tok(np.array([1, 2], np.int32)), [1, 0])
    assert m.lengths(2) == [0, 4]
    m.set_length(2, 0)                                  # back to one shared length
    m.prefill(_tok(synth.tokens(shape, 2, 3)), 1)
    assert m.lengths(2) == [3, 3]
    m.close()


def _run_mixed(dev, shape, w, lens, chunks, mode, k, max_ctx, seed):
    """Slots 0 .. B-1 hold prompts of `lens`; slot B receives a new prompt
    whose first chunk is prefilled alone and whose later chunks ride along
    with one decode token of every other slot (dory_step_mixed).  Every row
    against its own sequence's oracle; then one ragged decode of all slots."""
    B = len(lens)
    dt = np.float64 if shape.d <= 256 else np.float32
    m = dev.Model(shape, w, max_batch=B + 1, max_ctx=max_ctx,
                  max_chunk=max(max(lens), max(chunks)), k_max=k, cache_mode=mode)
    oracles, cur = [], []
    for b, T in enumerate(lens):
        prompt = synth.tokens(shape, 1, T, seed=seed + b)
        o = oracle.Oracle(shape, w, dtype=dt)
        z = o.prefill(prompt, k, mode)["logits"][0, -1]
        check_logits(m.prefill_slot(b, _tok(prompt[0]), k, mode).cpu().numpy(), z)
        oracles.append(o)
        cur.append(int(np.argmax(z)))
    oc = oracle.Oracle(shape, w, dtype=dt)
    new = synth.tokens(shape, 1, sum(chunks), seed=seed + 50)[0]
    t0 = chunks[0]
    zc = oc.prefill(new[None, :t0], k, mode)["logits"][0, -1]
    check_logits(m.prefill_slot(B, _tok(new[:t0]), k, mode).cpu().numpy(), zc)
    for C in chunks[1:]:
        lg, g = m.step_mixed(_tok(np.array(cur, np.int32)), B, _tok(new[t0:t0 + C]), k, mode)
        lg, g = lg.cpu().numpy(), g.cpu().numpy()
        for b, o in enumerate(oracles):
            r = o.decode(np.array([cur[b]], np.int32), k, mode)
            check_logits(lg[b:b + 1], r["logits"])
            check_greedy(g[b:b + 1], r["logits"])
        r = oc.prefill(new[None, t0:t0 + C], k, mode)
        check_logits(lg[B:B + 1], r["logits"][:, -1])
        cur = [int(x) for x in np.argmax(lg[:B], axis=-1)]
        t0 += C
    # a step with no decode rows, then every slot decodes together
    lg, g = m.step_mixed(_tok(np.zeros(0, np.int32)), B, _tok(new[:3]), k, mode)
    r = oc.prefill(new[None, :3], k, mode)
    check_logits(lg.cpu().numpy()[0:1], r["logits"][:, -1])
    assert g is None
    allc = np.array(cur + [int(np.argmax(r["logits"][0, -1]))], np.int32)
    lg, _ = m.decode_ragged(_tok(allc), k, mode)
    for b, o in enumerate(oracles + [oc]):
        check_logits(lg.cpu().numpy()[b:b + 1], o.decode(allc[b:b + 1], k, mode)["logits"])
    assert m.lengths(B + 1) == [o.length for o in oracles + [oc]]
    assert m.device_status() == 0
    m.close()


@pytest.mark.parametrize("mode", [oracle.LAST_LOOP, oracle.PER_LOOP], ids=["last", "perloop"])
def test_mixed_steps_tiny(dev, mode):
    shape = synth.TINY_LOOPFULL                      # window 16: the rings wrap
    _run_mixed(dev, shape, synth.make_weights(shape), [5, 23, 12], [7, 4, 19, 1], mode, 2,
               max_ctx=96, seed=5)


@pytest.mark.parametrize("mode", [oracle.LAST_LOOP, oracle.PER_LOOP], ids=["last", "perloop"])
def test_mixed_steps_4b_width(dev, mode):
    """Chunks of 5 (8 rows: the GEMV path) and 40 / 64 (43 and 67 rows: the
    tensor-core GEMMs) after decode rows of three slots, window 128."""
    shape = synth.DORY4B_SLIM.replace(window=128)
    _run_mixed(dev, shape, synth.make_weights(shape), [70, 150, 131], [100, 5, 40, 64], mode, 2,
               max_ctx=384, seed=9)


@pytest.mark.parametrize("mode", [oracle.LAST_LOOP, oracle.PER_LOOP], ids=["last", "perloop"])
def test_ragged_batched_path_tiny(dev, mode):
    """20 sequences (more rows than the few-row projections take: the
    swapped tensor-core GEMMs), ragged lengths, one slot extended
    mid-stream."""
    shape = synth.TINY_LOOPFULL
    lens = [3 + 2 * b for b in range(20)]
    _run(dev, shape, synth.make_weights(shape), lens, mode, 2, steps=3, max_ctx=64,
         extend=(1, 7, 5), seed=200 + mode)


def test_per_sequence_loop_counts_batched_path_tiny(dev):
    shape = synth.TINY_LOOPFULL
    lens = [4 + 3 * b for b in range(18)]
    _run(dev, shape, synth.make_weights(shape), lens, oracle.LAST_LOOP, 0, steps=3, max_ctx=80,
         seed=300, ks=[1 + b % 4 for b in range(18)])


def test_ragged_batched_path_4b_width(dev):
    """18 sequences at the 4B-class width through the swapped GEMMs and the
    TMA decode attention at ragged positions (window 128: some rings wrap)."""
    shape = synth.DORY4B_SLIM.replace(window=128)
    lens = [10 + 11 * b for b in range(18)]
    _run(dev, shape, synth.make_weights(shape), lens, oracle.LAST_LOOP, 2, steps=2, max_ctx=256,
         seed=400)
