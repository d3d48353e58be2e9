"""Greedy decode with the argmax fused into the LM head and the next token fed
back on the device (mk_decode_greedy): the same tokens, logits and caches as
a host loop of mk_decode_step + argmax, and the oracle's greedy tokens."""
import numpy as np
import pytest
import torch

from decode_megakernel_03_gb300 import mk, synth

from tests.parity_util import Pair, bf16_bits, compare_logits

pytestmark = pytest.mark.gpu


def _host_loop(pair, tok, pos, n):
    """n steps of mk_decode_step, each next token the fp32 argmax on the host
    (numpy's first index among equal logits)."""
    toks = []
    cur = list(tok)
    for s in range(n):
        logits = pair.gpu_step(cur, [p + s for p in pos])
        cur = [int(np.argmax(logits[b].astype(np.float32))) for b in range(pair.batch)]
        toks.append(cur)
    return np.array(toks, np.int32), logits


def _device_loop(pair, tok, pos, n):
    out = torch.zeros(n * pair.batch, dtype=torch.int32, device="cuda")
    pair.dec.decode_greedy(tok, pos, n, out, pair.logits)
    assert pair.dec.status() == mk.MK_OK, pair.dec.last_error()
    return out.cpu().numpy().reshape(n, pair.batch), pair.logits.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("name,batch,n", [("tiny", 1, 12), ("tiny", 4, 8), ("llama1b", 1, 4)])
def test_greedy_equals_host_argmax_loop(name, batch, n):
    wl = synth.WORKLOADS[name]
    cap = 256 if name == "tiny" else wl.capacity
    ctx = tuple(40 + 23 * b for b in range(batch)) if name == "tiny" else wl.ctx
    t0 = int(synth.step_tokens(wl)[0][0])
    tok = [(t0 + 17 * b) % wl.shape.vocab for b in range(batch)]
    pos = list(ctx)
    a = Pair(wl.shape, batch, cap, ctx=ctx)
    want_tok, want_logits = _host_loop(a, tok, pos, n)
    caches_a = [bf16_bits(t) for t in a.kc + a.vc]
    a.close()
    b = Pair(wl.shape, batch, cap, ctx=ctx)
    got_tok, got_logits = _device_loop(b, tok, pos, n)
    caches_b = [bf16_bits(t) for t in b.kc + b.vc]
    b.close()
    np.testing.assert_array_equal(got_tok, want_tok)
    np.testing.assert_array_equal(got_logits, want_logits)
    for x, y in zip(caches_a, caches_b):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("name,batch,n", [("tiny", 1, 12), ("tiny", 4, 8), ("llama1b", 1, 4),
                                          ("tiny", 2, mk.MAX_STEPS_PER_LAUNCH)])
def test_one_launch_greedy_equals_greedy(name, batch, n):
    """All steps in one persistent launch: the same tokens, final logits and
    caches as one launch per step."""
    wl = synth.WORKLOADS[name]
    cap = 256 if name == "tiny" else wl.capacity
    ctx = tuple(40 + 23 * b for b in range(batch)) if name == "tiny" else wl.ctx
    t0 = int(synth.step_tokens(wl)[0][0])
    tok = [(t0 + 17 * b) % wl.shape.vocab for b in range(batch)]
    a = Pair(wl.shape, batch, cap, ctx=ctx)
    want_tok, want_logits = _device_loop(a, tok, list(ctx), n)
    caches_a = [bf16_bits(t) for t in a.kc + a.vc]
    a.close()
    b = Pair(wl.shape, batch, cap, ctx=ctx)
    out = torch.zeros(n * batch, dtype=torch.int32, device="cuda")
    b.dec.decode_greedy_persistent(tok, list(ctx), n, out, b.logits)
    assert b.dec.status() == mk.MK_OK, b.dec.last_error()
    got_tok = out.cpu().numpy().reshape(n, batch)
    got_logits = b.logits.cpu().numpy().astype(np.float64)
    caches_b = [bf16_bits(t) for t in b.kc + b.vc]
    b.close()
    np.testing.assert_array_equal(got_tok, want_tok)
    np.testing.assert_array_equal(got_logits, want_logits)
    for x, y in zip(caches_a, caches_b):
        np.testing.assert_array_equal(x, y)


def test_greedy_at_its_maximum_step_count():
    """MAX_GREEDY_STEPS steps in one call, one sequence on the tiny shape:
    the tokens, final logits and caches of a host argmax loop."""
    wl = synth.WORKLOADS["tiny"]
    n = mk.MAX_GREEDY_STEPS
    ctx = (17,)
    cap = ctx[0] + n + 15
    a = Pair(wl.shape, 1, cap, ctx=ctx)
    want_tok, want_logits = _host_loop(a, [9], list(ctx), n)
    caches_a = [bf16_bits(t) for t in a.kc + a.vc]
    a.close()
    b = Pair(wl.shape, 1, cap, ctx=ctx)
    got_tok, got_logits = _device_loop(b, [9], list(ctx), n)
    caches_b = [bf16_bits(t) for t in b.kc + b.vc]
    b.close()
    np.testing.assert_array_equal(got_tok, want_tok)
    np.testing.assert_array_equal(got_logits, want_logits)
    for x, y in zip(caches_a, caches_b):
        np.testing.assert_array_equal(x, y)


def test_greedy_follows_the_oracle():
    """Tiny shape, two sequences: the device-fed tokens are the oracle's greedy
    tokens (compared until a step whose oracle top-1/top-2 margin is below
    1e-3, where either choice is right), and every step's logits meet the
    parity tolerances."""
    wl = synth.WORKLOADS["tiny"]
    batch, n, cap = 2, 10, 128
    ctx = (30, 51)
    tok = [5, 4000]
    pair = Pair(wl.shape, batch, cap, ctx=ctx)
    got_tok, got_logits = _device_loop(pair, tok, list(ctx), n)
    cur = list(tok)
    compared = 0
    for s in range(n):
        want = pair.oracle_step(cur, [c + s for c in ctx])
        w32 = want.astype(np.float32)
        srt = np.sort(w32, axis=1)
        if np.any(srt[:, -1] - srt[:, -2] < 1e-3):
            break  # a near tie: from here on either token is right
        nxt = [int(np.argmax(w32[b])) for b in range(batch)]
        np.testing.assert_array_equal(got_tok[s], nxt)
        cur = nxt
        compared += 1
    assert compared >= 3
    if compared == n:
        for st in compare_logits(got_logits, want):
            assert st["rel_l2"] <= 1e-2 and st["max_abs"] <= 5e-2 and st["top1"]
    pair.close()


def test_greedy_rejects_bad_arguments():
    wl = synth.WORKLOADS["tiny"]
    pair = Pair(wl.shape, 1, 128, ctx=(20,))
    out = torch.zeros(16, dtype=torch.int32, device="cuda")
    for n, pos in ((0, 20), (mk.MAX_GREEDY_STEPS + 1, 20), (10, 120)):
        with pytest.raises(mk.MkError) as e:
            pair.dec.decode_greedy([1], [pos], n, out, pair.logits)
        assert e.value.code == mk.MK_ERR_INVALID
    for n, pos in ((0, 20), (mk.MAX_STEPS_PER_LAUNCH + 1, 20), (10, 120)):
        with pytest.raises(mk.MkError) as e:
            pair.dec.decode_greedy_persistent([1], [pos], n, out, pair.logits)
        assert e.value.code == mk.MK_ERR_INVALID
    pair.close()
