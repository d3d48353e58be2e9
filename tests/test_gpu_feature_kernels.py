"""The paged-cache and greedy-decode kernels chosen by head shape: batch 8
with head_dim 64 and four query heads per kv-head, and batch 1 with
head_dim 128 and four query heads per kv-head, each on a small two-layer
model. A paged step gives the contiguous step's logits and k/v rows bit for
bit, greedy decode on the device gives a host argmax loop's tokens, logits
and caches, and the one-launch form gives the same again."""
import numpy as np
import pytest
import torch

from decode_megakernel_03_gb300 import mk, synth

from tests.parity_util import Pair, bf16_bits
from tests.test_gpu_greedy import _device_loop, _host_loop
from tests.test_gpu_paged import _cache_from, _pool_from

pytestmark = pytest.mark.gpu

G4_B8 = synth.ModelShape("g4", 2, 512, 8, 2, 64, 1024, 4096, tied=False, rope_theta=10000.0)
D128_G4 = synth.ModelShape("d128g4", 2, 512, 4, 1, 128, 1024, 4096, tied=True,
                           rope_theta=500000.0)
CASES = [(G4_B8, 8), (D128_G4, 1)]


def _ctx(batch):
    return tuple(33 + 29 * b for b in range(batch))  # ragged, none a multiple of 16


@pytest.mark.parametrize("shape,batch", CASES, ids=lambda c: getattr(c, "name", c))
def test_paged_matches_contiguous(shape, batch):
    bs, cap, steps = 16, 256, 3
    ctx = _ctx(batch)
    dev = torch.device("cuda")
    w = synth.make_weights(shape, seed=3, device=dev)
    kc, vc = synth.make_kv(shape, batch, cap, ctx, seed=4, device=dev)
    mb = cap // bs
    n_blocks = batch * mb + 5
    table = np.random.default_rng(9).permutation(n_blocks)[:batch * mb]
    table = table.reshape(batch, mb).astype(np.int32)
    kp = [_pool_from(t, table, n_blocks, bs) for t in kc]
    vp = [_pool_from(t, table, n_blocks, bs) for t in vc]
    dc = mk.Decoder(shape, w, kc, vc, batch)
    dp = mk.Decoder(shape, w, kp, vp, batch, paged=(bs, n_blocks, cap))
    lc = torch.empty((batch, shape.vocab), dtype=torch.float32, device=dev)
    lp = torch.empty_like(lc)
    for s in range(steps):
        tok = [(101 * s + 37 * b + 2) % shape.vocab for b in range(batch)]
        pos = [c + s for c in ctx]
        dc.step(tok, pos, lc)
        dp.step_paged(tok, pos, table, lp)
        assert dc.status() == mk.MK_OK and dp.status() == mk.MK_OK, dp.last_error()
        np.testing.assert_array_equal(lp.cpu().numpy(), lc.cpu().numpy())
    for l in range(shape.n_layers):
        assert torch.equal(_cache_from(kp[l], table, batch, cap, bs), kc[l])
        assert torch.equal(_cache_from(vp[l], table, batch, cap, bs), vc[l])
    dc.close()
    dp.close()


@pytest.mark.parametrize("shape,batch", CASES, ids=lambda c: getattr(c, "name", c))
def test_greedy_on_the_device(shape, batch):
    n, cap = 6, 256
    ctx = _ctx(batch)
    tok = [(7 + 113 * b) % shape.vocab for b in range(batch)]
    a = Pair(shape, batch, cap, ctx=ctx)
    want_tok, want_logits = _host_loop(a, tok, list(ctx), n)
    want_caches = [bf16_bits(t) for t in a.kc + a.vc]
    a.close()
    b = Pair(shape, batch, cap, ctx=ctx)
    got_tok, got_logits = _device_loop(b, tok, list(ctx), n)
    got_caches = [bf16_bits(t) for t in b.kc + b.vc]
    b.close()
    np.testing.assert_array_equal(got_tok, want_tok)
    np.testing.assert_array_equal(got_logits, want_logits)
    for x, y in zip(want_caches, got_caches):
        np.testing.assert_array_equal(x, y)
    c = Pair(shape, batch, cap, ctx=ctx)
    out = torch.zeros(n * batch, dtype=torch.int32, device="cuda")
    c.dec.decode_greedy_persistent(tok, list(ctx), n, out, c.logits)
    assert c.dec.status() == mk.MK_OK, c.dec.last_error()
    np.testing.assert_array_equal(out.cpu().numpy().reshape(n, batch), want_tok)
    np.testing.assert_array_equal(c.logits.cpu().numpy().astype(np.float64), want_logits)
    for x, y in zip(want_caches, [bf16_bits(t) for t in c.kc + c.vc]):
        np.testing.assert_array_equal(x, y)
    c.close()
