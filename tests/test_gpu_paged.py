"""Paged KV cache (mk_create_paged / mk_decode_step_paged): the same step on
the same cached keys, held in a shuffled block pool, gives bit-identical
logits and appends the same k/v rows as the contiguous cache."""
import numpy as np
import pytest
import torch

from decode_megakernel_03_gb300 import mk, synth

pytestmark = pytest.mark.gpu


def _pool_from(cache, table, n_blocks, bs):
    """[B][nkv][S][D] -> [n_blocks][nkv][bs][D] with block table[b][i] holding
    positions i*bs .. i*bs + bs - 1 of sequence b."""
    B, nkv, S, D = cache.shape
    pool = torch.zeros((n_blocks, nkv, bs, D), dtype=cache.dtype, device=cache.device)
    for b in range(B):
        for i in range(S // bs):
            pool[table[b, i]] = cache[b, :, i * bs:(i + 1) * bs, :]
    return pool


def _cache_from(pool, table, B, S, bs):
    nkv, D = pool.shape[1], pool.shape[3]
    out = torch.empty((B, nkv, S, D), dtype=pool.dtype, device=pool.device)
    for b in range(B):
        for i in range(S // bs):
            out[b, :, i * bs:(i + 1) * bs, :] = pool[table[b, i]]
    return out


# block sizes: one position per block (every key its own copy), sizes that do
# not divide a 64-key page (runs break inside pages), and whole pages
@pytest.mark.parametrize("name,batch,bs,steps", [("tiny", 2, 16, 4), ("llama1b", 1, 32, 3),
                                                 ("tiny", 2, 1, 3), ("tiny", 2, 5, 3),
                                                 ("tiny", 4, 48, 2)])
def test_paged_matches_contiguous(name, batch, bs, steps):
    wl = synth.WORKLOADS[name]
    shape = wl.shape
    cap = 256 if name == "tiny" else wl.capacity
    cap = cap // bs * bs
    ctx = tuple(45 + 30 * b for b in range(batch)) if name == "tiny" else wl.ctx
    dev = torch.device("cuda")
    w = synth.make_weights(shape, seed=0, device=dev)
    kc, vc = synth.make_kv(shape, batch, cap, ctx, seed=1, device=dev)
    mb = cap // bs
    n_blocks = batch * mb + 7
    rng = np.random.default_rng(5)
    table = rng.permutation(n_blocks)[:batch * mb].reshape(batch, mb).astype(np.int32)
    kp = [_pool_from(t, table, n_blocks, bs) for t in kc]
    vp = [_pool_from(t, table, n_blocks, bs) for t in vc]
    dc = mk.Decoder(shape, w, kc, vc, batch)
    dp = mk.Decoder(shape, w, kp, vp, batch, paged=(bs, n_blocks, cap))
    lc = torch.empty((batch, shape.vocab), dtype=torch.float32, device=dev)
    lp = torch.empty_like(lc)
    toks = synth.step_tokens(wl)
    for s in range(steps):
        tok = [int(toks[s, 0] + 11 * b) % shape.vocab for b in range(batch)]
        pos = [c + s for c in ctx]
        dc.step(tok, pos, lc)
        dp.step_paged(tok, pos, table, lp)
        assert dc.status() == mk.MK_OK and dp.status() == mk.MK_OK, dp.last_error()
        np.testing.assert_array_equal(lp.cpu().numpy(), lc.cpu().numpy())
    for l in range(shape.n_layers):
        assert torch.equal(_cache_from(kp[l], table, batch, cap, bs), kc[l])
        assert torch.equal(_cache_from(vp[l], table, batch, cap, bs), vc[l])
    with pytest.raises(mk.MkError) as e:
        dc.step_paged([1] * batch, list(ctx), table, lc)  # not a paged handle
    assert e.value.code == mk.MK_ERR_INVALID
    bad = table.copy()
    bad[0, ctx[0] // bs] = n_blocks
    with pytest.raises(mk.MkError) as e:
        dp.step_paged([1] * batch, list(ctx), bad, lp)
    assert e.value.code == mk.MK_ERR_INVALID
    with pytest.raises(mk.MkError) as e:
        dp.step([1] * batch, list(ctx), lp)  # a paged handle takes step_paged only
    assert e.value.code == mk.MK_ERR_INVALID
    dc.close()
    dp.close()


@pytest.mark.parametrize("name,batch,bs,steps,ctx", [
    ("tiny", 2, 16, 6, (45, 75)),
    ("tiny", 2, 5, 4, (33, 90)),
    ("llama1b", 1, 32, 8, (512,)),
    ("llama1b_ctx8k", 1, 16, 4, (8192,)),
])
def test_paged_matches_the_oracle(name, batch, bs, steps, ctx):
    """The paged path against the CPU oracle itself, not only against the
    contiguous CUDA path: the oracle decodes with a contiguous cache holding
    the same keys; the GPU reads them from a shuffled block pool through the
    block table. Per step the logits are within the parity bounds, the k/v row
    the GPU appends (into its block) agrees with the oracle's appended row
    within one bf16 ulp, and top-1 agreement holds over the run."""
    from tests.parity_util import KV_ATOL, KV_RTOL, Tally, bf16_bits, bits_to_f64, compare_logits
    from oracle import oracle as O
    wl = synth.WORKLOADS[name]
    shape = wl.shape
    cap = (256 if name == "tiny" else wl.capacity) // bs * bs
    dev = torch.device("cuda")
    w = synth.make_weights(shape, seed=0, device=dev)
    kc, vc = synth.make_kv(shape, batch, cap, ctx, seed=1, device=dev)
    model = O.Model(shape.as_dict(), synth.oracle_weights(w))
    ok = [bf16_bits(t).copy() for t in kc]
    ov = [bf16_bits(t).copy() for t in vc]
    mb = cap // bs
    n_blocks = batch * mb + 3
    rng = np.random.default_rng(11)
    table = rng.permutation(n_blocks)[:batch * mb].reshape(batch, mb).astype(np.int32)
    kp = [_pool_from(t, table, n_blocks, bs) for t in kc]
    vp = [_pool_from(t, table, n_blocks, bs) for t in vc]
    del kc, vc
    dp = mk.Decoder(shape, w, kp, vp, batch, paged=(bs, n_blocks, cap))
    lp = torch.empty((batch, shape.vocab), dtype=torch.float32, device=dev)
    toks = synth.step_tokens(wl)
    tally = Tally()
    for s in range(steps):
        tok = [int(toks[s % toks.shape[0], b % toks.shape[1]] + 7 * b) % shape.vocab
               for b in range(batch)]
        pos = [c + s for c in ctx]
        dp.step_paged(tok, pos, table, lp)
        assert dp.status() == mk.MK_OK, dp.last_error()
        want = model.decode_step(ok, ov, tok, pos)
        tally.add(compare_logits(lp.cpu().numpy().astype(np.float64), want))
        for l in range(shape.n_layers):
            for b, p in enumerate(pos):
                blk, row = int(table[b, p // bs]), p % bs
                np.testing.assert_allclose(bits_to_f64(bf16_bits(kp[l][blk, :, row])),
                                           bits_to_f64(ok[l][b][:, p]), rtol=KV_RTOL, atol=KV_ATOL)
                np.testing.assert_allclose(bits_to_f64(bf16_bits(vp[l][blk, :, row])),
                                           bits_to_f64(ov[l][b][:, p]), rtol=KV_RTOL, atol=KV_ATOL)
    print(name, bs, tally.check())
    dp.close()
