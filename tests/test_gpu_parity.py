"""Parity of the CUDA decode path (through the C ABI) with the CPU oracle.

Every test feeds both sides the same seeded inputs and compares the logits of
every decode step (relative L2 <= 1e-2, max-abs <= 5e-2, top-1 agreement),
the KV-cache slot each step writes (within one bf16 ulp) and, bit-exactly,
the untouched slots and the final counter values of the schedule.
"""
import numpy as np
import pytest
import torch

from decode_megakernel_03_gb300 import mk, synth
from oracle import oracle as O
from tests.parity_util import (Pair, Tally, bf16_bits, bits_to_f64, check_kv_step, check_untouched,
                               check_written_rows, compare_logits, counters_match)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _tiny_prefilled():
    """The tiny workload: a 64-token prompt prefilled into the KV cache by the
    oracle's causal forward (the same bytes go to both sides)."""
    wl = synth.WORKLOADS["tiny"]
    shape = wl.shape
    w = synth.make_weights(shape, seed=wl.weight_seed)
    model = O.Model(shape.as_dict(), synth.oracle_weights(w))
    prompt = synth.prompt_tokens(wl).numpy()
    _, kf, vf = model.forward_full(prompt, want_kv=True)
    ks, vs = [], []
    for l in range(shape.n_layers):
        k = np.zeros((1, shape.n_kv_heads, wl.capacity, shape.head_dim), np.uint16)
        v = k.copy()
        k[0, :, :wl.prompt] = kf[l]
        v[0, :, :wl.prompt] = vf[l]
        ks.append(k)
        vs.append(v)
    return wl, ks, vs


def test_tiny_teacher_forced_decode():
    wl, ks, vs = _tiny_prefilled()
    pair = Pair(wl.shape, 1, wl.capacity, kv_from_oracle=(ks, vs), weight_seed=wl.weight_seed)
    toks = synth.step_tokens(wl)
    tally = Tally()
    for s in range(wl.steps):
        tok, pos = [int(toks[s, 0])], synth.step_positions(wl, s)
        bk = [bf16_bits(t) for t in pair.kc]
        bv = [bf16_bits(t) for t in pair.vc]
        got = pair.gpu_step(tok, pos)
        want = pair.oracle_step(tok, pos)
        tally.add(compare_logits(got, want))
        check_kv_step(pair, pos, bk, bv)
        counters_match(pair, pos)
    print("tiny", tally.check())
    pair.close()


def test_tiny_decode_from_empty_cache_matches_full_forward():
    """The GPU decodes the whole 80-token sequence one token at a time from an
    empty cache; its logits and final cache match the oracle's causal forward."""
    wl = synth.WORKLOADS["tiny"]
    pair = Pair(wl.shape, 1, wl.capacity, weight_seed=wl.weight_seed)
    toks = np.concatenate([synth.prompt_tokens(wl).numpy(), synth.step_tokens(wl)[:, 0].numpy()])
    full, kf, vf = pair.model.forward_full(toks, want_kv=True)
    tally = Tally()
    for t in range(len(toks)):
        got = pair.gpu_step([int(toks[t])], [t])
        tally.add(compare_logits(got, full[t:t + 1]))
    for l in range(wl.shape.n_layers):
        n = len(toks)
        np.testing.assert_allclose(bits_to_f64(bf16_bits(pair.kc[l])[0, :, :n]), bits_to_f64(kf[l]),
                                   rtol=2.0 ** -7, atol=1e-3)
        np.testing.assert_allclose(bits_to_f64(bf16_bits(pair.vc[l])[0, :, :n]), bits_to_f64(vf[l]),
                                   rtol=2.0 ** -7, atol=1e-3)
    print("tiny from empty", tally.check())
    pair.close()


@pytest.mark.parametrize("shape_name", ["tiny", "llama1b", "llama1b_b8"])
def test_multilaunch_graph_and_generic_kernel_are_bit_identical(shape_name):
    wl = synth.WORKLOADS[shape_name]
    ctx = (200,) if shape_name == "tiny" else wl.ctx
    cap = 256 if shape_name == "tiny" else wl.capacity
    batch = wl.batch
    toks = synth.step_tokens(wl)
    outs = {}
    caches = {}
    for mode in ("mega", "multi", "graph", "generic"):
        pair = Pair(wl.shape, batch, cap, ctx=ctx)
        if mode == "generic":  # the instantiation that reads the head shape at run time
            pair.dec.use_generic_kernel(True)
        res = []
        for s in range(3):
            tok = [int(t) for t in toks[s][:batch]]
            res.append(pair.gpu_step(tok, [c + s for c in ctx],
                                     mode="mega" if mode == "generic" else mode))
        outs[mode] = np.stack(res)
        caches[mode] = [bf16_bits(t) for t in pair.kc + pair.vc]
        if mode == "mega":
            counters_match(pair, [c + 2 for c in ctx])
        pair.close()
    for other in ("multi", "graph", "generic"):
        np.testing.assert_array_equal(outs["mega"], outs[other])
        for a, b in zip(caches["mega"], caches[other]):
            np.testing.assert_array_equal(a, b)


WIDE = synth.ModelShape("wide", 2, 2304, 4, 2, 64, 1024, 4096, tied=False, rope_theta=10000.0)


@pytest.mark.parametrize("batch", [1, 2])
def test_wide_rows_whole_x_matches_the_oracle_and_the_multilaunch_build(batch):
    """Rows wider than 2048 columns: the chunk-3 down-projection storers write
    the layer output whole in the megakernel, while the multi-launch build's
    readers add up its five sources; both round the same way, so the builds
    agree bit for bit, and both match the oracle."""
    cap = 128
    ctx = tuple(40 + 17 * b for b in range(batch))
    outs = {}
    tally = Tally()
    for mode in ("mega", "multi", "graph"):
        pair = Pair(WIDE, batch, cap, ctx=ctx)
        res = []
        for s_ in range(3):
            tok = [(71 * s_ + 13 * b + 5) % WIDE.vocab for b in range(batch)]
            pos = [c + s_ for c in ctx]
            got = pair.gpu_step(tok, pos, mode=mode).copy()
            if mode == "mega":
                tally.add(compare_logits(got, pair.oracle_step(tok, pos)))
            res.append(got)
        outs[mode] = np.stack(res)
        pair.close()
    np.testing.assert_array_equal(outs["mega"], outs["multi"])
    np.testing.assert_array_equal(outs["mega"], outs["graph"])
    print("wide", batch, tally.check())


@pytest.mark.parametrize("name", ["llama1b", "llama1b_ctx8k", "llama8b", "llama1b_b8"])
def test_full_size_parity(name):
    """Each workload at full size on its seeded context, over every one of its
    teacher-forced decode steps (128 for the 1B shape at ctx 512, 64 for the
    others): per-step logit bounds, top-1 agreement over the run, the k/v row
    each step appends (GPU and oracle each append their own), the untouched
    slots bit-exact at the end, and the counters of every step."""
    wl = synth.WORKLOADS[name]
    pair = Pair(wl.shape, wl.batch, wl.capacity, ctx=wl.ctx, weight_seed=wl.weight_seed,
                kv_seed=wl.kv_seed)
    toks = synth.step_tokens(wl)
    before_k = [bf16_bits(t) for t in pair.kc]
    before_v = [bf16_bits(t) for t in pair.vc]
    written = [set() for _ in range(wl.batch)]
    tally = Tally()
    for s in range(wl.steps):
        tok = [int(t) for t in toks[s]]
        pos = synth.step_positions(wl, s)
        got = pair.gpu_step(tok, pos)
        want = pair.oracle_step(tok, pos)
        tally.add(compare_logits(got, want))
        check_written_rows(pair, pos)
        counters_match(pair, pos)
        for b, p in enumerate(pos):
            written[b].add(p)
    check_untouched(pair, before_k, before_v, written)
    print(name, tally.check())
    pair.close()


def test_edge_positions_first_and_last_slot():
    shape = synth.TINY
    cap = 96
    pair = Pair(shape, 2, cap, ctx=(0, cap - 1))
    tally = Tally()
    for tok, pos in (([5, 6], [0, cap - 1]), ([7, 8], [1, cap - 1])):
        bk = [bf16_bits(t) for t in pair.kc]
        bv = [bf16_bits(t) for t in pair.vc]
        got = pair.gpu_step(tok, pos)
        want = pair.oracle_step(tok, pos)
        tally.add(compare_logits(got, want))
        check_kv_step(pair, pos, bk, bv)
    tally.check()
    pair.close()


@pytest.mark.parametrize("batch", [2, 4])
def test_other_batch_sizes(batch):
    shape = synth.TINY
    cap = 160
    ctx = tuple(17 + 37 * b for b in range(batch))
    pair = Pair(shape, batch, cap, ctx=ctx)
    tally = Tally()
    for s in range(2):
        tok = [(11 * s + 3 * b) % shape.vocab for b in range(batch)]
        pos = [c + s for c in ctx]
        got = pair.gpu_step(tok, pos)
        want = pair.oracle_step(tok, pos)
        tally.add(compare_logits(got, want))
    tally.check()
    pair.close()


def test_repeated_steps_are_bitwise_deterministic():
    """1000 repetitions of one step, and the same step with the per-SM queues
    handed to the CTAs in several random orders: every result is bit-identical
    and every counter ends at its target."""
    wl = synth.WORKLOADS["llama1b"]
    pair = Pair(wl.shape, 1, wl.capacity, ctx=wl.ctx)
    ref = pair.gpu_step([17], [512]).copy()
    for _ in range(1000):
        pair.dec.step([17], [512], pair.logits)
    assert pair.dec.status() == mk.MK_OK
    np.testing.assert_array_equal(pair.logits.cpu().numpy().astype(np.float64), ref)
    for seed in (1, 2, 3, 4):
        pair.dec.permute_queues(seed)
        got = pair.gpu_step([17], [512])
        np.testing.assert_array_equal(got, ref)
        counters_match(pair, [512])
    pair.dec.permute_queues(0)
    pair.close()


@pytest.mark.parametrize("wl_name", ["tiny_b2", "llama1b"])
def test_builds_interleaved_on_one_handle(wl_name):
    """Values handed between instructions carry the step's stamp, which
    alternates from step to step on a handle. One handle that interleaves the
    megakernel, the multi-launch build (plain and as a CUDA graph) and
    several-step greedy launches gives, step for step, the same bits as a
    handle that runs only megakernel steps: the results do not depend on the
    stamp, and every build keeps the stamp sequence consistent."""
    if wl_name == "tiny_b2":
        shape, batch, cap, ctx = synth.TINY, 2, 128, (40, 71)
    else:
        wl = synth.WORKLOADS["llama1b"]
        shape, batch, cap, ctx = wl.shape, 1, wl.capacity, wl.ctx
    a = Pair(shape, batch, cap, ctx=ctx)
    b = Pair(shape, batch, cap, ctx=ctx)
    dev = torch.device("cuda")
    toks_out = torch.empty((8, batch), dtype=torch.int32, device=dev)
    modes = ["mega", "multi", "graph", "greedy3", "mega", "graph", "greedy2", "multi", "mega"]
    s = 0
    for mode in modes:
        tok = [(29 * s + 5 * i + 3) % shape.vocab for i in range(batch)]
        pos = [c + s for c in ctx]
        if mode.startswith("greedy"):
            n = int(mode[-1])
            a.dec.decode_greedy_persistent(tok, pos, n, toks_out, a.logits)
            assert a.dec.status() == mk.MK_OK, a.dec.last_error()
            got = a.logits.cpu().numpy().astype(np.float64)
            seq = toks_out[:n].cpu().numpy()
            cur = tok
            for k in range(n):
                want = b.gpu_step(cur, [c + s + k for c in ctx]).copy()
                nxt = [int(np.argmax(want[i].astype(np.float32))) for i in range(batch)]
                assert list(seq[k]) == nxt
                cur = nxt
            np.testing.assert_array_equal(got, want)
            s += n
        else:
            got = a.gpu_step(tok, pos, mode=mode).copy()
            want = b.gpu_step(tok, pos)
            np.testing.assert_array_equal(got, want)
            s += 1
    for x, y in zip(a.kc + a.vc, b.kc + b.vc):
        assert torch.equal(x, y)
    a.close()
    b.close()


def test_unsatisfiable_wait_times_out_and_recovers():
    """A host-built schedule with one wait that can never be met: the bounded
    device wait expires, the step reports MK_ERR_TIMEOUT, the next step call is
    refused until the status is read, and the handle then works again."""
    shape = synth.TINY
    pair = Pair(shape, 1, 128, ctx=(40,))
    good = pair.gpu_step([3], [40]).copy()
    pair.dec.set_timeout(50_000_000)  # 50 ms
    pair.dec.inject_unsatisfiable_wait(True)
    pair.dec.step([3], [40], pair.logits)
    torch.cuda.synchronize()
    with pytest.raises(mk.MkError) as e:
        pair.dec.step([3], [40], pair.logits)
    assert e.value.code == mk.MK_ERR_TIMEOUT
    assert pair.dec.status() == mk.MK_ERR_TIMEOUT
    assert pair.dec.status() == mk.MK_OK
    pair.dec.inject_unsatisfiable_wait(False)
    pair.dec.set_timeout(2_000_000_000)
    again = pair.gpu_step([3], [40])
    np.testing.assert_array_equal(again, good)
    pair.close()


# shapes the workloads do not cover: 8 query heads per kv-head (the most the
# tensor-core attention takes in one product), head_dim 128 with several
# sequences, and a tied head on the generic kernels
G8 = synth.ModelShape("g8", 2, 512, 8, 1, 64, 1024, 4096, tied=False, rope_theta=10000.0)
D128 = synth.ModelShape("d128", 2, 512, 4, 2, 128, 1024, 4096, tied=True, rope_theta=10000.0)


@pytest.mark.parametrize("shape,batch", [(G8, 1), (G8, 2), (G8, 8), (D128, 1), (D128, 2)])
def test_other_head_shapes(shape, batch):
    cap = 256
    ctx = tuple(70 + 41 * b % 150 for b in range(batch))
    pair = Pair(shape, batch, cap, ctx=ctx)
    tally = Tally()
    for s in range(2):
        tok = [(13 * s + 7 * b + 1) % shape.vocab for b in range(batch)]
        pos = [c + s for c in ctx]
        bk = [bf16_bits(t) for t in pair.kc]
        bv = [bf16_bits(t) for t in pair.vc]
        got = pair.gpu_step(tok, pos)
        want = pair.oracle_step(tok, pos)
        tally.add(compare_logits(got, want))
        check_kv_step(pair, pos, bk, bv)
    print(shape.name, batch, tally.check())
    pair.close()
