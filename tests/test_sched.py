"""Host scheduler checks (no GPU): the per-SM queues cover every output exactly
once, counter targets equal what the producers add up to, the queues cannot
deadlock under any interleaving of co-resident SMs, and every read-after-write
and write-after-read on the shared scratch is ordered by a counter chain.

The queues are the pre-planned per-SM instruction sequences of "3 · L'interpréteur
sur GPU" (§3.2); the counters are the zero-initialised global counters of §3.4,
including the four-chunk MLP dependency."""
import random

import numpy as np
import pytest

from decode_megakernel_03_gb300 import build as mkbuild
from decode_megakernel_03_gb300 import mk, synth

OPS = mk


@pytest.fixture(scope="module", autouse=True)
def _lib():
    mkbuild.build()


def _fused(B, shape):
    """One sequence with at most 2048 attention columns: no reduction
    instruction; the O-projection reduces the attention partials while it
    stages its input."""
    return B == 1 and shape.n_heads * shape.head_dim <= 2048


def _plan(shape, B, S, n_sm, pos):
    ins, off, tg = mk.schedule(shape, B, S, n_sm, pos)
    sm = np.zeros(len(ins), dtype=np.int64)
    for s in range(n_sm):
        sm[off[s]:off[s + 1]] = s
    return ins, off, tg, sm


CASES = [
    (synth.TINY, 1, 128, 8, [70]),
    (synth.TINY, 1, 128, 152, [0]),
    (synth.TINY, 2, 128, 5, [3, 127]),
    (synth.LLAMA_1B, 1, 640, 152, [512]),
    (synth.LLAMA_1B, 1, 8256, 152, [8200]),
    (synth.LLAMA_8B, 1, 2112, 152, [2048]),
    (synth.LLAMA_1B, 8, 4160, 152, list(synth.WORKLOADS["llama1b_b8"].ctx)),
    # four query heads per kv-head at batch 8, and head_dim 128 with a single kv-head
    (synth.ModelShape("g4", 2, 512, 8, 2, 64, 1024, 4096, tied=False, rope_theta=1e4), 8, 256, 152,
     [33 + 29 * b for b in range(8)]),
    (synth.ModelShape("d128g4", 2, 512, 4, 1, 128, 1024, 4096, tied=True, rope_theta=5e5), 1, 256,
     152, [33]),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0].name}-B{c[1]}-sm{c[3]}")
def test_deterministic(case):
    a = mk.schedule(*case)
    b = mk.schedule(*case)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def _ranges(ins, mask):
    r = sorted((int(a), int(b)) for a, b in zip(ins["a0"][mask], ins["a1"][mask]))
    return r


def _check_partition(r, n):
    assert r, "no work"
    assert r[0][0] == 0 and r[-1][1] == n
    for (a0, a1), (b0, b1) in zip(r, r[1:]):
        assert a1 == b0
    assert all(a < b for a, b in r)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0].name}-B{c[1]}-sm{c[3]}")
def test_every_output_produced_exactly_once(case):
    shape, B, S, n_sm, pos = case
    ins, off, tg, sm = _plan(*case)
    L, H, G = shape.n_layers, shape.hidden, shape.n_heads // shape.n_kv_heads
    pairs = shape.n_kv_heads * (G + 2) * (shape.head_dim // 2)
    Fc = shape.ffn // 4
    op, layer = ins["op"], ins["layer"]
    for l in range(L):
        _check_partition(_ranges(ins, (op == mk.OP_QKV) & (layer == l)), pairs)
        _check_partition(_ranges(ins, (op == mk.OP_OPROJ) & (layer == l)), H)
        for c in range(4):
            gu = (op == mk.OP_GATEUP) & (layer == l) & (ins["a2"] == c)
            r = _ranges(ins, gu)
            assert r[0][0] == c * Fc and r[-1][1] == (c + 1) * Fc
            _check_partition([(a - c * Fc, b - c * Fc) for a, b in r], Fc)
            _check_partition(_ranges(ins, (op == mk.OP_DOWN) & (layer == l) & (ins["a2"] == c)), H)
        # attention: each (b, g) has partitions 0..P-1 once, and its reduction
        # (a reduction instruction, or every O-projection unit) uses that P
        att = ins[(op == mk.OP_ATTN) & (layer == l)]
        if _fused(B, shape):
            assert not np.any((op == mk.OP_RED) & (layer == l))
            o = ins[(op == mk.OP_OPROJ) & (layer == l)]
            assert len(set(int(x) for x in o["a2"])) == 1
            red = [(0, g, int(o["a2"][0])) for g in range(shape.n_kv_heads)]
        else:
            red = [(int(r["a0"]), int(r["a1"]), int(r["a2"]))
                   for r in ins[(op == mk.OP_RED) & (layer == l)]]
        assert len(red) == B * shape.n_kv_heads
        for b, g, P in red:
            mine = att[(att["a0"] == b) & (att["a1"] == g)]
            assert sorted(int(x) >> 16 for x in mine["a2"]) == list(range(P))
            assert all((int(x) & 0xFFFF) == P for x in mine["a2"])
            assert 1 <= P <= min(64, pos[b] + 1)
        # a QKV instruction never spans two kv-head groups (one counter each)
        q = ins[(op == mk.OP_QKV) & (layer == l)]
        per = (G + 2) * (shape.head_dim // 2)
        assert np.all(q["a0"] // per == (q["a1"] - 1) // per)
    _check_partition(_ranges(ins, op == mk.OP_LMHEAD), shape.vocab)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0].name}-B{c[1]}-sm{c[3]}")
def test_every_gemv_fits_the_result_buffer_and_the_epilogue(case):
    """A GEMV instruction's results (items x rows per item x batch floats)
    fit one of the storer's result buffers, sized for the item cap of a
    row-pair instruction (64 items at batch 1, 32 at batch 2, 16 beyond), and
    its items fit the epilogue's two items per lane (at most 64)."""
    shape, B = case[0], case[1]
    ins, off, tg, sm = _plan(*case)
    cap = 64 if B == 1 else (32 if B == 2 else 16)
    res_floats = cap * 2 * B
    for op in (mk.OP_QKV, mk.OP_OPROJ, mk.OP_GATEUP, mk.OP_DOWN, mk.OP_LMHEAD):
        r = ins[ins["op"] == op]
        items = r["a1"] - r["a0"]
        rows = 2 if op in (mk.OP_QKV, mk.OP_GATEUP) else 1
        assert np.all(items >= 1)
        assert np.all(items <= 64), mk.OPS[op]
        assert np.all(items * rows * B <= res_floats), mk.OPS[op]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0].name}-B{c[1]}-sm{c[3]}")
def test_counter_targets(case):
    ins, off, tg, sm = _plan(*case)
    sums = np.zeros_like(tg)
    for c, a in zip(ins["sig_ctr"], ins["sig_amount"]):
        if c >= 0:
            sums[c] += a
    np.testing.assert_array_equal(sums, tg)
    w = ins["wait_ctr"] >= 0
    np.testing.assert_array_equal(ins["wait_target"][w], tg[ins["wait_ctr"][w]])
    assert np.all(tg[ins["wait_ctr"][w]] > 0), "every awaited counter is produced"


def _x_whole(shape, B):
    """Whether the chunk-3 down-projection storers write the layer output x
    whole (several sequences, or rows wider than 2048 columns)."""
    return B > 1 or shape.hidden > 2048


def _data_deps(ins, whole=True):
    """The waits that are not counters: when x is written whole, the storer
    of a chunk-3 down-projection instruction polls the shares of chunks 0..2
    (stamped words) before it writes the layer's output, so it publishes only
    after every chunk-0..2 instruction of its layer (and step) has published.
    Returns {instruction index: [instruction indices it waits for]}. (The
    simulations always add these waits: more waits cannot hide a deadlock.)"""
    if not whole:
        return {}
    dn = np.nonzero(ins["op"] == mk.OP_DOWN)[0]
    by_layer = {}
    for i in dn:
        if int(ins["a2"][i]) < 3:
            by_layer.setdefault(int(ins["layer"][i]), []).append(int(i))
    return {int(i): by_layer.get(int(ins["layer"][i]), []) for i in dn if int(ins["a2"][i]) == 3}


def _simulate(ins, off, tg, n_sm, pick):
    """Runs the queues on a CPU model: an SM may run the head of its queue
    once that instruction's counter reached its target."""
    ctr = np.zeros(len(tg), dtype=np.int64)
    head = [int(off[s]) for s in range(n_sm)]
    end = [int(off[s + 1]) for s in range(n_sm)]
    deps = _data_deps(ins)
    finished = np.zeros(len(ins), dtype=bool)
    done = 0
    total = int(off[-1])
    while done < total:
        ready = []
        for s in range(n_sm):
            if head[s] < end[s]:
                i = head[s]
                c = ins["wait_ctr"][i]
                if (c < 0 or ctr[c] >= ins["wait_target"][i]) and all(finished[d] for d in deps.get(i, ())):
                    ready.append(s)
        if not ready:
            return False
        s = pick(ready)
        i = head[s]
        if ins["sig_ctr"][i] >= 0:
            ctr[ins["sig_ctr"][i]] += ins["sig_amount"][i]
        finished[i] = True
        head[s] += 1
        done += 1
    np.testing.assert_array_equal(ctr, tg)
    return True


@pytest.mark.parametrize("case", CASES[:3] + [(synth.LLAMA_1B, 1, 640, 24, [600])],
                         ids=lambda c: f"{c[0].name}-B{c[1]}-sm{c[3]}")
def test_no_deadlock_under_any_interleaving(case):
    shape, B, S, n_sm, pos = case
    ins, off, tg, sm = _plan(*case)
    rng = random.Random(7)
    assert _simulate(ins, off, tg, n_sm, lambda r: r[0])
    assert _simulate(ins, off, tg, n_sm, lambda r: r[-1])
    for _ in range(3):
        assert _simulate(ins, off, tg, n_sm, lambda r: rng.choice(r))


def test_simulation_detects_a_bad_schedule():
    # the same check must fail when a wait can never be met
    ins, off, tg, sm = _plan(synth.TINY, 1, 128, 4, [10])
    bad = ins.copy()
    i = int(np.nonzero(bad["wait_ctr"] >= 0)[0][-1])
    bad["wait_target"][i] += 1
    assert not _simulate(bad, off, tg, 4, lambda r: r[0])


def _happens_before(ins, off, n_sm, whole=True):
    """Ancestor sets (as Python int bitmasks) of the DAG made of per-SM program
    order and counter edges (every producer of a counter precedes every
    instruction that waits for it)."""
    n = len(ins)
    preds = [[] for _ in range(n)]
    for s in range(n_sm):
        for i in range(int(off[s]) + 1, int(off[s + 1])):
            preds[i].append(i - 1)
    producers = {}
    for i in range(n):
        c = int(ins["sig_ctr"][i])
        if c >= 0:
            producers.setdefault(c, []).append(i)
    for i in range(n):
        c = int(ins["wait_ctr"][i])
        if c >= 0:
            preds[i].extend(producers[c])
    for i, ds in _data_deps(ins, whole).items():
        preds[i].extend(ds)
    # topological order by Kahn
    indeg = [len(p) for p in preds]
    succ = [[] for _ in range(n)]
    for i, ps in enumerate(preds):
        for p in ps:
            succ[p].append(i)
    order = [i for i in range(n) if indeg[i] == 0]
    k = 0
    while k < len(order):
        for j in succ[order[k]]:
            indeg[j] -= 1
            if indeg[j] == 0:
                order.append(j)
        k += 1
    assert len(order) == n, "cycle in the dependency graph"
    anc = [0] * n
    for i in order:
        a = 0
        for p in preds[i]:
            a |= anc[p] | (1 << p)
        anc[i] = a
    return anc


def _accesses(ins, shape, B):
    """Exact element keys of the shared scratch each instruction reads and
    writes (q, xa, the down-projection shares, x, h, partials and attention
    output are one buffer reused by every layer; the KV cache is per layer).
    A layer's output x (xa + its four down-projection shares, summed by the
    chunk-3 instructions' storers) is read by the next layer's QKV (all rows)
    and O-projection (its rows) and the LM head."""
    L, H, D, nkv = shape.n_layers, shape.hidden, shape.head_dim, shape.n_kv_heads
    G = shape.n_heads // nkv
    half = D // 2
    per = (G + 2) * half
    Fc = shape.ffn // 4
    whole = _x_whole(shape, B)

    def x_rows(lo, hi):
        if whole:
            return {("x", k) for k in range(lo, hi)}
        return ({("xa", k) for k in range(lo, hi)} |
                {("xpart", c, k) for c in range(4) for k in range(lo, hi)})

    acc = []
    for r in ins:
        op, l, a0, a1, a2 = int(r["op"]), int(r["layer"]), int(r["a0"]), int(r["a1"]), int(r["a2"])
        R, W = set(), set()
        if op == mk.OP_QKV:
            if l > 0:
                R |= x_rows(0, H)
            for j in range(a0, a1):
                slot = (j % per) // half
                W.add(("q", j) if slot < G else ("kv", l, j))
        elif op == mk.OP_ATTN:
            for j in range(a1 * per, (a1 + 1) * per):
                slot = (j % per) // half
                R.add(("q", j) if slot < G else ("kv", l, j))
            W.add(("part", a0, a1, a2 >> 16))
        elif op == mk.OP_RED:
            R |= {("part", a0, a1, p) for p in range(a2)}
            W.add(("attn", a0, a1))
        elif op == mk.OP_OPROJ:
            if _fused(B, shape):  # reduces every head's partitions while staging
                R |= {("part", 0, g, p) for g in range(nkv) for p in range(a2)}
            else:
                R |= {("attn", b, g) for b in range(B) for g in range(nkv)}
            if l > 0:
                R |= x_rows(a0, a1)
            W |= {("xa", k) for k in range(a0, a1)}
        elif op == mk.OP_GATEUP:
            R |= {("xa", k) for k in range(H)}
            W |= {("h", j) for j in range(a0, a1)}
        elif op == mk.OP_DOWN:
            R |= {("h", j) for j in range(a2 * Fc, (a2 + 1) * Fc)}
            if a2 == 3 and whole:  # the storer sums xa and the other shares into x
                R |= {("xa", k) for k in range(a0, a1)}
                R |= {("xpart", c, k) for c in range(3) for k in range(a0, a1)}
                W |= x_rows(a0, a1)
            else:
                W |= {("xpart", a2, k) for k in range(a0, a1)}
        elif op == mk.OP_LMHEAD:
            R |= x_rows(0, H)
        acc.append((R, W))
    return acc


WIDE = synth.ModelShape("wide", 2, 2304, 4, 2, 64, 1024, 512, tied=False, rope_theta=1e4)


@pytest.mark.parametrize("case", [(synth.TINY, 1, 128, 7, [70]), (synth.TINY, 2, 128, 3, [5, 90]),
                                  (synth.TINY, 1, 128, 152, [100]), (WIDE, 1, 128, 5, [40])],
                         ids=lambda c: f"B{c[1]}-sm{c[3]}")
def test_no_unordered_hazards(case):
    """Every pair of accesses to one scratch element, at least one of them a
    write (RAW, WAR, WAW), is ordered by program order or a counter chain."""
    shape, B, S, n_sm, pos = case
    ins, off, tg, sm = _plan(*case)
    anc = _happens_before(ins, off, n_sm, _x_whole(shape, B))
    touches = {}
    for i, (R, W) in enumerate(_accesses(ins, shape, B)):
        for k in R:
            touches.setdefault(k, []).append((i, False))
        for k in W:
            touches.setdefault(k, []).append((i, True))
    checked = 0
    for key, lst in touches.items():
        writers = [i for i, w in lst if w]
        for wi in writers:
            for j, _ in lst:
                if j == wi:
                    continue
                if not ((anc[j] >> wi) & 1 or (anc[wi] >> j) & 1):
                    raise AssertionError(f"unordered access to {key}: #{wi} {ins[wi]} / #{j} {ins[j]}")
                checked += 1
    assert checked > 1000


def _unordered(ins, anc, accs):
    touches = {}
    for i, (R, W) in enumerate(accs):
        for k in R:
            touches.setdefault(k, []).append((i, False))
        for k in W:
            touches.setdefault(k, []).append((i, True))
    for key, lst in touches.items():
        for wi in [i for i, w in lst if w]:
            for j, _ in lst:
                if j != wi and not ((anc[j] >> wi) & 1 or (anc[wi] >> j) & 1):
                    return key
    return None


def test_hazard_model_needs_the_chunk3_poll():
    """Without the chunk-3 storers' poll of the other shares, writing x whole
    would read the shares unordered: the hazard check must find it."""
    case = (synth.TINY, 2, 128, 3, [5, 90])
    ins, off, tg, sm = _plan(*case)
    accs = _accesses(ins, synth.TINY, 2)
    assert _unordered(ins, _happens_before(ins, off, 3, True), accs) is None
    key = _unordered(ins, _happens_before(ins, off, 3, False), accs)
    assert key is not None and key[0] == "xpart"


@pytest.mark.parametrize("B", [1, 8])
def test_chunked_down_waits_only_for_its_chunk(B):
    # the down-projection of chunk c waits for chunk c of h, not for the whole
    # hidden state; every SM runs the four gate/up chunks, then the
    # down-projection of one chunk (two where its range crosses a boundary)
    ctx = [512] if B == 1 else list(synth.WORKLOADS["llama1b_b8"].ctx)
    ins, off, tg, sm = _plan(synth.LLAMA_1B, B, 4160, 152, ctx)
    n_two = 0
    for s in range(152):
        q = ins[off[s]:off[s + 1]]
        l0 = q[q["layer"] == 0]
        seq = [(int(r["op"]), int(r["a2"])) for r in l0 if r["op"] in (mk.OP_GATEUP, mk.OP_DOWN)]
        gu = [x for x in seq if x[0] == mk.OP_GATEUP]
        dn_chunks = sorted(set(c for o, c in seq if o == mk.OP_DOWN))
        assert [c for _, c in gu] == [0, 1, 2, 3] and seq[:4] == gu, seq
        assert 1 <= len(dn_chunks) <= 2 and dn_chunks == list(range(dn_chunks[0], dn_chunks[-1] + 1))
        n_two += len(dn_chunks) == 2
    assert n_two <= 3  # only at the three chunk boundaries
    dn = ins[ins["op"] == mk.OP_DOWN]
    gu = ins[ins["op"] == mk.OP_GATEUP]
    for c in range(4):
        ctrs_dn = set(dn["wait_ctr"][dn["a2"] == c])
        ctrs_gu = set(gu["sig_ctr"][gu["a2"] == c])
        assert len(ctrs_dn) == 16 and ctrs_dn <= ctrs_gu
    # every layer's output counter counts the rows of all four chunks
    qkv = ins[(ins["op"] == mk.OP_QKV) & (ins["layer"] > 0)]
    assert np.all(qkv["wait_target"] == 4 * synth.LLAMA_1B.hidden)


def test_work_is_balanced_across_sms():
    ins, off, tg, sm = _plan(synth.LLAMA_1B, 1, 640, 152, [512])
    shape = synth.LLAMA_1B
    rowb = {mk.OP_QKV: 2 * shape.hidden * 2, mk.OP_OPROJ: shape.n_heads * shape.head_dim * 2,
            mk.OP_GATEUP: 2 * shape.hidden * 2, mk.OP_DOWN: shape.ffn // 4 * 2,
            mk.OP_LMHEAD: shape.hidden * 2}
    per_sm = np.zeros(152)
    for r, s in zip(ins, sm):
        if int(r["op"]) in rowb:
            per_sm[s] += (int(r["a1"]) - int(r["a0"])) * rowb[int(r["op"])]
    assert per_sm.max() / per_sm.mean() < 1.02


def _simulate_dynamic(ins, off, tg, n_sm, pick):
    """_simulate for a plan with a dynamic LM head: an SM whose head is the
    dynamic instruction (its wait met) may take the next ticket -- a row block
    counted into the LM head's counter -- until none is left, then moves on."""
    ctr = np.zeros(len(tg), dtype=np.int64)
    head = [int(off[s]) for s in range(n_sm)]
    end = [int(off[s + 1]) for s in range(n_sm)]
    next_ticket = 0
    taken = np.zeros(n_sm, dtype=np.int64)
    deps = _data_deps(ins)
    finished = np.zeros(len(ins), dtype=bool)
    while any(head[s] < end[s] for s in range(n_sm)):
        ready = []
        for s in range(n_sm):
            if head[s] < end[s]:
                i = head[s]
                c = ins["wait_ctr"][i]
                if (c < 0 or ctr[c] >= ins["wait_target"][i]) and all(finished[d] for d in deps.get(i, ())):
                    ready.append(s)
        if not ready:
            return False, None
        s = pick(ready)
        r = ins[head[s]]
        if r["op"] == mk.OP_LMHEAD and r["a2"] > 0:
            rows, total = int(r["a0"]), int(r["a1"])
            if next_ticket * rows < total:
                ctr[r["sig_ctr"]] += min(total, (next_ticket + 1) * rows) - next_ticket * rows
                next_ticket += 1
                taken[s] += 1
                continue
            head[s] += 1  # no ticket left
            continue
        if r["sig_ctr"] >= 0:
            ctr[r["sig_ctr"]] += r["sig_amount"]
        finished[head[s]] = True
        head[s] += 1
    return np.array_equal(ctr, tg), taken


@pytest.mark.parametrize("case", [CASES[0], CASES[2], (synth.LLAMA_1B, 1, 640, 24, [600]),
                                  (synth.LLAMA_1B, 8, 4160, 40, list(synth.WORKLOADS["llama1b_b8"].ctx))],
                         ids=lambda c: f"{c[0].name}-B{c[1]}-sm{c[3]}")
def test_dynamic_lm_head_plan(case):
    """Dynamic LM head (MK_DYN_LMHEAD): every SM's queue ends with one
    dynamic instruction over all vocabulary rows, its counter's target is the
    vocabulary size, and under any interleaving the SMs take every ticket
    exactly once, the counters reach their targets and nothing deadlocks;
    an SM that runs ahead takes more of the LM head."""
    shape, B, S, n_sm, pos = case
    ins, off, tg = mk.schedule(shape, B, S, n_sm, pos, dyn=mk.DYN_LMHEAD)
    st, _, tg_static = mk.schedule(shape, B, S, n_sm, pos)
    lm = ins[ins["op"] == mk.OP_LMHEAD]
    assert len(lm) == n_sm and np.all(lm["a2"] > 0) and np.all(lm["a1"] == shape.vocab)
    for s in range(n_sm):
        q = ins[off[s]:off[s + 1]]
        assert q[-1]["op"] == mk.OP_LMHEAD
    np.testing.assert_array_equal(tg, tg_static)
    # everything before the LM head is the static plan
    np.testing.assert_array_equal(ins[ins["op"] != mk.OP_LMHEAD], st[st["op"] != mk.OP_LMHEAD])
    rng = random.Random(3)
    ok, taken = _simulate_dynamic(ins, off, tg, n_sm, lambda r: r[0])
    assert ok
    n_tickets = -(-shape.vocab // int(lm["a0"][0]))
    assert taken.sum() == n_tickets
    assert taken[0] > taken[-1]  # SM 0 always runs first here: it takes the most
    for _ in range(2):
        ok, taken = _simulate_dynamic(ins, off, tg, n_sm, lambda r: rng.choice(r))
        assert ok and taken.sum() == n_tickets


# ---------------------------------------------------------------------------
# A model of the three warp roles of every SM, not only of the instruction
# waits: the loader issues each instruction's pages in queue order into a ring
# of `ring` slots (a slot frees when the compute warps have read its page),
# and holds -- issues no page of a later instruction -- while an attention
# unit is being computed and not yet published; in a prefill step
# it fetches an attention unit's keys only once the unit's counter is met.
# The compute warps raise the hold on reaching a critical instruction (before
# its waits), run an instruction once its counter is met and one of the
# kResBufs result buffers is free, and read its pages as they arrive. The
# storer publishes the computed instructions in order.

RESBUFS = 4


def _pages(r, shape, B, pos):
    """Pages the loader issues for instruction r (the kernel's page geometry)."""
    op, a0, a1, a2 = int(r["op"]), int(r["a0"]), int(r["a1"]), int(r["a2"])
    H, D, QD, Fc = shape.hidden, shape.head_dim, shape.n_heads * shape.head_dim, shape.ffn // 4
    if op == mk.OP_ATTN:
        p = pos[a0] + ((int(r["layer"]) >> 10) & 31)
        pidx, P = a2 >> 16, a2 & 0xFFFF
        t0, t1 = pidx * (p + 1) // P, (pidx + 1) * (p + 1) // P
        nc = max(0, min(t1, p) - t0)
        kpp = 16384 // (4 * D)
        return -(-nc // kpp)
    if op == mk.OP_RED:
        return 0
    K = {mk.OP_QKV: H, mk.OP_OPROJ: QD, mk.OP_GATEUP: H, mk.OP_DOWN: Fc, mk.OP_LMHEAD: H}[op]
    R = 2 if op in (mk.OP_QKV, mk.OP_GATEUP) else 1
    ipp = 16384 // (R * K * 2)
    return -(-(a1 - a0) // ipp)


def _critical(r):
    # the instruction whose output goes out behind a release fence
    return r["op"] == mk.OP_ATTN


def _simulate_roles(ins, off, tg, n_sm, shape, B, pos, ring, pick, prefill=False,
                    hold_own_pages=False, lm_of_step=None):
    """Runs the role model; returns True when every queue completes with the
    counters at their targets, False on a deadlock (no role can move).
    lm_of_step: for a plan of several steps in one launch, the LM-head counter
    of each step; the loader fetches a step s > 0 attention unit's keys only
    once step s - 1's LM head is complete (its keys were written by step
    s - 1). hold_own_pages plants a mistake for the model's own check: the
    hold also stops the pages of the critical instruction itself."""
    ctr = np.zeros(len(tg), dtype=np.int64)
    pages = [[_pages(ins[i], shape, B, pos) for i in range(int(off[s]), int(off[s + 1]))]
             for s in range(n_sm)]
    n = [int(off[s + 1] - off[s]) for s in range(n_sm)]
    lp = [0] * n_sm      # loader: instruction, pages issued of it
    lpg = [0] * n_sm
    issued = [0] * n_sm  # pages issued in total
    used = [0] * n_sm    # pages read by the compute warps in total
    cp = [0] * n_sm      # compute: instruction, and whether its wait is met
    cwait = [False] * n_sm
    cpg = [0] * n_sm     # pages of it read
    sp = [0] * n_sm      # storer: instructions published
    hold = [-1] * n_sm

    def I(s, k):
        return ins[int(off[s]) + k]

    def met(r):
        c = int(r["wait_ctr"])
        return c < 0 or ctr[c] >= r["wait_target"]

    deps = _data_deps(ins)
    stored = np.zeros(len(ins), dtype=bool)

    def enter(s):
        if cp[s] < n[s] and _critical(I(s, cp[s])):
            hold[s] = cp[s]

    for s in range(n_sm):
        enter(s)

    while any(sp[s] < n[s] for s in range(n_sm)):
        acts = []
        for s in range(n_sm):
            # loader: the next page
            if lp[s] < n[s]:
                if lpg[s] >= pages[s][lp[s]]:
                    acts.append(("ladv", s))
                else:
                    h = hold[s]
                    held = h >= 0 and sp[s] <= h and (lp[s] > h or (hold_own_pages and lp[s] == h))
                    r = I(s, lp[s])
                    gated = prefill and r["op"] == mk.OP_ATTN and not met(r)
                    st = (int(r["layer"]) >> 10) & 31
                    if lm_of_step is not None and r["op"] == mk.OP_ATTN and st > 0:
                        c = lm_of_step[st - 1]
                        gated = gated or ctr[c] < tg[c]
                    if issued[s] - used[s] < ring and not held and not gated:
                        acts.append(("load", s))
            # compute
            if cp[s] < n[s]:
                r = I(s, cp[s])
                if not cwait[s]:
                    if met(r) and cp[s] - sp[s] < RESBUFS:
                        acts.append(("cwait", s))
                elif cpg[s] < pages[s][cp[s]]:
                    if used[s] < issued[s]:
                        acts.append(("use", s))
                else:
                    acts.append(("cdone", s))
            # storer (a chunk-3 down-projection's storer polls the other
            # chunks' shares first)
            if sp[s] < cp[s] and all(stored[d] for d in deps.get(int(off[s]) + sp[s], ())):
                acts.append(("store", s))
        if not acts:
            return False
        kind, s = pick(acts)
        if kind == "ladv":
            lp[s] += 1
            lpg[s] = 0
        elif kind == "load":
            # every page that fits: the ring state after a run of single
            # issues, with fewer interleavings to walk through
            k = min(pages[s][lp[s]] - lpg[s], ring - (issued[s] - used[s]))
            lpg[s] += k
            issued[s] += k
        elif kind == "cwait":
            cwait[s] = True
        elif kind == "use":
            k = min(pages[s][cp[s]] - cpg[s], issued[s] - used[s])
            cpg[s] += k
            used[s] += k
        elif kind == "cdone":
            cp[s] += 1
            cwait[s] = False
            cpg[s] = 0
            enter(s)
        else:
            r = I(s, sp[s])
            if r["sig_ctr"] >= 0:
                ctr[r["sig_ctr"]] += r["sig_amount"]
            stored[int(off[s]) + sp[s]] = True
            sp[s] += 1
    return bool(np.array_equal(ctr, tg))


ROLE_CASES = [
    (synth.TINY, 1, 128, 8, [70], 12),
    (synth.TINY, 2, 128, 5, [3, 127], 6),
    (synth.TINY, 8, 128, 7, [5 * b + 1 for b in range(8)], 6),
    (synth.LLAMA_1B, 1, 640, 24, [600], 6),
    (synth.LLAMA_8B, 1, 2112, 16, [2048], 12),
]


@pytest.mark.parametrize("case", ROLE_CASES, ids=lambda c: f"{c[0].name}-B{c[1]}-sm{c[3]}-ring{c[5]}")
def test_roles_cannot_deadlock(case):
    """Loader, compute warps and storer of every SM, with the page ring, the
    result buffers and the loader's hold: every random interleaving finishes
    and the counters reach their targets."""
    shape, B, S, n_sm, pos, ring = case
    ins, off, tg, sm = _plan(shape, B, S, n_sm, pos)
    rng = random.Random(11)
    picks = [lambda a: a[0], lambda a: rng.choice(a)]
    if shape is synth.TINY:
        picks += [lambda a: a[-1]] + [lambda a: rng.choice(a)] * 3
    for pick in picks:
        assert _simulate_roles(ins, off, tg, n_sm, shape, B, pos, ring, pick)


def test_roles_prefill_cannot_deadlock():
    """A prefill step (the batch rows are consecutive tokens of one sequence):
    the loader also waits for each attention unit's counter before its keys."""
    shape = synth.TINY
    pos = [40 + b for b in range(8)]
    ins, off, tg, sm = _plan(shape, 8, 128, 6, pos)
    rng = random.Random(12)
    for pick in (lambda a: a[0], lambda a: a[-1], lambda a: rng.choice(a)):
        assert _simulate_roles(ins, off, tg, 6, shape, 8, pos, 6, pick, prefill=True)


def test_role_model_detects_a_hold_on_the_critical_instructions_own_pages():
    """The same model deadlocks when the hold also stops the critical
    instruction's own pages: its compute waits for pages the loader will not
    issue until the instruction is published (8 SMs: attention units of 10
    key pages, more than the 6-page ring lets the loader issue ahead)."""
    shape, pos = synth.LLAMA_1B, [600]
    ins, off, tg, sm = _plan(shape, 1, 640, 8, pos)
    assert not _simulate_roles(ins, off, tg, 8, shape, 1, pos, 6, lambda a: a[0],
                               hold_own_pages=True)
    assert _simulate_roles(ins, off, tg, 8, shape, 1, pos, 6, lambda a: a[0])


# ---------------------------------------------------------------------------
# Several greedy steps in one launch (the plan of mk_decode_greedy_persistent)

STEP_CASES = [
    (synth.TINY, 2, 128, 5, [3, 60], 3),
    (synth.TINY, 1, 128, 8, [0], 4),
    (synth.TINY, 8, 128, 7, [5 * b + 1 for b in range(8)], 2),
    (synth.LLAMA_1B, 1, 640, 24, [500], 2),
]


def _lm_counter(shape, B):
    L, nkv = shape.n_layers, shape.n_kv_heads
    return 3 * L + L * nkv + L * B * nkv + L * 4


@pytest.mark.parametrize("case", STEP_CASES, ids=lambda c: f"{c[0].name}-B{c[1]}-k{c[5]}")
def test_steps_plan_is_the_step_plans_in_sequence(case):
    """Step s of the one-launch plan is the single-step plan at positions + s
    with its counters offset by s times the per-step count; only step s > 0's
    layer-0 QKV instructions differ: they wait for step s - 1's LM head (their
    token is its argmax), which every queue holds before them."""
    shape, B, S, n_sm, pos, k = case
    ins, off, tg = mk.schedule_steps(shape, B, S, n_sm, pos, k)
    n = len(tg) // k
    assert len(tg) == k * n
    lm = _lm_counter(shape, B)
    st = (ins["layer"] >> 10) & 31
    for m in range(n_sm):
        q = st[off[m]:off[m + 1]]
        assert np.all(np.diff(q) >= 0), "each queue runs its steps in order"
    for s_ in range(k):
        one, o1, t1 = mk.schedule(shape, B, S, n_sm, [p + s_ for p in pos])
        np.testing.assert_array_equal(tg[s_ * n:(s_ + 1) * n], t1)
        for m in range(n_sm):
            q = ins[off[m]:off[m + 1]]
            q = q[((q["layer"] >> 10) & 31) == s_].copy()
            r = one[o1[m]:o1[m + 1]]
            q["layer"] &= 1023
            g = q["sig_ctr"] >= 0
            q["sig_ctr"][g] -= s_ * n
            first = (q["op"] == mk.OP_QKV) & (q["layer"] == 0)
            if s_ > 0:
                assert np.all(q["wait_ctr"][first] == (s_ - 1) * n + lm)
                assert np.all(q["wait_target"][first] == shape.vocab)
                q["wait_ctr"][first] = r["wait_ctr"][first]
                q["wait_target"][first] = r["wait_target"][first]
            w = (q["wait_ctr"] >= 0) & ~(first & (s_ > 0))
            q["wait_ctr"][w] -= s_ * n
            np.testing.assert_array_equal(q, r)


@pytest.mark.parametrize("case", STEP_CASES, ids=lambda c: f"{c[0].name}-B{c[1]}-k{c[5]}")
def test_steps_plan_cannot_deadlock(case):
    """Instruction-level waits and the three-role model with the loader's
    acquire of the previous step's LM head before a later step's keys."""
    shape, B, S, n_sm, pos, k = case
    ins, off, tg = mk.schedule_steps(shape, B, S, n_sm, pos, k)
    n = len(tg) // k
    lm = [s_ * n + _lm_counter(shape, B) for s_ in range(k)]
    rng = random.Random(13)
    picks = [lambda a: a[0]]
    if shape is synth.TINY:
        picks += [lambda a: a[-1], lambda a: rng.choice(a), lambda a: rng.choice(a)]
    for pick in picks:
        assert _simulate(ins, off, tg, n_sm, pick)
        assert _simulate_roles(ins, off, tg, n_sm, shape, B, pos, 6, pick, lm_of_step=lm)


def test_role_model_detects_a_key_fetch_gated_on_its_own_steps_lm_head():
    """Gating step s's key fetch on step s's own LM head (which follows the
    attention in every queue) deadlocks the model."""
    shape, B, S, n_sm, pos, k = STEP_CASES[0]
    ins, off, tg = mk.schedule_steps(shape, B, S, n_sm, pos, k)
    n = len(tg) // k
    lm = [s_ * n + _lm_counter(shape, B) for s_ in range(k)]
    assert not _simulate_roles(ins, off, tg, n_sm, shape, B, pos, 6, lambda a: a[0],
                               lm_of_step=lm[1:])


def test_steps_schedule_rejects_bad_arguments():
    with pytest.raises(mk.MkError):
        mk.schedule_steps(synth.TINY, 1, 128, 4, [0], 0)
    with pytest.raises(mk.MkError):
        mk.schedule_steps(synth.TINY, 1, 128, 4, [0], mk.MAX_STEPS_PER_LAUNCH + 1)
    with pytest.raises(mk.MkError):
        mk.schedule_steps(synth.TINY, 1, 128, 4, [126], 3)  # 126 + 2 reaches capacity
    mk.schedule_steps(synth.TINY, 1, 128, 4, [125], 3)
