"""Decode benchmark: one decode step of a Llama-style model per "step".

Default workload: the Llama-3.2-1B-shaped decoder (16 layers, hidden 2048,
32/8 heads, FFN 8192, vocab 128256, tied), batch 1, KV context 512, timed over
the workload's 128 teacher-forced decode steps (positions 512..639). Weights and
caches are seeded synthetic data (random init), resident in HBM before the
timed region. Every step streams ~2.49 GB (all weights + the KV read), far more
than the 129 MB L2, so no flush is needed between steps.

Prints ONE JSON line. `--impl reference` times the CPU oracle instead (the
reference arm of this comparison), on a bounded sample of the same workload.
Under torchrun (N > 1) every rank runs an independent replica (no collective
on the data path) and rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode µs/token & tokens/s, Llama-1B shape batch 1; % of GB300 HBM roofline"


def algorithmic_bytes(shape, batch, positions):
    """Bytes the method must move per step: every weight matrix and norm gain,
    the final norm, the LM head, one embedding row per sequence, and the KV
    cache read over slots 0..pos of every layer and sequence (the new slot
    included). Logit writes and scratch traffic are not counted."""
    H, D, F, V, L = shape.hidden, shape.head_dim, shape.ffn, shape.vocab, shape.n_layers
    per_layer = 2 * (H * shape.n_heads * D * 2 + H * shape.n_kv_heads * D * 2 + 3 * H * F + 2 * H)
    weights = L * per_layer + 2 * H + 2 * V * H + 2 * H * batch
    kv = sum(L * 2 * shape.n_kv_heads * D * 2 * (p + 1) for p in positions)
    return weights, kv


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_oracle_rate(wl, w_host, target_s=12.0, max_steps=64):
    """Times the oracle as it stands on this host's cores: decode steps of the
    same workload until about target_s seconds of CPU work."""
    from oracle import oracle as O
    shape = wl.shape
    model = O.Model(shape.as_dict(), w_host)
    from decode_megakernel_03_gb300 import synth
    kc, vc = synth.make_kv(shape, wl.batch, wl.capacity, wl.ctx, seed=wl.kv_seed)
    ks = [synth.bits(t).copy() for t in kc]
    vs = [synth.bits(t).copy() for t in vc]
    toks = synth.step_tokens(wl)
    threads = O.default_threads()
    t0 = time.perf_counter()
    n = 0
    while n < max_steps:
        model.decode_step(ks, vs, [int(t) for t in toks[n % wl.steps]],
                          synth.step_positions(wl, n % wl.steps), nthreads=threads)
        n += 1
        if time.perf_counter() - t0 > target_s:
            break
    dt = time.perf_counter() - t0
    return n * wl.batch / dt, n, dt, threads


def oracle_timings(names=("tiny", "llama1b", "llama8b"), steps=2):
    """The oracle as it stands, timed on this host: one decode step of each
    workload (its first teacher-forced step, on its seeded context) with one
    thread and with every host thread. Prints one JSON line."""
    from oracle import oracle as O
    from decode_megakernel_03_gb300 import synth
    out = {"kind": "oracle", "cores": O.default_threads(), "workloads": {}}
    for name in names:
        wl = synth.WORKLOADS[name]
        w = synth.make_weights(wl.shape, seed=wl.weight_seed)
        model = O.Model(wl.shape.as_dict(), synth.oracle_weights(w))
        del w
        kc, vc = synth.make_kv(wl.shape, wl.batch, wl.capacity, wl.ctx, seed=wl.kv_seed)
        ks = [synth.bits(t).copy() for t in kc]
        vs = [synth.bits(t).copy() for t in vc]
        toks = synth.step_tokens(wl)
        res = {}
        for threads in (1, O.default_threads()):
            dt = []
            for s in range(steps):
                t0 = time.perf_counter()
                model.decode_step(ks, vs, [int(t) for t in toks[s]], synth.step_positions(wl, s),
                                  nthreads=threads)
                dt.append(time.perf_counter() - t0)
            res[f"s_per_step_{threads}_threads"] = min(dt)
        res["tokens_per_s_all_threads"] = wl.batch / res[f"s_per_step_{O.default_threads()}_threads"]
        out["workloads"][name] = res
        print(name, res, file=sys.stderr, flush=True)
    print(json.dumps(out), flush=True)


def trace_summary(args, wl):
    """One decode step of the workload with the per-instruction trace on
    (mk_set_trace), summarised: per layer the time from its QKV's ready to the
    next layer's, per instruction kind the mean staging, compute, page-wait
    and publication times, the dependency hops (consumer ready - last
    producer published), and the LM head's span. Prints one JSON line."""
    import numpy as np
    import torch
    from decode_megakernel_03_gb300 import build as mkbuild
    from decode_megakernel_03_gb300 import mk, synth
    mkbuild.build()
    dev = torch.device("cuda")
    shape = wl.shape
    w = synth.make_weights(shape, seed=wl.weight_seed, device=dev)
    kc, vc = synth.make_kv(shape, wl.batch, wl.capacity, wl.ctx, seed=wl.kv_seed, device=dev)
    dec = mk.Decoder(shape, w, kc, vc, wl.batch)
    logits = torch.empty((wl.batch, shape.vocab), dtype=torch.float32, device=dev)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    tok = [int(t) for t in synth.step_tokens(wl)[0]]
    pos = synth.step_positions(wl, 0)
    ins, off, _ = mk.schedule(shape, wl.batch, wl.capacity, n_sm, pos)
    buf = torch.zeros(len(ins) * mk.TRACE_DTYPE.itemsize, dtype=torch.uint8, device=dev)
    for _ in range(5):
        dec.step(tok, pos, logits)
    dec.set_trace(buf)
    dec.step(tok, pos, logits)
    torch.cuda.synchronize()
    assert dec.status() == mk.MK_OK, dec.last_error()
    dec.set_trace(None)
    dec.close()
    rec = np.frombuffer(buf.cpu().numpy().tobytes(), dtype=mk.TRACE_DTYPE)
    t0 = rec["t_start"].min()
    us = lambda a: (a.astype(np.float64) - t0) / 1e3
    ts, tr, te, tst = us(rec["t_start"]), us(rec["t_ready"]), us(rec["t_end"]), us(rec["t_stored"])
    op, layer = rec["op"], rec["layer"]
    L = shape.n_layers
    ready = [float(tr[(layer == l) & (op == mk.OP_QKV)].min()) for l in range(L)]
    lm = op == mk.OP_LMHEAD
    ready.append(float(tr[lm].min()))
    out = {"workload": wl.name, "step_us": float(te.max()), "layer_us": np.diff(ready).round(2).tolist(),
           "lm_head_us": float(te[lm].max() - tr[lm].min()), "per_op": {}, "hops_us": {}}
    mid = (layer >= 2) & (layer < L - 2)
    for o, name in mk.OPS.items():
        m = (op == o) & (mid | (o == mk.OP_LMHEAD))
        if not m.any():
            continue
        out["per_op"][name] = {
            "n": int(m.sum()),
            "stage_us": float(rec["stage_ns"][m].mean() / 1e3),
            "ready_to_end_us": float(np.mean(te[m] - tr[m])),
            "page_wait_us": float(rec["page_wait_ns"][m].mean() / 1e3),
            "end_to_published_us": float(np.mean(tst[m] - te[m])),
            "idle_before_start_us": float(np.mean(tr[m] - ts[m])),
        }
    prod = {}
    for k in range(len(ins)):
        c = int(ins["sig_ctr"][k])
        if c >= 0:
            prod[c] = max(prod.get(c, -1e18), tst[k])
    hops = {}
    for k in range(len(ins)):
        c = int(ins["wait_ctr"][k])
        if c >= 0 and c in prod and mid[k]:
            hops.setdefault(mk.OPS[int(ins["op"][k])], []).append(tr[k] - prod[c])
    out["hops_us"] = {k: {"median": float(np.median(v)), "p90": float(np.percentile(v, 90))}
                      for k, v in hops.items()}
    out["copy_issue"] = copy_issue_profile(rec, ins, shape, wl, pos, tr)
    print(json.dumps(out), flush=True)


def copy_issue_profile(rec, ins, shape, wl, pos, tr):
    """How fast the loaders hand bytes to the memory system, from the trace's
    per-instruction copy issue windows: each instruction's bytes (weight rows,
    or an attention unit's cached K and V rows) spread evenly over its window
    [first copy issued, last copy issued] on its SM, summed over SMs in
    0.25 us bins. A loader issues a page only into a free ring slot, so while
    the rate stays below the HBM bandwidth the memory system has less work
    than it could do. Per middle layer (2 .. L-3), between its first QKV
    instruction's input and the next layer's: the mean rate over the
    attention chain (until the first gate/up instruction's input) and over
    the MLP, and the fraction of the layer's bins below half the measured
    HBM peak."""
    import numpy as np
    from decode_megakernel_03_gb300 import mk
    peak_gbs, _ = read_peaks()
    H, D, QD, F = shape.hidden, shape.head_dim, shape.n_heads * shape.head_dim, shape.ffn
    nbytes = np.zeros(len(rec))
    for k in range(len(rec)):
        op, a0, a1, a2 = int(ins["op"][k]), int(ins["a0"][k]), int(ins["a1"][k]), int(ins["a2"][k])
        items = a1 - a0
        if op == mk.OP_QKV or op == mk.OP_GATEUP:
            nbytes[k] = items * 2 * H * 2
        elif op == mk.OP_OPROJ:
            nbytes[k] = items * QD * 2
        elif op == mk.OP_DOWN:
            nbytes[k] = items * (F // 4) * 2
        elif op == mk.OP_LMHEAD:
            nbytes[k] = items * H * 2
        elif op == mk.OP_ATTN:
            p = pos[a0] + 1
            pidx, P = a2 >> 16, a2 & 0xFFFF
            keys = max(0, min((pidx + 1) * p // P, p - 1) - pidx * p // P)
            nbytes[k] = keys * D * 2 * 2
    t0 = rec["t_start"].min()
    f = (rec["t_issue_first"].astype(np.float64) - t0) / 1e3
    l_ = (rec["t_issue_last"].astype(np.float64) - t0) / 1e3
    ok = (nbytes > 0) & (rec["t_issue_first"] > 0) & (rec["t_issue_last"] >= rec["t_issue_first"])
    width = 0.25
    nb = int(np.ceil(l_[ok].max() / width)) + 2
    rate = np.zeros(nb)  # bytes per bin
    for a, b, n in zip(f[ok], l_[ok], nbytes[ok]):
        i0, i1 = int(a // width), int(b // width)
        rate[i0:i1 + 1] += n / (i1 - i0 + 1)
    gbs = rate / (width * 1e3)  # bytes per us / 1e3 = GB/s
    op, layer = rec["op"], rec["layer"]
    L = shape.n_layers
    res = []
    for l in range(2, L - 2):
        a = tr[(layer == l) & (op == mk.OP_QKV)].min()
        m = tr[(layer == l) & (op == mk.OP_GATEUP)].min()
        e = tr[(layer == l + 1) & (op == mk.OP_QKV)].min()
        ia, im, ie = int(a // width), int(m // width), int(e // width)
        res.append((gbs[ia:im].mean(), gbs[im:ie].mean(), float(np.mean(gbs[ia:ie] < peak_gbs / 2)),
                    m - a, e - m))
    r = np.array(res)
    return {"bin_us": width, "peak_gbs": peak_gbs,
            "attention_chain_us": float(r[:, 3].mean()), "mlp_us": float(r[:, 4].mean()),
            "attention_chain_issue_gbs": float(r[:, 0].mean()),
            "mlp_issue_gbs": float(r[:, 1].mean()),
            "layer_fraction_below_half_peak": float(r[:, 2].mean())}


def replica_env():
    """(world, rank, local rank) from the launcher's environment; one rank
    and no process group without torchrun."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's x. Replicas share no data, so the job
    advances at the pace of its slowest replica: its step time is the max
    of the ranks' step times. `device` holds the one-element reduction
    tensor (a CUDA device under NCCL, the CPU under gloo)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(batch: int, world: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every rank decodes `batch` sequences one token per
    step, and a step of the job takes the slowest rank's time."""
    return batch * world / (ms_per_step * 1e-3)


def rank_barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def run_reference(args, wl):
    _, rank, _ = replica_env()
    if rank != 0:
        return  # the reference arm runs on rank 0 alone
    from decode_megakernel_03_gb300 import synth
    w = synth.make_weights(wl.shape, seed=wl.weight_seed)
    w_host = synth.oracle_weights(w)
    del w
    from oracle import oracle as O
    model = O.Model(wl.shape.as_dict(), w_host)
    kc, vc = synth.make_kv(wl.shape, wl.batch, wl.capacity, wl.ctx, seed=wl.kv_seed)
    ks = [synth.bits(t).copy() for t in kc]
    vs = [synth.bits(t).copy() for t in vc]
    toks = synth.step_tokens(wl)
    threads = O.default_threads()
    for s in range(args.warmup):
        model.decode_step(ks, vs, [int(t) for t in toks[s % wl.steps]],
                          synth.step_positions(wl, s % wl.steps), nthreads=threads)
    times = []
    for s in range(args.steps):
        t0 = time.perf_counter()
        model.decode_step(ks, vs, [int(t) for t in toks[s % wl.steps]],
                          synth.step_positions(wl, s % wl.steps), nthreads=threads)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = wl.batch / (ms / 1e3)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": 0, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded random init, random KV context)",
        "config": {"workload": wl.name, "batch": wl.batch, "ctx": list(wl.ctx),
                   "l2": "inputs larger than L2"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{args.steps} decode steps of {wl.name} after {args.warmup} warm-up"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_gpu(args, wl):
    import torch
    import torch.distributed as dist
    from decode_megakernel_03_gb300 import build as mkbuild
    from decode_megakernel_03_gb300 import mk, synth

    world, rank, local = replica_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mkbuild.build()

    shape = wl.shape
    w = synth.make_weights(shape, seed=wl.weight_seed, device=dev)
    kc, vc = synth.make_kv(shape, wl.batch, wl.capacity, wl.ctx, seed=wl.kv_seed, device=dev)
    dec = mk.Decoder(shape, w, kc, vc, wl.batch)
    logits = torch.empty((wl.batch, shape.vocab), dtype=torch.float32, device=dev)
    toks = synth.step_tokens(wl)
    K, W = args.steps, args.warmup
    stream = torch.cuda.current_stream()

    def tok_pos(s):
        s = s % wl.steps
        return [int(t) for t in toks[s]], synth.step_positions(wl, s)

    def timed(mode):
        for s in range(W):
            t, p = tok_pos(s)
            if mode == "mega":
                dec.step(t, p, logits)
            else:
                dec.step_multilaunch(t, p, logits, graph=(mode == "graph"))
        torch.cuda.synchronize()
        rank_barrier(world)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        for s in range(K):
            t, p = tok_pos(s)
            ev[s][0].record(stream)
            if mode == "mega":
                dec.step(t, p, logits)
            else:
                dec.step_multilaunch(t, p, logits, graph=(mode == "graph"))
            ev[s][1].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t_wall
        rank_barrier(world)
        assert dec.status() == mk.MK_OK, dec.last_error()
        per = [a.elapsed_time(b) for a, b in ev]
        return per, wall

    with ClockSampler(local) as clk:
        per_mega, wall_mega = timed("mega")
    per_multi, _ = timed("multi")
    per_graph, _ = timed("graph")

    # end to end through the public call: host ids/positions in, logits read back
    host_logits = torch.empty((wl.batch, shape.vocab), dtype=torch.float32, pin_memory=True)
    for s in range(W):
        t, p = tok_pos(s)
        dec.step(t, p, logits)
        host_logits.copy_(logits, non_blocking=True)
    torch.cuda.synchronize()
    rank_barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for s in range(K):
        t, p = tok_pos(s)
        dec.step(t, p, logits)
        host_logits.copy_(logits, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    rank_barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / K, world, dev)

    # greedy decode through mk_decode_greedy: 16 steps per call, each next
    # token fed back on the device, the call's token ids read back to the host
    g_steps = 16
    g_calls = max(1, K // g_steps)
    tok_dev = torch.empty(g_steps * wl.batch, dtype=torch.int32, device=dev)
    tok_host = torch.empty(g_steps * wl.batch, dtype=torch.int32, pin_memory=True)
    t0_, p0_ = tok_pos(0)
    dec.decode_greedy(t0_, p0_, g_steps, tok_dev, logits)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(g_calls):
        dec.decode_greedy(t0_, p0_, g_steps, tok_dev, logits)
        tok_host.copy_(tok_dev, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    assert dec.status() == mk.MK_OK, dec.last_error()
    greedy_ms = e0.elapsed_time(e1) / (g_calls * g_steps)
    # the same 16 steps in one persistent launch per call
    dec.decode_greedy_persistent(t0_, p0_, g_steps, tok_dev, logits)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(g_calls):
        dec.decode_greedy_persistent(t0_, p0_, g_steps, tok_dev, logits)
        tok_host.copy_(tok_dev, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    assert dec.status() == mk.MK_OK, dec.last_error()
    greedy_one_ms = e0.elapsed_time(e1) / (g_calls * g_steps)
    # the same greedy decode as a host loop: one step per call, the logits read
    # back and their argmax taken on the host before the next call (what the
    # device-fed argmax removes), wall-clock tokens/s of 32 steps
    def host_loop(n):
        tk = [int(x) for x in t0_]
        for s_ in range(n):
            dec.step(tk, [q + s_ for q in p0_], logits)
            host = logits.cpu()
            tk = [int(i) for i in torch.argmax(host, dim=1)]
        return tk
    host_loop(4)
    torch.cuda.synchronize()
    t0w = time.perf_counter()
    host_loop(32)
    host_loop_tps = 32 * wl.batch / (time.perf_counter() - t0w)
    # one-launch greedy, 32 steps per call, tokens read back, wall clock
    tok32 = torch.empty(32 * wl.batch, dtype=torch.int32, device=dev)
    dec.decode_greedy_persistent(t0_, p0_, 32, tok32, logits)
    torch.cuda.synchronize()
    t0w = time.perf_counter()
    dec.decode_greedy_persistent(t0_, p0_, 32, tok32, logits)
    tok32.cpu()
    greedy32_tps = 32 * wl.batch / (time.perf_counter() - t0w)

    # the same steps on a paged KV cache: the caches' contents in pools of
    # 16-position blocks (and, second, 64-position blocks: one run per
    # 64-key page boundary instead of four) in shuffled order, a host block
    # table per step
    paged_ms = {}
    for bs in (16, 64):
        mb = wl.capacity // bs
        n_blocks = wl.batch * mb
        perm = torch.randperm(n_blocks, generator=torch.Generator().manual_seed(7))
        table = perm.view(wl.batch, mb).numpy().astype(np.int32)

        def to_pool(c):
            blocks = c[:, :, :mb * bs].reshape(wl.batch, shape.n_kv_heads, mb, bs, shape.head_dim)
            blocks = blocks.permute(0, 2, 1, 3, 4).reshape(n_blocks, shape.n_kv_heads, bs,
                                                           shape.head_dim)
            pool = torch.empty_like(blocks)
            pool[perm.to(dev)] = blocks
            return pool
        kp, vp = [to_pool(c) for c in kc], [to_pool(c) for c in vc]
        dp = mk.Decoder(shape, w, kp, vp, wl.batch, paged=(bs, n_blocks, mb * bs))
        for s in range(W):
            t, p = tok_pos(s)
            dp.step_paged(t, p, table, logits)
        torch.cuda.synchronize()
        e0.record(stream)
        for s in range(K):
            t, p = tok_pos(s)
            dp.step_paged(t, p, table, logits)
        e1.record(stream)
        torch.cuda.synchronize()
        assert dp.status() == mk.MK_OK, dp.last_error()
        paged_ms[bs] = e0.elapsed_time(e1) / K
        dp.close()
        del kp, vp

    # host side of a step (no device work timed): the C-ABI call with its plan
    # cached (argument checks, plan lookup, launch), and building a plan
    # (the host scheduler alone, what a plan miss adds before its upload)
    n_sm = torch.cuda.get_device_properties(local).multi_processor_count
    t, p = tok_pos(0)
    torch.cuda.synchronize()
    reps = 200
    t0h = time.perf_counter()
    for _ in range(reps):
        dec.step(t, p, logits)
    host_call_us = (time.perf_counter() - t0h) / reps * 1e6
    torch.cuda.synchronize()
    t0h = time.perf_counter()
    for _ in range(20):
        mk.schedule(shape, wl.batch, wl.capacity, n_sm, p)
    host_plan_us = (time.perf_counter() - t0h) / 20 * 1e6

    # prefill through mk_prefill: a 512-token prompt of this model in chunks of
    # 8 tokens (a batch-8 handle on its own cache), tokens/s
    prefill_tps = None
    if wl.batch == 1 and shape.name.startswith("llama-3.2-1b"):
        kp, vp = synth.empty_kv(shape, 8, 640, device=dev)
        dpre = mk.Decoder(shape, w, kp, vp, 8)
        plog = torch.empty(shape.vocab, dtype=torch.float32, device=dev)
        prompt = [int(x) for x in synth.make_tokens(shape.vocab, 512, seed=5)]
        dpre.prefill(prompt, 0, plog)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(3):
            dpre.prefill(prompt, 0, plog)
        e1.record(stream)
        torch.cuda.synchronize()
        assert dpre.status() == mk.MK_OK, dpre.last_error()
        prefill_tps = 512 * 3 / (e0.elapsed_time(e1) * 1e-3)
        dpre.close()
        del kp, vp

    ms = sum(per_mega) / K
    ms_all = max_over_ranks(ms, world, dev)

    positions = [synth.step_positions(wl, s % wl.steps) for s in range(K)]
    wb, kvb = zip(*[algorithmic_bytes(shape, wl.batch, p) for p in positions])
    bytes_step = (sum(wb) + sum(kvb)) / K
    peak, peak_kind = read_peaks()
    achieved = bytes_step / (ms * 1e-3) / 1e9
    t_min_ms = bytes_step / (peak * 1e9) * 1e3
    multi_ms = sum(per_multi) / K
    graph_ms = sum(per_graph) / K

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        w_host = synth.oracle_weights(w)
        rate, n, dt, cores = cpu_oracle_rate(wl, w_host)
        cpu = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} decode steps of {wl.name} ({dt:.1f} s, all host threads)"}

    traffic = recorded_traffic(wl.name)

    if rank == 0:
        clocks = clk.summary()
        line = {
            "metric": METRIC,
            "value": job_rate(wl.batch, world, ms_all),
            "unit": "tokens/s",
            "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": ms_all,
            "us_per_token": ms_all * 1e3 / wl.batch,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16 weights/KV, fp32 activations",
            "data": "synthetic (seeded random init weights, random bf16 KV context)",
            "config": {"workload": wl.name, "model": shape.name, "batch": wl.batch,
                       "ctx": list(wl.ctx), "positions": [positions[0][0], positions[-1][0]],
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2 (2.5 GB/step streamed), no flush"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind,
                         "algorithmic_bytes_per_step": bytes_step, "traffic": traffic,
                         "t_min_us": t_min_ms * 1e3},
            "cpu_baseline": cpu,
            "e2e": {"value": job_rate(wl.batch, world, e2e_ms), "unit": "tokens/s",
                    "h2d_bytes_per_step": 8 * wl.batch,
                    "d2h_bytes_per_step": 4 * wl.batch * shape.vocab},
            "gpu_launches": K,
            "clocks": clocks,
            "comparison": {
                "megakernel_us": ms * 1e3,
                "megakernel_p50_us": statistics.median(per_mega) * 1e3,
                "megakernel_p90_us": float(np.percentile(per_mega, 90)) * 1e3,
                "multilaunch_us": multi_ms * 1e3,
                "multilaunch_graph_us": graph_ms * 1e3,
                # per layer QKV, attention, (reduction,) O-projection, gate/up,
                # down; one sequence with at most 2048 attention columns has
                # no reduction instruction (the O-projection's staging reduces)
                "multilaunch_launches_per_step":
                    (5 if wl.batch == 1 and shape.n_heads * shape.head_dim <= 2048 else 6)
                    * shape.n_layers + 1,
                "recovered_overhead_vs_multilaunch": (multi_ms - ms) / (multi_ms - t_min_ms),
                "recovered_overhead_vs_graph": (graph_ms - ms) / (graph_ms - t_min_ms),
                "overhead_megakernel": (ms - t_min_ms) / ms,
                "overhead_multilaunch": (multi_ms - t_min_ms) / multi_ms,
                "wall_s_megakernel": wall_mega,
                "greedy_us_per_step": greedy_ms * 1e3,
                "greedy_steps_per_call": g_steps,
                "greedy_one_launch_us_per_step": greedy_one_ms * 1e3,
                "greedy_32_one_launch_tokens_per_s": greedy32_tps,
                "greedy_32_host_argmax_loop_tokens_per_s": host_loop_tps,
                "paged_kv_us_per_step": paged_ms[16] * 1e3,
                "paged_kv_block_size": 16,
                "paged_kv_64_us_per_step": paged_ms[64] * 1e3,
                "host_step_call_us": host_call_us,
                "host_plan_build_us": host_plan_us,
                "prefill_tokens_per_s": prefill_tps,
                "prefill_chunk": 8,
            },
        }
        print(json.dumps(line), flush=True)
    dec.close()
    if world > 1:
        dist.destroy_process_group()


def kernel_sources_sha1() -> str:
    """Hash of the CUDA/C++ sources of the decode kernel (any change to them
    invalidates DRAM counters captured earlier)."""
    import hashlib
    d = os.path.join(ROOT, "decode_megakernel_03_gb300", "csrc")
    h = hashlib.sha1()
    for f in sorted(os.listdir(d)):
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()


def recorded_traffic(workload: str):
    """dram__bytes_read.sum + dram__bytes_write.sum of one megakernel launch,
    from the ncu summary in profiles/, or None if it was taken on other
    kernel sources or another workload."""
    path = os.path.join(ROOT, "profiles", f"megakernel_{workload}_dram.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("kernel_sources_sha1") != kernel_sources_sha1():
        return None
    try:
        return float(kv["dram_bytes_read_per_launch"]) + float(kv["dram_bytes_write_per_launch"])
    except (KeyError, ValueError):
        return None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="mk", choices=["mk", "reference"])
    ap.add_argument("--workload", default="llama1b")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--trace", action="store_true",
                    help="summarise the per-instruction trace of one step of --workload")
    ap.add_argument("--oracle-timings", action="store_true",
                    help="time the CPU oracle (1 and all host threads) on tiny, 1B and 8B; no GPU")
    args = ap.parse_args()
    if args.oracle_timings:
        oracle_timings()
        return
    if args.trace:
        from decode_megakernel_03_gb300 import synth as _s
        trace_summary(args, _s.WORKLOADS[args.workload])
        return
    from decode_megakernel_03_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    if args.warmup < 3 and args.impl != "reference":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_gpu(args, wl)


if __name__ == "__main__":
    main()
