"""Helpers shared by the GPU parity tests: build the CUDA decoder and the CPU
oracle from the same seeded inputs, and compare their logits with the
tolerances the decode path is held to (per step: relative L2 error <= 1e-2,
max-abs error <= 5e-2; top-1 agreement >= 99% over a run)."""
from __future__ import annotations

import numpy as np
import torch

from decode_megakernel_03_gb300 import build as mkbuild
from decode_megakernel_03_gb300 import mk, synth
from oracle import oracle as O

REL_L2 = 1e-2
MAX_ABS = 5e-2
TOP1 = 0.99
# one bf16 ulp relative (8 significant bits), plus a small absolute floor:
# the kernel rounds its fp32 k/v, the oracle rounds fp32(its fp64 k/v)
KV_RTOL = 2.0 ** -7
KV_ATOL = 1e-3


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


class Pair:
    """A GPU decoder and an oracle model over identical weights and caches."""

    def __init__(self, shape, batch, capacity, ctx=None, weight_seed=0, kv_seed=1,
                 kv_from_oracle=None):
        mkbuild.build()
        self.shape, self.batch, self.capacity = shape, batch, capacity
        dev = torch.device("cuda")
        self.w = synth.make_weights(shape, seed=weight_seed, device=dev)
        self.model = O.Model(shape.as_dict(), synth.oracle_weights(self.w))
        if kv_from_oracle is not None:
            ks, vs = kv_from_oracle
            self.kc = [torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).to(dev) for k in ks]
            self.vc = [torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).to(dev) for v in vs]
        elif ctx is not None:
            self.kc, self.vc = synth.make_kv(shape, batch, capacity, ctx, seed=kv_seed, device=dev)
        else:
            self.kc, self.vc = synth.empty_kv(shape, batch, capacity, device=dev)
        self.ok = [bf16_bits(t).copy() for t in self.kc]
        self.ov = [bf16_bits(t).copy() for t in self.vc]
        self.dec = mk.Decoder(shape, self.w, self.kc, self.vc, batch)
        self.logits = torch.empty((batch, shape.vocab), dtype=torch.float32, device=dev)

    def gpu_step(self, tok, pos, mode="mega"):
        if mode == "mega":
            self.dec.step(tok, pos, self.logits)
        elif mode == "multi":
            self.dec.step_multilaunch(tok, pos, self.logits, graph=False)
        else:
            self.dec.step_multilaunch(tok, pos, self.logits, graph=True)
        rc = self.dec.status()
        assert rc == mk.MK_OK, self.dec.last_error()
        return self.logits.cpu().numpy().astype(np.float64)

    def oracle_step(self, tok, pos):
        return self.model.decode_step(self.ok, self.ov, tok, pos)

    def close(self):
        self.dec.close()


def compare_logits(got: np.ndarray, want: np.ndarray):
    """Per-sequence relative L2 and max-abs error, and top-1 agreement taken
    in fp32 on both sides (the kernel's precision)."""
    out = []
    for b in range(want.shape[0]):
        g, w = got[b], want[b]
        rel = float(np.linalg.norm(g - w) / np.linalg.norm(w))
        mab = float(np.max(np.abs(g - w)))
        w32 = w.astype(np.float32)
        t_got, t_want = int(np.argmax(got[b].astype(np.float32))), int(np.argmax(w32))
        srt = np.sort(w32)
        margin = float(srt[-1] - srt[-2])
        out.append(dict(rel_l2=rel, max_abs=mab, top1=t_got == t_want, margin=margin))
    return out


class Tally:
    def __init__(self):
        self.rows = []

    def add(self, stats):
        self.rows.extend(stats)

    def check(self):
        """Every step within the rel-L2 and max-abs bounds, and top-1
        agreement of at least 99 % over the run. The oracle's top-1/top-2
        margin of every disagreement is reported, not excused."""
        assert self.rows
        worst_rel = max(r["rel_l2"] for r in self.rows)
        worst_abs = max(r["max_abs"] for r in self.rows)
        agree = sum(r["top1"] for r in self.rows) / len(self.rows)
        misses = [r["margin"] for r in self.rows if not r["top1"]]
        assert worst_rel <= REL_L2, f"rel-L2 {worst_rel}"
        assert worst_abs <= MAX_ABS, f"max-abs {worst_abs}"
        assert agree >= TOP1, f"top-1 agreement {agree} over {len(self.rows)} steps, margins {misses}"
        return dict(rel_l2=worst_rel, max_abs=worst_abs, top1=agree, n=len(self.rows),
                    miss_margins=misses)


def check_kv_step(pair: Pair, pos, before_k, before_v):
    """Bit-exact: every slot except positions[b] is unchanged; the written slot
    agrees with the oracle's within one bf16 ulp."""
    for l in range(pair.shape.n_layers):
        gk, gv = bf16_bits(pair.kc[l]), bf16_bits(pair.vc[l])
        for b, p in enumerate(pos):
            mask = np.ones(pair.capacity, bool)
            mask[p] = False
            np.testing.assert_array_equal(gk[b][:, mask], before_k[l][b][:, mask])
            np.testing.assert_array_equal(gv[b][:, mask], before_v[l][b][:, mask])
            np.testing.assert_allclose(bits_to_f64(gk[b][:, p]), bits_to_f64(pair.ok[l][b][:, p]),
                                       rtol=KV_RTOL, atol=KV_ATOL)
            np.testing.assert_allclose(bits_to_f64(gv[b][:, p]), bits_to_f64(pair.ov[l][b][:, p]),
                                       rtol=KV_RTOL, atol=KV_ATOL)


def written_rows(pair: Pair, pos):
    """The k and v rows this step wrote (slot positions[b] of every layer and
    sequence) on the GPU, as bf16 bits [L][B][nkv][D]; a small gather."""
    ks = np.stack([np.stack([bf16_bits(pair.kc[l][b, :, p]) for b, p in enumerate(pos)])
                   for l in range(pair.shape.n_layers)])
    vs = np.stack([np.stack([bf16_bits(pair.vc[l][b, :, p]) for b, p in enumerate(pos)])
                   for l in range(pair.shape.n_layers)])
    return ks, vs


def check_written_rows(pair: Pair, pos):
    """The slot each step writes agrees with the oracle's within one bf16 ulp
    (the oracle has appended its own row at the same slot)."""
    gk, gv = written_rows(pair, pos)
    for l in range(pair.shape.n_layers):
        for b, p in enumerate(pos):
            np.testing.assert_allclose(bits_to_f64(gk[l][b]), bits_to_f64(pair.ok[l][b][:, p]),
                                       rtol=KV_RTOL, atol=KV_ATOL)
            np.testing.assert_allclose(bits_to_f64(gv[l][b]), bits_to_f64(pair.ov[l][b][:, p]),
                                       rtol=KV_RTOL, atol=KV_ATOL)


def check_untouched(pair: Pair, before_k, before_v, written):
    """Bit-exact: after a run, every slot that no step wrote still holds its
    initial bits. written: per sequence, the set of positions the run wrote."""
    for l in range(pair.shape.n_layers):
        gk, gv = bf16_bits(pair.kc[l]), bf16_bits(pair.vc[l])
        for b in range(pair.batch):
            mask = np.ones(pair.capacity, bool)
            mask[sorted(written[b])] = False
            np.testing.assert_array_equal(gk[b][:, mask], before_k[l][b][:, mask])
            np.testing.assert_array_equal(gv[b][:, mask], before_v[l][b][:, mask])


def counters_match(pair: Pair, pos):
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    _, _, targets = mk.schedule(pair.shape, pair.batch, pair.capacity, n_sm, pos)
    got = pair.dec.counters()
    np.testing.assert_array_equal(got, targets)
