"""Pins of the oracle's whole decode step.

Special weights reduce the step to closed forms built from the single ops
pinned in test_oracle_pins.py, so that each wiring choice of the decoder
(which kv-head a q-head reads, which cache slots attention covers, the residual
adds, gate vs up, per-layer weight indexing, the tied LM head) is checked by a
case in which a plausible mistake changes the answer. The last tests compare
incremental decoding through the KV cache with a full causal recompute.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from decode_megakernel_03_gb300 import synth

SMALL = dict(n_layers=1, hidden=128, n_heads=4, n_kv_heads=2, head_dim=32, ffn=64, vocab=50,
             tied=False, rms_eps=1e-5, rope_theta=10000.0)


def _b(a):
    t = torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _rand(rng, *shape, std=0.3):
    return _b(rng.standard_normal(shape) * std)


def _weights(cfg, rng, **over):
    H, D, F, V = cfg["hidden"], cfg["head_dim"], cfg["ffn"], cfg["vocab"]
    nh, nkv, L = cfg["n_heads"], cfg["n_kv_heads"], cfg["n_layers"]
    w = {
        "embed": _rand(rng, V, H, std=1.0),
        "lm_head": _rand(rng, V, H),
        "final_norm": _b(1 + 0.1 * rng.standard_normal(H)),
        "attn_norm": [_b(1 + 0.1 * rng.standard_normal(H)) for _ in range(L)],
        "wq": [_rand(rng, nh * D, H) for _ in range(L)],
        "wk": [_rand(rng, nkv * D, H) for _ in range(L)],
        "wv": [_rand(rng, nkv * D, H) for _ in range(L)],
        "wo": [_rand(rng, H, nh * D) for _ in range(L)],
        "mlp_norm": [_b(1 + 0.1 * rng.standard_normal(H)) for _ in range(L)],
        "wgate": [_rand(rng, F, H) for _ in range(L)],
        "wup": [_rand(rng, F, H) for _ in range(L)],
        "wdown": [_rand(rng, H, F) for _ in range(L)],
    }
    w.update(over)
    return w


def _zeros(*shape):
    return np.zeros(shape, dtype=np.uint16)  # bf16 +0.0


def _cache(cfg, B, S, rng, fill_after=None):
    shp = (B, cfg["n_kv_heads"], S, cfg["head_dim"])
    ks = [_rand(rng, *shp, std=1.0) for _ in range(cfg["n_layers"])]
    vs = [_rand(rng, *shp, std=1.0) for _ in range(cfg["n_layers"])]
    return ks, vs


def _f(bits):
    return O.bf16_to_f64(bits)


def test_attention_wiring_gqa_range_and_residual():
    """Wq = Wk = 0 makes every score 0, so each q-head's output is the plain mean
    of its kv-head's values over slots 0..pos. Wo = I and a zero MLP then make
    x = embed + attn, so the logits expose the mapping h -> h / (nh/nkv), the
    inclusive range, the freshly written slot and the residual add."""
    cfg = dict(SMALL)
    rng = np.random.default_rng(20)
    H, D, nh, nkv = cfg["hidden"], cfg["head_dim"], cfg["n_heads"], cfg["n_kv_heads"]
    eye = _b(np.eye(H))
    w = _weights(cfg, rng, wq=[_zeros(nh * D, H)], wk=[_zeros(nkv * D, H)], wo=[eye],
                 wgate=[_zeros(cfg["ffn"], H)], wup=[_zeros(cfg["ffn"], H)])
    m = O.Model(cfg, w)
    B, S = 2, 16
    ks, vs = _cache(cfg, B, S, rng)
    # slots after pos hold huge values: reading one of them would swamp the mean
    pos = [5, 11]
    for b in range(B):
        vs[0][b, :, pos[b] + 1:, :] = _b(np.full((nkv, S - pos[b] - 1, D), 3.0e4))
    v_before = vs[0].copy()
    k_before = ks[0].copy()
    tok = [7, 42]
    logits = m.decode_step(ks, vs, tok, pos, nthreads=2)

    for b in range(B):
        e = _f(w["embed"][tok[b]])
        n = O.rmsnorm(e, w["attn_norm"][0], cfg["rms_eps"])
        v_new = O.f64_to_bf16(O.matvec(w["wv"][0], n))
        # the new slot holds bf16(v); k = RoPE(0) = 0
        for g in range(nkv):
            np.testing.assert_array_equal(vs[0][b, g, pos[b]], v_new[g * D:(g + 1) * D])
            np.testing.assert_array_equal(_f(ks[0][b, g, pos[b]]), np.zeros(D))
        # every other slot is untouched
        mask = np.ones(S, bool)
        mask[pos[b]] = False
        np.testing.assert_array_equal(vs[0][b][:, mask], v_before[b][:, mask])
        np.testing.assert_array_equal(ks[0][b][:, mask], k_before[b][:, mask])
        attn = np.zeros(nh * D)
        for h in range(nh):
            g = h // (nh // nkv)
            attn[h * D:(h + 1) * D] = _f(vs[0][b, g, :pos[b] + 1]).mean(axis=0)
        x = e + attn
        want = O.matvec(w["lm_head"], O.rmsnorm(x, w["final_norm"], cfg["rms_eps"]))
        np.testing.assert_allclose(logits[b], want, rtol=1e-10, atol=1e-10)


def test_mlp_wiring_gate_up_down_and_layer_order():
    """With Wv = 0 and a zero value cache the attention output is 0, so each
    layer adds only Wd (SiLU(Wg n) * Wu n) with n = RMSNorm(x, mlp_norm[l]).
    Two layers with different weights pin the layer order and indexing."""
    cfg = dict(SMALL, n_layers=2)
    rng = np.random.default_rng(21)
    H, D, nkv = cfg["hidden"], cfg["head_dim"], cfg["n_kv_heads"]
    w = _weights(cfg, rng, wv=[_zeros(nkv * D, H)] * 2)
    m = O.Model(cfg, w)
    B, S = 1, 8
    shp = (B, nkv, S, D)
    ks = [_rand(rng, *shp, std=1.0) for _ in range(2)]
    vs = [_zeros(*shp) for _ in range(2)]
    tok, pos = [3], [4]
    logits = m.decode_step(ks, vs, tok, pos, nthreads=1)
    x = _f(w["embed"][3])
    for l in range(2):
        n = O.rmsnorm(x, w["mlp_norm"][l], cfg["rms_eps"])
        g = O.matvec(w["wgate"][l], n)
        u = O.matvec(w["wup"][l], n)
        h = np.array([O.silu(a) for a in g]) * u
        x = x + O.matvec(w["wdown"][l], h)
    want = O.matvec(w["lm_head"], O.rmsnorm(x, w["final_norm"], cfg["rms_eps"]))
    np.testing.assert_allclose(logits[0], want, rtol=1e-10, atol=1e-10)


def test_tied_head_is_embedding():
    cfg = dict(SMALL)
    rng = np.random.default_rng(22)
    w = _weights(cfg, rng)
    w_untied = dict(w, lm_head=w["embed"].copy())
    w_tied = dict(w, lm_head=None)
    B, S = 1, 8
    ks, vs = _cache(cfg, B, S, rng)
    a = O.Model(cfg, w_untied).decode_step([k.copy() for k in ks], [v.copy() for v in vs], [9], [3])
    b = O.Model(dict(cfg, tied=True), w_tied).decode_step(ks, vs, [9], [3])
    np.testing.assert_array_equal(a, b)


def test_batch_rows_are_independent():
    cfg = dict(SMALL, n_layers=2)
    rng = np.random.default_rng(23)
    m = O.Model(cfg, _weights(cfg, rng))
    B, S = 3, 12
    ks, vs = _cache(cfg, B, S, rng)
    tok, pos = [1, 2, 3], [0, 7, 11]
    ks2, vs2 = [k.copy() for k in ks], [v.copy() for v in vs]
    both = m.decode_step(ks, vs, tok, pos)
    for b in range(B):
        kb = [np.ascontiguousarray(k[b:b + 1]) for k in ks2]
        vb = [np.ascontiguousarray(v[b:b + 1]) for v in vs2]
        one = m.decode_step(kb, vb, [tok[b]], [pos[b]])
        np.testing.assert_array_equal(one[0], both[b])
        for l in range(2):
            np.testing.assert_array_equal(kb[l][0], ks[l][b])


def test_rejects_bad_inputs():
    cfg = dict(SMALL)
    rng = np.random.default_rng(24)
    m = O.Model(cfg, _weights(cfg, rng))
    ks, vs = _cache(cfg, 1, 8, rng)
    with pytest.raises(ValueError):
        m.decode_step(ks, vs, [cfg["vocab"]], [0])
    with pytest.raises(ValueError):
        m.decode_step(ks, vs, [0], [8])


def _tiny_model():
    shape = synth.TINY
    w = synth.oracle_weights(synth.make_weights(shape, seed=0))
    return O.Model(shape.as_dict(), w), shape


def test_incremental_decode_equals_full_recompute():
    """Decoding 80 tokens one at a time through the KV cache gives the same
    logits and cache contents as one causal forward over all 80 tokens."""
    m, shape = _tiny_model()
    n = 80
    toks = synth.make_tokens(shape.vocab, n, seed=5).numpy()
    full, kf, vf = m.forward_full(toks, want_kv=True)
    ks = [np.zeros((1, shape.n_kv_heads, 96, shape.head_dim), np.uint16)
          for _ in range(shape.n_layers)]
    vs = [k.copy() for k in ks]
    for t in range(n):
        lg = m.decode_step(ks, vs, [int(toks[t])], [t])
        np.testing.assert_allclose(lg[0], full[t], rtol=1e-12, atol=1e-12)
    for l in range(shape.n_layers):
        np.testing.assert_array_equal(ks[l][0, :, :n], kf[l])
        np.testing.assert_array_equal(vs[l][0, :, :n], vf[l])
        assert not ks[l][0, :, n:].any()


def test_logit_scale_is_sane():
    # random init keeps activations O(1): the norms hold the scale, the logits
    # have a spread well above fp32 rounding (so top-1 comparisons are meaningful)
    m, shape = _tiny_model()
    toks = synth.make_tokens(shape.vocab, 4, seed=6).numpy()
    lg = m.forward_full(toks)
    assert np.all(np.isfinite(lg))
    sd = lg.std(axis=1)
    assert np.all(sd > 0.05) and np.all(sd < 50)


def _composed_step(cfg, w, ks, vs, tok, pos):
    """One decode step of one sequence written out from the single ops pinned
    in test_oracle_pins.py, in the order of the seven fused instructions
    ("3 · L'interpréteur sur GPU", §3.2): attention scale 1/sqrt(head_dim),
    rotate-half RoPE on every q-head and every k-head at the absolute
    position, k/v rounded to bf16 through fp32 before they enter the cache,
    q-head h reading kv-head h // (n_heads / n_kv_heads) over slots 0..pos."""
    H, D, nh, nkv = cfg["hidden"], cfg["head_dim"], cfg["n_heads"], cfg["n_kv_heads"]
    group, eps, theta = nh // nkv, cfg["rms_eps"], cfg["rope_theta"]
    x = _f(w["embed"][tok])
    for l in range(cfg["n_layers"]):
        n = O.rmsnorm(x, w["attn_norm"][l], eps)
        q = O.matvec(w["wq"][l], n)
        k = O.matvec(w["wk"][l], n)
        v = O.matvec(w["wv"][l], n)
        q = np.concatenate([O.rope(q[h * D:(h + 1) * D], pos, theta) for h in range(nh)])
        k = np.concatenate([O.rope(k[h * D:(h + 1) * D], pos, theta) for h in range(nkv)])
        for h in range(nkv):
            ks[l][0, h, pos] = _b(k[h * D:(h + 1) * D].astype(np.float32))
            vs[l][0, h, pos] = _b(v[h * D:(h + 1) * D].astype(np.float32))
        att = np.concatenate([
            O.attend(q[h * D:(h + 1) * D], ks[l][0, h // group, :pos + 1],
                     vs[l][0, h // group, :pos + 1], 1.0 / np.sqrt(D)) for h in range(nh)])
        x = x + O.matvec(w["wo"][l], att)
        n = O.rmsnorm(x, w["mlp_norm"][l], eps)
        g = O.matvec(w["wgate"][l], n)
        u = O.matvec(w["wup"][l], n)
        hh = np.array([O.silu(z) for z in g]) * u
        x = x + O.matvec(w["wdown"][l], hh)
    lm = w["embed"] if cfg["tied"] else w["lm_head"]
    return O.matvec(lm, O.rmsnorm(x, w["final_norm"], eps))


@pytest.mark.parametrize("tied", [False, True])
def test_decode_step_equals_composition_of_pinned_ops(tied):
    """Two layers with every weight random (Wq and Wk included, so the scores,
    their 1/sqrt(head_dim) scale and the rotation of q AND k all matter): the
    whole decode step equals its composition from the individually pinned
    ops at several positions, including slot 0 and the last slot. A wrong
    scale (1/sqrt(hidden), none), k left unrotated, a wrong GQA mapping or a
    wrong slot range would all change these logits."""
    cfg = dict(SMALL, n_layers=2, tied=tied)
    rng = np.random.default_rng(31)
    w = _weights(cfg, rng)
    m = O.Model(cfg, w)
    S = 12
    for pos in (0, 5, S - 1):
        ks, vs = _cache(cfg, 1, S, rng)
        ks2 = [k.copy() for k in ks]
        vs2 = [v.copy() for v in vs]
        tok = int(rng.integers(cfg["vocab"]))
        got = m.decode_step(ks, vs, [tok], [pos], nthreads=1)[0]
        want = _composed_step(cfg, w, ks2, vs2, tok, pos)
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
        for a, b in zip(ks + vs, ks2 + vs2):
            np.testing.assert_array_equal(a, b)
        # the scores are far from zero: the test is sensitive to the scale
        assert np.std(want) > 1e-3


def test_composition_detects_a_wrong_attention_scale():
    """The composed reference is sensitive to what it pins: with the scale
    1/sqrt(hidden) instead of 1/sqrt(head_dim) its logits move well past the
    comparison tolerance above."""
    cfg = dict(SMALL, n_layers=1)
    rng = np.random.default_rng(32)
    w = _weights(cfg, rng)
    S, pos = 12, 9
    ks, vs = _cache(cfg, 1, S, rng)
    tok = 7
    good = _composed_step(cfg, w, [k.copy() for k in ks], [v.copy() for v in vs], tok, pos)
    real_attend = O.attend
    try:
        O.attend = lambda q, K, V, scale: real_attend(q, K, V, 1.0 / np.sqrt(cfg["hidden"]))
        bad = _composed_step(cfg, w, [k.copy() for k in ks], [v.copy() for v in vs], tok, pos)
    finally:
        O.attend = real_attend
    assert np.max(np.abs(good - bad)) > 1e-3
