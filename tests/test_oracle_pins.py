"""Pins of the oracle's single operations to things other than itself.

Each op is checked against hand-derived closed forms (tests/golden), invariants
that the textbook definitions imply, special cases that reduce to a library
routine, and brute force on tiny inputs. The cases are picked so that a dropped
term, a wrong sign, a swapped pair index or a wrong exponent fails one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.txt")


def _bits_of(vals):
    t = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _golden_cases():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            op, inp, exp = [p.strip() for p in line.split("|")]
            fields = {}
            for part in inp.split(";"):
                toks = part.split()
                fields[toks[0]] = [float(t) for t in toks[1:]]
            cases.append((op, fields, [float(t) for t in exp.split()]))
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c[0])
def test_golden_closed_forms(case):
    op, f, expected = case
    if op == "rmsnorm":
        got = O.rmsnorm(f["x"], _bits_of(f["w"]), f["eps"][0])
    elif op == "rope":
        got = O.rope(f["v"], int(f["pos"][0]), f["theta"][0])
    elif op == "silu":
        got = [O.silu(f["z"][0])]
    elif op == "attend":
        q = np.array(f["q"])
        d = q.size
        K = _bits_of(f["k"]).reshape(-1, d)
        V = _bits_of(f["v"]).reshape(-1, d)
        got = O.attend(q, K, V, 1.0 / math.sqrt(d))
    elif op == "bf16":
        got = [int(O.f64_to_bf16([f["v"][0]])[0])]
        assert got == [int(expected[0])]
        return
    else:
        raise AssertionError(op)
    np.testing.assert_allclose(got, expected, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------- bf16

def test_bf16_widening_exact():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 65536, 5000, dtype=np.uint32).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # finite only
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    lib = O.lib()
    got = np.array([lib.ref_bf16_to_f64(int(b)) for b in bits])
    np.testing.assert_array_equal(got, t)


def test_bf16_rounding_matches_library():
    # torch's fp32 -> bf16 conversion rounds to nearest even: an independent routine
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(3000) * 10 ** rng.uniform(-6, 6, 3000),
                        [0.0, -0.0, 1e-40, 3.0e38]])
    v32 = v.astype(np.float32)
    want = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.f64_to_bf16(v32.astype(np.float64))
    np.testing.assert_array_equal(got, want)


# ----------------------------------------------------------------- RMSNorm

def test_rmsnorm_constant_vector():
    rng = np.random.default_rng(2)
    for c in (-3.5, 0.125, 7.0):
        w = _bits_of(rng.standard_normal(96))
        wf = O.bf16_to_f64(w)
        eps = 1e-5
        got = O.rmsnorm(np.full(96, c), w, eps)
        np.testing.assert_allclose(got, wf * c / math.sqrt(c * c + eps), rtol=1e-13)


def test_rmsnorm_scale_invariance_and_unit_rms():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(256)
    ones = _bits_of(np.ones(256))
    a = O.rmsnorm(x, ones, 0.0)
    b = O.rmsnorm(x * 37.25, ones, 0.0)
    np.testing.assert_allclose(a, b, rtol=1e-13)
    assert abs(np.sqrt(np.mean(a * a)) - 1.0) < 1e-13


# ----------------------------------------------------------------- RoPE

def test_rope_identity_at_zero():
    rng = np.random.default_rng(4)
    v = rng.standard_normal(128)
    np.testing.assert_array_equal(O.rope(v, 0, 500000.0), v)


def test_rope_preserves_pair_norms():
    rng = np.random.default_rng(5)
    D = 64
    v = rng.standard_normal(D)
    r = O.rope(v, 1234, 10000.0)
    h = D // 2
    np.testing.assert_allclose(r[:h] ** 2 + r[h:] ** 2, v[:h] ** 2 + v[h:] ** 2, rtol=1e-12)


def test_rope_relative_position():
    # <R_m q, R_n k> depends only on m - n
    rng = np.random.default_rng(6)
    D = 64
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    ref = np.dot(O.rope(q, 17, 10000.0), O.rope(k, 5, 10000.0))
    for m, n in ((112, 100), (4012, 4000), (12, 0)):
        np.testing.assert_allclose(np.dot(O.rope(q, m, 10000.0), O.rope(k, n, 10000.0)), ref,
                                   rtol=1e-9)


def test_rope_frequency_of_each_pair():
    # pair i turns at rate theta^(-2i/D): after pos steps the angle of pair i is pos*rate
    D, theta, pos = 16, 500000.0, 3
    for i in range(D // 2):
        v = np.zeros(D)
        v[i] = 1.0
        r = O.rope(v, pos, theta)
        ang = math.atan2(r[i + D // 2], r[i])
        want = math.remainder(pos * theta ** (-2.0 * i / D), 2 * math.pi)
        assert abs(ang - want) < 1e-12


# ----------------------------------------------------------------- SiLU

def test_silu_limits():
    assert O.silu(0.0) == 0.0
    assert abs(O.silu(40.0) - 40.0) < 1e-12
    assert abs(O.silu(-40.0)) < 1e-15
    # SiLU(z) - SiLU(-z) = z  (since sigma(z) + sigma(-z) = 1)
    for z in (0.3, 1.7, 5.0):
        assert abs(O.silu(z) - O.silu(-z) - z) < 1e-14


# ----------------------------------------------------------------- matvec

def test_matvec_brute_force():
    rng = np.random.default_rng(7)
    for rows, cols in ((1, 1), (3, 5), (17, 64), (64, 33)):
        W = _bits_of(rng.standard_normal((rows, cols)).ravel()).reshape(rows, cols)
        x = rng.standard_normal(cols)
        Wf = O.bf16_to_f64(W)
        want = np.array([sum(Wf[r, c] * x[c] for c in range(cols)) for r in range(rows)])
        for nt in (1, 3):
            np.testing.assert_allclose(O.matvec(W, x, nt), want, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(O.matvec(W, x), Wf @ x, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------- attention

def test_attend_single_key_returns_value():
    rng = np.random.default_rng(8)
    D = 64
    K = _bits_of(rng.standard_normal(D)).reshape(1, D)
    V = _bits_of(rng.standard_normal(D)).reshape(1, D)
    out = O.attend(rng.standard_normal(D) * 10, K, V, 0.125)
    np.testing.assert_array_equal(out, O.bf16_to_f64(V[0]))


def test_attend_equal_keys_average_values():
    rng = np.random.default_rng(9)
    D, n = 64, 37
    k = _bits_of(rng.standard_normal(D))
    K = np.tile(k, (n, 1))
    V = _bits_of(rng.standard_normal(n * D)).reshape(n, D)
    out = O.attend(rng.standard_normal(D), K, V, 0.125)
    np.testing.assert_allclose(out, O.bf16_to_f64(V).mean(axis=0), rtol=1e-12, atol=1e-14)


def test_attend_matches_library_softmax():
    from scipy.special import softmax
    rng = np.random.default_rng(10)
    D, n = 64, 50
    K = _bits_of(rng.standard_normal(n * D)).reshape(n, D)
    V = _bits_of(rng.standard_normal(n * D)).reshape(n, D)
    q = rng.standard_normal(D) * 3
    Kf, Vf = O.bf16_to_f64(K), O.bf16_to_f64(V)
    p = softmax(Kf @ q * 0.125)
    assert abs(p.sum() - 1.0) < 1e-12
    np.testing.assert_allclose(O.attend(q, K, V, 0.125), p @ Vf, rtol=1e-11, atol=1e-13)


def test_attend_split_combine_equals_single_pass():
    # the split-KV algebra the GPU uses: partial (o_p, m_p, l_p) over disjoint key
    # ranges combine to the unsplit result
    rng = np.random.default_rng(11)
    D, n = 64, 90
    K = _bits_of(rng.standard_normal(n * D)).reshape(n, D)
    V = _bits_of(rng.standard_normal(n * D)).reshape(n, D)
    q = rng.standard_normal(D)
    full = O.attend(q, K, V, 0.125)
    parts = []
    for a, b in ((0, 31), (31, 64), (64, 90)):
        s = O.bf16_to_f64(K[a:b]) @ q * 0.125
        m = s.max()
        e = np.exp(s - m)
        parts.append((e @ O.bf16_to_f64(V[a:b]), m, e.sum()))
        # each part is itself the oracle's attention over its range, times l
        np.testing.assert_allclose(parts[-1][0] / parts[-1][2], O.attend(q, K[a:b], V[a:b], 0.125),
                                   rtol=1e-11, atol=1e-13)
    M = max(p[1] for p in parts)
    num = sum(np.exp(p[1] - M) * p[0] for p in parts)
    den = sum(np.exp(p[1] - M) * p[2] for p in parts)
    np.testing.assert_allclose(num / den, full, rtol=1e-11, atol=1e-13)
