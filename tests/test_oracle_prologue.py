"""Pins for the oracle's q/k/v prologue ("Chasing speed of light on TPU v6e",
section "The Long Tail": the q/k/v RMS norms and RoPE run right before
attention).  Each pin comes from the mathematics, not from the oracle's own
code: RMS norm closed forms and scale invariance; RoPE as multiplication of
the complex numbers y_i + i y_{i+D/2} by e^{i a} (numpy complex arithmetic);
rotation preserves each pair's length; position 0 and theta <= 0 are the
identity; the dot product of a rotated query and key depends only on the
difference of their positions.  Planted mistakes (interleaved pairs, a flipped
sign, a wrong frequency exponent, a sum instead of a mean, eps outside the
root) each fail at least one pin.
"""

from __future__ import annotations

import numpy as np
import pytest

import oracle


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- pins


def pin_norm_closed_forms(norm):
    ok = True
    # A constant row c * 1 normalises to sign(c) * 1 (eps = 0).
    for c in (3.0, -0.25, 1e4):
        y = norm(np.full((1, 16), c), np.ones(16), 0.0)
        ok &= np.allclose(y, np.sign(c), rtol=1e-12, atol=0)
    # [3, 4]: mean square 12.5.
    y = norm(np.array([[3.0, 4.0]]), np.ones(2), 0.0)
    ok &= np.allclose(y, np.array([[3.0, 4.0]]) / np.sqrt(12.5), rtol=1e-12, atol=0)
    # eps: a zero row stays zero; eps = mean square halves the square.
    ok &= np.all(norm(np.zeros((1, 8)), np.ones(8), 1e-6) == 0.0)
    y = norm(np.array([[1.0, 1.0, 1.0, 1.0]]), np.ones(4), 1.0)
    ok &= np.allclose(y, 1.0 / np.sqrt(2.0), rtol=1e-12, atol=0)
    # The weight scales each dimension.
    w = np.arange(1.0, 9.0)
    x = _rng(1).normal(size=(3, 8))
    ok &= np.allclose(norm(x, w, 0.0), norm(x, np.ones(8), 0.0) * w, rtol=1e-12, atol=0)
    return bool(ok)


def pin_norm_invariants(norm):
    x = _rng(2).normal(size=(50, 64))
    y = norm(x, np.ones(64), 0.0)
    ok = np.allclose(np.mean(y * y, axis=-1), 1.0, rtol=1e-12, atol=0)
    ok &= np.allclose(norm(7.5 * x, np.ones(64), 0.0), y, rtol=1e-12, atol=0)
    return bool(ok)


def pin_rope_complex(rope):
    """rope == multiplication by e^{i pos theta^(-2j/D)} of z_j = y_j + i y_{j+D/2}."""
    rng = _rng(3)
    ok = True
    for D, theta in ((4, 100.0), (64, 10000.0), (256, 1e6)):
        n = 7
        y = rng.normal(size=(n, 3, D))
        pos = rng.integers(0, 1 << 20, size=n)
        z = y[..., : D // 2] + 1j * y[..., D // 2:]
        j = np.arange(D // 2)
        a = pos[:, None].astype(np.float64) * theta ** (-2.0 * j / D)
        w = z * np.exp(1j * a)[:, None, :]
        want = np.concatenate([w.real, w.imag], axis=-1)
        ok &= np.allclose(rope(y, pos, theta), want, rtol=0, atol=1e-9)
    return bool(ok)


def pin_rope_worked_example(rope):
    """D = 4, theta = 100: frequencies 1 and 1/10; y = (1, 2, 3, 4) at
    position 2 turns the pair (1, 3) by 2 rad and (2, 4) by 0.2 rad."""
    got = rope(np.array([[1.0, 2.0, 3.0, 4.0]]), np.array([2]), 100.0)[0]
    c2, s2, c02, s02 = np.cos(2.0), np.sin(2.0), np.cos(0.2), np.sin(0.2)
    want = np.array([c2 - 3 * s2, 2 * c02 - 4 * s02, 3 * c2 + s2, 4 * c02 + 2 * s02])
    return bool(np.allclose(got, want, rtol=0, atol=1e-12))


def pin_rope_identities(rope):
    rng = _rng(4)
    y = rng.normal(size=(5, 2, 32))
    ok = np.allclose(rope(y, np.zeros(5, dtype=np.int64), 10000.0), y, rtol=0, atol=0)
    ok &= np.allclose(rope(y, np.arange(5) * 1000, 0.0), y, rtol=0, atol=0)
    # Each pair keeps its length.
    out = rope(y, rng.integers(0, 100000, size=5), 10000.0)
    ok &= np.allclose(out[..., :16] ** 2 + out[..., 16:] ** 2,
                      y[..., :16] ** 2 + y[..., 16:] ** 2, rtol=1e-12, atol=0)
    return bool(ok)


def pin_rope_relative(rope):
    """<rope(q, m), rope(k, n)> depends on m - n only."""
    rng = _rng(5)
    D = 64
    q = rng.normal(size=(1, 1, D))
    k = rng.normal(size=(1, 1, D))
    ok = True
    for m, n, shift in ((10, 3, 1000), (0, 500, 77), (123456, 123000, 99999)):
        d0 = np.sum(rope(q, np.array([m]), 10000.0) * rope(k, np.array([n]), 10000.0))
        d1 = np.sum(rope(q, np.array([m + shift]), 10000.0) *
                    rope(k, np.array([n + shift]), 10000.0))
        ok &= abs(d0 - d1) <= 1e-9 * max(1.0, abs(d0))
    # ... and does change with m - n.
    d2 = np.sum(rope(q, np.array([11]), 10000.0) * rope(k, np.array([3]), 10000.0))
    d0 = np.sum(rope(q, np.array([10]), 10000.0) * rope(k, np.array([3]), 10000.0))
    ok &= abs(d2 - d0) > 1e-6
    return bool(ok)


NORM_PINS = [pin_norm_closed_forms, pin_norm_invariants]
ROPE_PINS = [pin_rope_complex, pin_rope_worked_example, pin_rope_identities, pin_rope_relative]


@pytest.mark.parametrize("pin", NORM_PINS, ids=lambda f: f.__name__)
def test_rms_norm_pins(pin):
    assert pin(oracle.rms_norm)


@pytest.mark.parametrize("pin", ROPE_PINS, ids=lambda f: f.__name__)
def test_rope_pins(pin):
    assert pin(oracle.rope)


def test_token_positions():
    # Sequence 0: 3 new tokens ending at length 5; sequence 1: 1 token, length 1.
    assert list(oracle.token_positions([0, 3, 4], [5, 1])) == [2, 3, 4, 0]


def test_prologue_composes_norm_then_rope():
    rng = _rng(6)
    T, hq, hkv, D = 6, 4, 2, 32
    q, k, v = (rng.normal(size=(T, h, D)) for h in (hq, hkv, hkv))
    wq, wk, wv = (rng.uniform(0.5, 1.5, size=D) for _ in range(3))
    cu, kl = [0, 4, 6], [10, 2]
    qo, ko, vo = oracle.qkv_prologue(q, k, v, wq, wk, wv, 1e-6, 10000.0, cu, kl)
    pos = np.array([6, 7, 8, 9, 0, 1])
    # Position-wise: the same row rotated at its own position.
    for t in range(T):
        want = oracle.rope(oracle.rms_norm(q[t:t + 1], wq, 1e-6), pos[t:t + 1], 10000.0)
        assert np.allclose(qo[t:t + 1], want, rtol=0, atol=0)
    assert np.allclose(vo, oracle.rms_norm(v, wv, 1e-6), rtol=0, atol=0)
    # No norm weights: rotation only; no v weight: v unchanged.
    qo2, _, vo2 = oracle.qkv_prologue(q, k, v, None, None, None, 1e-6, 10000.0, cu, kl)
    assert np.allclose(qo2, oracle.rope(q, pos, 10000.0), rtol=0, atol=0)
    assert np.array_equal(vo2, v)


# ---------------------------------------------------------------- mutants


def _mut_rope(kind):
    def rope(y, pos, theta):
        y = np.asarray(y, dtype=np.float64)
        if theta <= 0:
            return y.copy()
        D = y.shape[-1]
        i = np.arange(D // 2, dtype=np.float64)
        expo = (-i / D) if kind == "exponent" else (-2.0 * i / D)
        a = np.asarray(pos, dtype=np.float64)[:, None] * float(theta) ** expo[None, :]
        shape = (a.shape[0],) + (1,) * (y.ndim - 2) + (D // 2,)
        c, s = np.cos(a).reshape(shape), np.sin(a).reshape(shape)
        if kind == "interleaved":
            lo, hi = y[..., 0::2], y[..., 1::2]
            out = np.empty_like(y)
            out[..., 0::2] = lo * c - hi * s
            out[..., 1::2] = hi * c + lo * s
            return out
        lo, hi = y[..., : D // 2], y[..., D // 2:]
        if kind == "sign":
            return np.concatenate([lo * c + hi * s, hi * c - lo * s], axis=-1)
        return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)
    return rope


def _mut_norm(kind):
    def norm(x, w, eps):
        x = np.asarray(x, dtype=np.float64)
        if kind == "sum":
            r = 1.0 / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)
        else:  # eps outside the root
            r = 1.0 / (np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + eps)
        return x * r * np.asarray(w, dtype=np.float64)
    return norm


@pytest.mark.parametrize("kind", ["interleaved", "sign", "exponent"])
def test_rope_pins_catch_planted_mistakes(kind):
    assert not all(pin(_mut_rope(kind)) for pin in ROPE_PINS)


@pytest.mark.parametrize("kind", ["sum", "eps_outside"])
def test_norm_pins_catch_planted_mistakes(kind):
    assert not all(pin(_mut_norm(kind)) for pin in NORM_PINS)
