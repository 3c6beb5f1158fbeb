"""Pins of the oracle's HQQ zero-point refinement against things other than
its own formulas (River-LLM explainer, section 六: HQQ is the exit layers'
default quantizer; it needs no calibration data).

* the shrinkage at p = 1 is the proximal operator of |.| (soft threshold),
  checked against a numerical minimiser of |y| + beta/2 (y - x)^2;
* the zero-point step is the least-squares minimiser of its objective,
  checked against a numerical minimiser;
* with beta = infinity (no shrinkage) the iteration stands still: min-max's
  zero and codes come back unchanged;
* groups on an exact grid come back exactly;
* on random bf16 weights no group's lp error exceeds min-max's, and the
  whole tensor's lp, L1 and L2 errors are lower;
* planted mistakes (a sign in the zero step, no shrinkage) are caught.
"""
import numpy as np
import pytest
from scipy.optimize import minimize_scalar

import oracle.quant as oq
from oracle.quant import (dequantize_linear, hqq_shrink, hqq_zero_step, quantize_linear,
                          quantize_linear_hqq, unpack_nibbles)


def _random_bf16(rng, N, K, std=0.02):
    torch = pytest.importorskip("torch")
    w = torch.from_numpy(rng.standard_normal((N, K)).astype(np.float32) * std)
    return w.to(torch.bfloat16).float().numpy()


@pytest.mark.parametrize("beta", [0.5, 3.0, 40.0])
def test_shrink_at_p1_is_the_proximal_operator_of_abs(beta):
    xs = np.array([-2.0, -0.7, -0.2, -0.01, 0.0, 0.03, 0.25, 0.6, 1.5])
    got = hqq_shrink(xs, beta, 1.0)
    for x, g in zip(xs, got):
        r = minimize_scalar(lambda y: abs(y) + 0.5 * beta * (y - x) ** 2, bounds=(-3, 3),
                            method="bounded", options={"xatol": 1e-12})
        assert abs(r.x - g) < 1e-6, (x, g, r.x)


def test_shrink_below_p1_keeps_sign_and_shrinks():
    xs = np.linspace(-0.05, 0.05, 41)
    y = hqq_shrink(xs, 10.0, 0.7)
    assert np.all(np.abs(y) <= np.abs(xs))
    assert np.all((y == 0) | (np.sign(y) == np.sign(xs)))
    assert hqq_shrink(np.array([0.0]), 10.0, 0.7)[0] == 0.0


def test_zero_step_is_the_least_squares_minimiser():
    rng = np.random.default_rng(3)
    n = 128
    w = rng.standard_normal(n) * 0.02
    s = 0.004
    q = np.clip(np.rint(w / s + 7.3), 0, 15)
    e = rng.standard_normal(n) * 1e-3
    mask = np.ones(n, bool)
    z = hqq_zero_step(w[None], q[None], e[None], np.array([s]), mask[None])[0]
    r = minimize_scalar(lambda zz: np.sum((q - zz - (w - e) / s) ** 2), bounds=(-20, 40),
                        method="bounded", options={"xatol": 1e-12})
    assert abs(z - r.x) < 1e-6
    # a ragged group: only the valid entries count
    mask[100:] = False
    z2 = hqq_zero_step(w[None], q[None], e[None], np.array([s]), mask[None])[0]
    r2 = minimize_scalar(lambda zz: np.sum((q[:100] - zz - (w[:100] - e[:100]) / s) ** 2),
                         bounds=(-20, 40), method="bounded", options={"xatol": 1e-12})
    assert abs(z2 - r2.x) < 1e-6


def test_no_shrinkage_leaves_min_max_unchanged():
    rng = np.random.default_rng(4)
    w = _random_bf16(rng, 16, 384)
    a = quantize_linear(w)
    b = quantize_linear_hqq(w, beta=np.inf)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_grid_aligned_groups_come_back_exactly():
    rng = np.random.default_rng(5)
    N, K, G = 6, 384, 128
    s = np.float32(2.0 ** -6)
    zint = rng.integers(0, 16, size=(N, K // G))
    q = rng.integers(0, 16, size=(N, K))
    q[:, ::G] = 0
    q[:, 1::G] = 15
    w = ((q - np.repeat(zint, G, axis=1)).astype(np.float32) * s).astype(np.float32)
    qw, sc, zz = quantize_linear_hqq(w, G)
    assert np.array_equal(zz.astype(np.float32), zint.astype(np.float32))
    assert np.array_equal(unpack_nibbles(qw, K), q.astype(np.uint8))
    assert np.array_equal(dequantize_linear(qw, sc, zz, K, G), w)


def _errors(w, qw, s, z, K):
    r = (w - dequantize_linear(qw, s, z, K)).astype(np.float64)
    return np.sum(np.abs(r) ** 0.7), np.abs(r).mean(), np.sqrt((r ** 2).mean())


def _group_lp(w, qw, s, z, K, G=128):
    r = np.abs((w - dequantize_linear(qw, s, z, K)).astype(np.float64)) ** 0.7
    pad = np.zeros((w.shape[0], s.shape[1] * G))
    pad[:, :K] = r
    return pad.reshape(w.shape[0], -1, G).sum(-1)


@pytest.mark.parametrize("K", [1024, 688])
def test_refinement_never_worse_per_group_and_better_overall(K):
    rng = np.random.default_rng(6)
    w = _random_bf16(rng, 96, K)
    a = quantize_linear(w)
    b = quantize_linear_hqq(w)
    assert np.array_equal(a[1], b[1]), "the scales are min-max's"
    ga, gb = _group_lp(w, *a, K), _group_lp(w, *b, K)
    assert np.all(gb <= ga * (1 + 1e-12))
    assert np.mean(gb < ga) > 0.3
    ea, eb = _errors(w, *a, K), _errors(w, *b, K)
    assert eb[0] < 0.99 * ea[0] and eb[1] < ea[1] and eb[2] < ea[2], (ea, eb)


def _trajectory(w, K):
    """Total lp error of min-max and of each iteration's zero point (no selection)."""
    _, s16, z16 = quantize_linear(w)
    wg, mask = oq._groups(w, 128, s16.shape[1])
    errs = [oq._lp_error(wg, s16.astype(np.float32), z16, mask, 0.7).sum()]
    for zc in oq.hqq_iterates(wg, s16, z16, mask):
        errs.append(oq._lp_error(wg, s16.astype(np.float32), zc, mask, 0.7).sum())
    return np.array(errs)


def test_iterations_descend():
    """Without the selection of the best zero, the iterations themselves lower
    the tensor's lp error step by step."""
    rng = np.random.default_rng(6)
    w = _random_bf16(rng, 64, 1024)
    e = _trajectory(w, 1024)
    assert e[-1] < 0.99 * e[0]
    assert np.all(np.diff(e) <= 1e-3 * e[0]), e


def test_planted_mistakes_are_caught(monkeypatch):
    rng = np.random.default_rng(6)
    w = _random_bf16(rng, 64, 1024)

    def flipped(w_, q, e, s, mask):
        v = np.where(mask, q + (w_ - e) / s[..., None], 0.0)
        return v.sum(axis=-1) / mask.sum(axis=-1)

    for name, fn in (("hqq_zero_step", flipped), ("hqq_shrink", lambda x, b, p: np.asarray(x, float))):
        with monkeypatch.context() as mp:
            mp.setattr(oq, name, fn)
            e = _trajectory(w, 1024)
        assert not (e[-1] < 0.99 * e[0] and np.all(np.diff(e) <= 1e-3 * e[0])), \
            f"mutation {name} not caught"
