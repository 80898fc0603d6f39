"""Pins of the oracle's q/k L2 normalisation (the "q/k L2-norm" variant of the
K3 README's test-status table, row L3/L4) and of its backward, against
invariants and finite differences, and of the composed path the parity tests
use (normalise q and k, run the scan, map dq and dk back to the raw q, k).
CPU only."""
import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def test_rows_have_unit_norm_and_keep_their_direction():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 3, 16)) * rng.uniform(0.01, 30.0, (7, 3, 1))
    y = oracle.l2norm(x)
    assert y.shape == x.shape
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), 1.0, rtol=0, atol=1e-14)
    # parallel and same sign: <y, x> = |x|, and the component orthogonal to x vanishes
    dots = np.sum(y * x, axis=-1)
    np.testing.assert_allclose(dots, np.linalg.norm(x, axis=-1), rtol=1e-13)
    perp = y - (dots / np.sum(x * x, axis=-1))[..., None] * x
    assert np.abs(perp).max() < 1e-14


def test_scale_and_sign():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 8))
    y = oracle.l2norm(x)
    np.testing.assert_allclose(oracle.l2norm(3.7 * x), y, rtol=0, atol=1e-15)
    np.testing.assert_allclose(oracle.l2norm(-x), -y, rtol=0, atol=1e-15)
    unit = np.eye(8)[:5]
    np.testing.assert_array_equal(oracle.l2norm(unit), unit)


def test_zero_row_maps_to_zero_and_the_floor_applies():
    x = np.zeros((2, 4))
    x[1, 2] = 1e-14           # norm below the floor 1e-12: divided by the floor
    y = oracle.l2norm(x)
    assert np.all(y[0] == 0.0)
    np.testing.assert_allclose(y[1, 2], 1e-14 / 1e-12, rtol=1e-15)


def test_backward_matches_finite_differences():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 6)) * 2.0
    w = rng.standard_normal((4, 6))
    dx = oracle.l2norm_bwd(x, w)
    eps = 1e-6
    fd = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += eps
        xm[idx] -= eps
        fd[idx] = (np.sum(w * oracle.l2norm(xp)) - np.sum(w * oracle.l2norm(xm))) / (2 * eps)
    np.testing.assert_allclose(dx, fd, rtol=0, atol=1e-8)


def test_backward_is_orthogonal_to_the_row_and_kills_radial_gradients():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((6, 10))
    dy = rng.standard_normal((6, 10))
    dx = oracle.l2norm_bwd(x, dy)
    assert np.abs(np.sum(dx * x, axis=-1)).max() < 1e-12
    # a gradient along the output itself changes nothing (the norm is fixed)
    np.testing.assert_allclose(oracle.l2norm_bwd(x, 2.5 * oracle.l2norm(x)), 0.0, atol=1e-14)


def _composed_loss(q, k, v, g, beta, s0, do, dht):
    o, ht = oracle.fwd_recurrent(oracle.l2norm(q), oracle.l2norm(k), v, g, beta, h0=s0)
    return float(np.sum(o * do) + np.sum(ht * dht))


@pytest.mark.parametrize("H,HV", [(2, 2), (1, 2)])
def test_normalise_then_scan_gradients_match_finite_differences(H, HV):
    """dq, dk of the scan on normalised inputs, mapped back with l2norm_bwd
    (after the GVA group sum), against central differences in the raw q, k."""
    rng = np.random.default_rng(5 + H)
    B, T, K, V = 1, 4, 6, 5
    q = rng.standard_normal((B, T, H, K)) * 1.5
    k = rng.standard_normal((B, T, H, K)) * 0.7
    v = rng.standard_normal((B, T, HV, V))
    g = -np.log1p(np.exp(rng.standard_normal((B, T, HV, K))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, HV))))
    s0 = 0.3 * rng.standard_normal((B, HV, K, V))
    do = rng.standard_normal((B, T, HV, V))
    dht = rng.standard_normal((B, HV, K, V))
    gr = oracle.bwd_recurrent(oracle.l2norm(q), oracle.l2norm(k), v, g, beta, do, h0=s0, dht=dht)
    dq = oracle.l2norm_bwd(q, gr["dq"])
    dk = oracle.l2norm_bwd(k, gr["dk"])
    eps = 1e-6
    for x, ref, name in ((q, dq, "dq"), (k, dk, "dk")):
        fd = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + eps
            lp = _composed_loss(q, k, v, g, beta, s0, do, dht)
            x[idx] = old - eps
            lm = _composed_loss(q, k, v, g, beta, s0, do, dht)
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(ref, fd, rtol=0, atol=1e-6, err_msg=name)
