"""Pins of the float64 oracle against facts fixed outside the oracle itself.

Each test checks one oracle function against something the pages or plain
mathematics fix: closed forms, invariants of the delta rule, agreement of two
independently written forms (token loop vs chunk form), and finite
differences for the backward.  The sources are the K3 README ("KDA 训练 → 推理
手写实现") table 实现路线表 (rows L1, L2, L6), its table 关键约束 / 风险点 (GVA,
scale, clamp at -5) and the "KDA CUDA Trainer" README section on the mixing
module (decay, then delta write, then the query reads the updated state).
"""
import numpy as np
import pytest

import oracle

rng_global = np.random.default_rng(1234)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def rand_inputs(B=2, T=16, H=2, HV=4, K=8, V=8, seed=0, g_lo=None, h0=True):
    rng = np.random.default_rng(seed)
    q = _unit(rng.standard_normal((B, T, H, K)))
    k = _unit(rng.standard_normal((B, T, H, K)))
    v = rng.standard_normal((B, T, HV, V))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, HV))))
    g = -np.log1p(np.exp(rng.standard_normal((B, T, HV, K)) * 2.0))
    if g_lo is not None:
        g = np.maximum(g, g_lo)
    s0 = 0.3 * rng.standard_normal((B, HV, K, V)) if h0 else None
    return q, k, v, g, beta, s0


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------

def test_beta_zero_leaves_decayed_initial_state():
    """beta = 0: no write, so S_T = diag(exp(sum_t max(g_t,-5))) S_0 and
    o_t = scale q_t^T diag(exp(G_t)) S_0 (K3 row L1 with the -5 clamp)."""
    q, k, v, g, beta, s0 = rand_inputs(T=12, seed=1)
    g = g * 3.0  # push some gates below -5 so the clamp is exercised
    assert (g < -5).any()
    beta = np.zeros_like(beta)
    B, T, H, K = q.shape
    HV, V = v.shape[2], v.shape[3]
    scale = K ** -0.5
    ghat = np.maximum(g, -5.0)
    Gcum = np.cumsum(ghat, axis=1)  # [B,T,HV,K]
    o_ref = np.zeros((B, T, HV, V))
    for b in range(B):
        for hv in range(HV):
            h = hv // (HV // H)
            for t in range(T):
                o_ref[b, t, hv] = scale * (q[b, t, h] * np.exp(Gcum[b, t, hv])) @ s0[b, hv]
    ht_ref = np.exp(Gcum[:, -1])[..., None] * s0
    for fn in (lambda: oracle.fwd_recurrent(q, k, v, g, beta, h0=s0),
               lambda: oracle.fwd_chunked(q, k, v, g, beta, chunk=4, h0=s0)):
        o, ht = fn()
        np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
        np.testing.assert_allclose(ht, ht_ref, rtol=0, atol=1e-13)


def test_g_zero_beta_zero_is_plain_readout():
    q, k, v, g, beta, s0 = rand_inputs(T=8, seed=2)
    o, ht = oracle.fwd_recurrent(q, k, v, np.zeros_like(g), np.zeros_like(beta), h0=s0)
    K = q.shape[-1]
    G = v.shape[2] // q.shape[2]
    qr = np.repeat(q, G, axis=2)
    o_ref = K ** -0.5 * np.einsum("btvk,bvkj->btvj", qr, s0)
    np.testing.assert_allclose(o, o_ref, atol=1e-13)
    np.testing.assert_allclose(ht, s0, atol=0)


def test_orthonormal_keys_are_written_exactly():
    """g = 0, beta = 1 and orthonormal keys k_1..k_T (T = K): the delta rule
    stores every value exactly, k_i^T S_T = v_i^T, whatever S_0 was."""
    rng = np.random.default_rng(3)
    K = V = 8
    T = 8
    Q, _ = np.linalg.qr(rng.standard_normal((K, K)))
    k = Q.T.reshape(1, T, 1, K)            # rows are orthonormal
    q = _unit(rng.standard_normal((1, T, 1, K)))
    v = rng.standard_normal((1, T, 1, V))
    s0 = rng.standard_normal((1, 1, K, V))
    _, ht = oracle.fwd_recurrent(q, k, v, np.zeros((1, T, 1, K)), np.ones((1, T, 1)), h0=s0)
    np.testing.assert_allclose(k[0, :, 0] @ ht[0, 0], v[0, :, 0], atol=1e-12)


def test_unit_key_reads_decayed_state_and_query_reads_updated_state():
    """With beta_t = 1 and a unit key the write makes k_t^T S_t = v_t exactly,
    for ANY gate -- but only if the key reads the DECAYED state (decay, then
    delta write).  With q_t = k_t and scale 1, the query must read the
    UPDATED state, so o_t = v_t (KDA CUDA Trainer README, mixing module)."""
    q, k, v, g, beta, s0 = rand_inputs(B=1, T=10, H=1, HV=1, K=6, V=5, seed=4)
    g = g - 0.5  # strong, nonzero decay
    o, _ = oracle.fwd_recurrent(k, k, v, g, np.ones_like(beta), scale=1.0, h0=s0)
    np.testing.assert_allclose(o, v, atol=1e-12)
    o2, _ = oracle.fwd_chunked(k, k, v, g, np.ones_like(beta), chunk=4, scale=1.0, h0=s0)
    np.testing.assert_allclose(o2, v, atol=1e-12)


def test_scalar_two_token_closed_form():
    """K = V = 1, T = 2, written out by hand:
    s1 = a1 s0 + b1 k1 (v1 - k1 a1 s0), o1 = c q1 s1, likewise for token 2."""
    s0, c = 0.7, 0.9
    q1, k1, v1, g1, b1 = 0.3, -1.2, 0.5, -0.4, 0.6
    q2, k2, v2, g2, b2 = -0.8, 0.9, -1.5, -7.0, 0.25   # g2 < -5: clamped
    a1, a2 = np.exp(g1), np.exp(-5.0)
    s1 = a1 * s0 + b1 * k1 * (v1 - k1 * a1 * s0)
    s2 = a2 * s1 + b2 * k2 * (v2 - k2 * a2 * s1)
    o_ref = np.array([c * q1 * s1, c * q2 * s2])
    arr = lambda a, b_: np.array([a, b_]).reshape(1, 2, 1, 1)
    o, ht = oracle.fwd_recurrent(arr(q1, q2), arr(k1, k2), arr(v1, v2), arr(g1, g2),
                                 np.array([b1, b2]).reshape(1, 2, 1), scale=c,
                                 h0=np.full((1, 1, 1, 1), s0))
    np.testing.assert_allclose(o.ravel(), o_ref, atol=1e-15)
    np.testing.assert_allclose(ht.ravel(), [s2], atol=1e-15)


# --------------------------------------------------------------------------
# Two independent forms and invariants
# --------------------------------------------------------------------------

@pytest.mark.parametrize("chunk", [1, 4, 16, 64])
@pytest.mark.parametrize("T", [64, 37])
def test_chunk_form_equals_token_loop(chunk, T):
    """K3 row L2 (cumsum, triangular system, solve, state passing) reaches the
    row-L1 recurrence exactly; chunk 1 is the recurrence itself."""
    q, k, v, g, beta, s0 = rand_inputs(B=2, T=T, H=2, HV=4, K=8, V=6, seed=5)
    g = g * 2.5  # include clamped gates and long pairwise decays
    o_r, ht_r = oracle.fwd_recurrent(q, k, v, g, beta, h0=s0)
    o_c, ht_c = oracle.fwd_chunked(q, k, v, g, beta, chunk=chunk, h0=s0)
    np.testing.assert_allclose(o_c, o_r, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ht_c, ht_r, rtol=0, atol=1e-12)


def test_decode_steps_equal_token_loop():
    """64 single-token steps on a [B,HV,K,V] state equal the T = 64 scan
    (K3 row L6 checked token by token against row L1)."""
    q, k, v, g, beta, s0 = rand_inputs(B=3, T=64, H=2, HV=4, K=8, V=8, seed=6)
    o_ref, ht_ref = oracle.fwd_recurrent(q, k, v, g, beta, h0=s0)
    state = s0.copy()
    for t in range(64):
        o_t = oracle.step(q[:, t], k[:, t], v[:, t], g[:, t], beta[:, t], state)
        np.testing.assert_allclose(o_t, o_ref[:, t], atol=1e-12)
    np.testing.assert_allclose(state, ht_ref, atol=1e-12)


def test_gva_equals_explicit_repeat():
    """GVA: value head hv uses key head hv // G (repeat_interleave order), and
    dq/dk are the group sums of the per-value-head gradients."""
    q, k, v, g, beta, s0 = rand_inputs(B=2, T=16, H=2, HV=4, K=8, V=8, seed=7)
    G = 2
    qr, kr = np.repeat(q, G, axis=2), np.repeat(k, G, axis=2)
    o1, h1 = oracle.fwd_recurrent(q, k, v, g, beta, h0=s0)
    o2, h2 = oracle.fwd_recurrent(qr, kr, v, g, beta, h0=s0)
    np.testing.assert_allclose(o1, o2, atol=1e-14)
    np.testing.assert_allclose(h1, h2, atol=1e-14)
    do = np.random.default_rng(8).standard_normal(o1.shape)
    g1 = oracle.bwd_recurrent(q, k, v, g, beta, do, h0=s0)
    g2 = oracle.bwd_recurrent(qr, kr, v, g, beta, do, h0=s0)
    B, T, H, K = q.shape
    np.testing.assert_allclose(g1["dq"], g2["dq"].reshape(B, T, H, G, K).sum(3), atol=1e-13)
    np.testing.assert_allclose(g1["dk"], g2["dk"].reshape(B, T, H, G, K).sum(3), atol=1e-13)
    for n in ("dv", "dg", "dbeta", "dh0"):
        np.testing.assert_allclose(g1[n], g2[n], atol=1e-13)


def test_jointly_linear_in_values_and_initial_state():
    q, k, v, g, beta, s0 = rand_inputs(T=20, seed=9)
    _, _, v2, _, _, s02 = rand_inputs(T=20, seed=10)
    al = -1.7
    oa, ha = oracle.fwd_recurrent(q, k, al * v + v2, g, beta, h0=al * s0 + s02)
    o1, h1 = oracle.fwd_recurrent(q, k, v, g, beta, h0=s0)
    o2, h2 = oracle.fwd_recurrent(q, k, v2, g, beta, h0=s02)
    np.testing.assert_allclose(oa, al * o1 + o2, atol=1e-12)
    np.testing.assert_allclose(ha, al * h1 + h2, atol=1e-12)


def test_state_chaining():
    q, k, v, g, beta, s0 = rand_inputs(T=24, seed=11)
    o, ht = oracle.fwd_recurrent(q, k, v, g, beta, h0=s0)
    a = slice(0, 10)
    b_ = slice(10, 24)
    oa, ha = oracle.fwd_recurrent(q[:, a], k[:, a], v[:, a], g[:, a], beta[:, a], h0=s0)
    ob, hb = oracle.fwd_chunked(q[:, b_], k[:, b_], v[:, b_], g[:, b_], beta[:, b_],
                                chunk=4, h0=ha)
    np.testing.assert_allclose(np.concatenate([oa, ob], 1), o, atol=1e-12)
    np.testing.assert_allclose(hb, ht, atol=1e-12)


def test_identity_padding_leaves_state():
    q, k, v, g, beta, s0 = rand_inputs(T=8, seed=12)
    _, ht = oracle.fwd_recurrent(q, k, v, g, beta, h0=s0)
    pad = lambda x, val: np.concatenate([x, np.full_like(x, val)], axis=1)
    _, ht2 = oracle.fwd_chunked(pad(q, 0.1), pad(k, 0.2), pad(v, 0.3), pad(g, 0.0),
                                pad(beta, 0.0), chunk=4, h0=s0)
    np.testing.assert_allclose(ht2, ht, atol=1e-13)


def test_value_columns_are_independent():
    """Columns of S evolve independently: running V in slices equals running
    it whole (the basis for splitting V across thread blocks)."""
    q, k, v, g, beta, s0 = rand_inputs(T=16, V=8, seed=13)
    o, ht = oracle.fwd_chunked(q, k, v, g, beta, chunk=8, h0=s0)
    for sl in (slice(0, 3), slice(3, 8)):
        o_s, h_s = oracle.fwd_recurrent(q, k, v[..., sl], g, beta, h0=s0[..., sl])
        np.testing.assert_allclose(o_s, o[..., sl], atol=1e-12)
        np.testing.assert_allclose(h_s, ht[..., sl], atol=1e-12)


def test_wy_quantities():
    """Step (3) of K3 row L2: T = (I + A)^{-1} with A strictly lower, so
    T = sum_{m<n} (-A)^m (A is nilpotent), W = T diag(beta) (k o exp(G)),
    U = T diag(beta) v; and A, Aqk match their element definitions."""
    rng = np.random.default_rng(14)
    n, K, V = 16, 8, 5
    k = _unit(rng.standard_normal((n, K)))
    qs = 0.5 * _unit(rng.standard_normal((n, K)))
    v = rng.standard_normal((n, V))
    g = -np.log1p(np.exp(2 * rng.standard_normal((n, K))))
    beta = rng.uniform(0.1, 0.9, n)
    w = oracle.chunk_wy(qs, k, v, g, beta)
    A, Tm = w["A"], w["T"]
    assert np.all(np.triu(A) == 0)
    np.testing.assert_allclose((np.eye(n) + A) @ Tm, np.eye(n), atol=1e-12)
    series = sum(np.linalg.matrix_power(-A, m) for m in range(n))
    np.testing.assert_allclose(Tm, series, atol=1e-12)
    G = np.cumsum(np.maximum(g, -5), axis=0)
    np.testing.assert_allclose(w["G"], G, atol=1e-14)
    np.testing.assert_allclose(w["W"], Tm @ (beta[:, None] * k * np.exp(G)), atol=1e-12)
    np.testing.assert_allclose(w["U"], Tm @ (beta[:, None] * v), atol=1e-12)
    i, j, c = 9, 4, slice(None)
    np.testing.assert_allclose(A[i, j], beta[i] * np.sum(k[i] * k[j] * np.exp(G[i] - G[j])),
                               atol=1e-14)
    np.testing.assert_allclose(w["Aqk"][i, i], np.sum(qs[i] * k[i]), atol=1e-14)
    assert w["Aqk"][3, 5] == 0.0


# --------------------------------------------------------------------------
# Backward: finite differences (K3 gradcheck settings: float64, eps 1e-6,
# atol 1e-4) and a directional (adjoint) check at longer T
# --------------------------------------------------------------------------

def _loss(inp, do, dht, scale=None):
    q, k, v, g, beta, s0 = inp
    o, ht = oracle.fwd_recurrent(q, k, v, g, beta, scale=scale, h0=s0)
    return float(np.sum(o * do) + np.sum(ht * dht))


def _away_from_kink(g, rng):
    bad = np.abs(g + 5.0) < 1e-3
    while bad.any():
        g[bad] = -np.log1p(np.exp(2 * rng.standard_normal(bad.sum())))
        bad = np.abs(g + 5.0) < 1e-3
    return g


@pytest.mark.parametrize("T,H,HV", [(4, 2, 4), (16, 2, 4), (16, 4, 4)])
def test_backward_matches_finite_differences(T, H, HV):
    rng = np.random.default_rng(15 + T + H)
    inp = list(rand_inputs(B=2, T=T, H=H, HV=HV, K=8, V=8, seed=16 + T + H))
    inp[3] = _away_from_kink(inp[3] * 2.5, rng)   # some gates below -5, none at it
    q, k, v, g, beta, s0 = inp
    do = rng.standard_normal(v.shape[:3] + (v.shape[3],))
    dht = rng.standard_normal(s0.shape)
    grads = oracle.bwd_recurrent(q, k, v, g, beta, do, h0=s0, dht=dht)
    names = ["dq", "dk", "dv", "dg", "dbeta", "dh0"]
    eps = 1e-6
    for idx, name in enumerate(names):
        x = inp[idx]
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            mi = it.multi_index
            old = x[mi]
            x[mi] = old + eps
            lp = _loss(inp, do, dht)
            x[mi] = old - eps
            lm = _loss(inp, do, dht)
            x[mi] = old
            fd[mi] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grads[name], fd, rtol=0, atol=1e-4, err_msg=name)
    # clamped gates carry no gradient
    assert np.all(grads["dg"][g < -5.0] == 0.0)


@pytest.mark.parametrize("T", [64, 256])
def test_backward_adjoint_identity(T):
    """<grad, dx> summed over all inputs equals the directional derivative of
    L = <do, o> + <dht, S_T> along a random tangent (central difference)."""
    rng = np.random.default_rng(40 + T)
    inp = list(rand_inputs(B=1, T=T, H=2, HV=4, K=16, V=16, seed=41 + T))
    inp[3] = _away_from_kink(inp[3] * 2.0, rng)
    q, k, v, g, beta, s0 = inp
    do = rng.standard_normal(v.shape)
    dht = rng.standard_normal(s0.shape)
    grads = oracle.bwd_recurrent(q, k, v, g, beta, do, h0=s0, dht=dht)
    tang = [rng.standard_normal(x.shape) for x in inp]
    gsum = sum(np.sum(grads[n] * t) for n, t in zip(["dq", "dk", "dv", "dg", "dbeta", "dh0"], tang))
    eps = 1e-6
    plus = [x + eps * t for x, t in zip(inp, tang)]
    minus = [x - eps * t for x, t in zip(inp, tang)]
    dd = (_loss(plus, do, dht) - _loss(minus, do, dht)) / (2 * eps)
    assert abs(gsum - dd) <= 1e-6 * max(1.0, abs(dd)), (gsum, dd)
