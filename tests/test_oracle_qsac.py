"""Pins of the QSAC-with-residual-range fit and of the Jensen term for codebook keys (oracle).

QuantWM (Innovations 2; Methodology): QSAC weighs the historical queries' sensitivity and the
range of the residuals when it picks INT2 key centroids, protecting the channels that matter
more; PSAC restores the key error along the dominant query subspace.  The readings are in
oracle/codebook.py and oracle/attention.py; these tests fix them by hand cases, closed forms,
a Monte Carlo expectation and invariants."""

import numpy as np
import pytest

from bit_kv_cache_28_b300 import synth
from oracle import codebook as C, attention as A

X = np.array([0, 1, 5, 10, 11, 12, 30, 40], np.float64)


def test_hand_case_sensitivity_moves_the_centroid():
    """x = {0, 1, 5, 10, 11, 12, 30, 40}: quantile init {1, 10, 12, 40}, clusters {0, 1, 5},
    {10, 11}, {12}, {30, 40} from the first assignment on.  Cluster 0 has mean 2 and
    mid-range 2.5: Lloyd (rho 0) gives 2 (largest residual 3, mean square 14/3), the fully
    sensitive channel (rho 1) gives 2.5 (largest residual 2.5, mean square 14.75/3), half
    sensitivity gives 2.25; the other clusters' mean and mid-range agree."""
    assert C.kmeans_1d_range(X, 0.0).tolist() == [2.0, 10.5, 12.0, 35.0]
    assert C.kmeans_1d_range(X, 1.0).tolist() == [2.5, 10.5, 12.0, 35.0]
    assert C.kmeans_1d_range(X, 0.5).tolist() == [2.25, 10.5, 12.0, 35.0]
    assert C.kmeans_1d(X).tolist() == [2.0, 10.5, 12.0, 35.0]


def test_weights_act_per_channel():
    """Two channels holding the same values with weights 4 and 1: rho = (1, 1/4)."""
    K = np.stack([X, X], 1).astype(np.float32)
    w = np.array([4.0, 1.0], np.float32)
    assert C.relative_sensitivity(w).tolist() == [1.0, 0.25]
    cent = C.fit_centroids_range(K, w)
    assert cent[0].tolist() == [2.5, 10.5, 12.0, 35.0]
    assert cent[1].tolist() == [2.125, 10.5, 12.0, 35.0]
    assert C.relative_sensitivity(np.zeros(3, np.float32)).tolist() == [0.0, 0.0, 0.0]


def test_zero_sensitivity_is_lloyd():
    K = synth.codebook_case(seed=3, H=1, d=16, n_cache=500, n_cur=1, n_hist=8)["K_cache"][0, 0]
    assert np.array_equal(C.fit_centroids_range(K, np.zeros(16, np.float32)), C.fit_centroids(K))


def test_full_sensitivity_reaches_the_midrange_fixed_point():
    """rho = 1, iterated to convergence: every centroid is the mid-range of its members, and the
    largest residual is no larger than Lloyd's on the same data."""
    rng = np.random.default_rng(4)
    for trial in range(20):
        x = np.round(rng.standard_normal(60) * 8) / 4
        mu = C.kmeans_1d_range(x, 1.0, iters=200)
        a = C.nearest(x, mu)
        for k in range(4):
            m = x[a == k]
            if m.size:
                assert mu[k] == (m.min() + m.max()) / 2
        lloyd = C.kmeans_1d(x, iters=200)
        r_range = np.abs(x - mu[a]).max()
        r_lloyd = np.abs(x - lloyd[C.nearest(x, lloyd)]).max()
        assert r_range <= r_lloyd + 1e-12


def test_weights_are_stored_as_fp32_of_the_token_order_sum():
    rng = np.random.default_rng(5)
    Q = rng.standard_normal((256, 8)).astype(np.float32)
    w = C.sensitivity_f32(Q)
    acc = np.zeros(8)
    for t in range(256):
        acc = acc + Q[t].astype(np.float64) ** 2
    assert np.array_equal(w, (acc / 256).astype(np.float32))


def test_residual_variance_hand_case():
    """Centroids {2, 10.5, 12, 35}: residuals -2, -1, 3, -0.5, 0.5, 0, -5, 5, mean square 64.5/8."""
    v = C.residual_var(X[:, None], np.array([[2.0, 10.5, 12.0, 35.0]], np.float32))
    assert v.tolist() == [64.5 / 8]


def test_codebook_jensen_equals_the_step_form_for_uniform_residuals():
    """A uniform residual of width s has variance s^2 / 12: the codebook form then equals the
    step-size form of uniform keys."""
    rng = np.random.default_rng(6)
    Q = rng.standard_normal((5, 32))
    s = np.abs(rng.standard_normal(32)) * 3
    tau = 1 / np.sqrt(32)
    a = A.codebook_jensen(Q, s * s / 12, tau, A.JENSEN_TAYLOR2)
    b = A.jensen_delta(Q, s[None], tau, A.JENSEN_TAYLOR2)[:, 0]
    assert np.allclose(a, b, rtol=1e-14, atol=0)
    ai = A.codebook_jensen(Q, s * s / 12, tau, A.JENSEN_ISOTROPIC)
    bi = A.jensen_delta(Q, s[None], tau, A.JENSEN_ISOTROPIC)[:, 0]
    assert np.allclose(ai, bi, rtol=1e-14, atol=0)


def test_codebook_jensen_is_exact_for_gaussian_residuals():
    """For e ~ N(0, diag v), E[exp(tau q.e)] = exp(tau^2/2 sum q_c^2 v_c) exactly: the Monte Carlo
    mean of exp(tau q.e - delta) is 1 within 3.5 standard errors."""
    rng = np.random.default_rng(7)
    d, n = 16, 200000
    q = rng.standard_normal(d) * 1.5
    v = rng.uniform(0.2, 2.0, d)
    tau = 0.4
    delta = A.codebook_jensen(q[None], v, tau, A.JENSEN_TAYLOR2)[0]
    e = rng.standard_normal((n, d)) * np.sqrt(v)
    z = np.exp(tau * e @ q - delta)
    assert abs(z.mean() - 1.0) < 3.5 * z.std() / np.sqrt(n)
    # a dropped factor 1/2 would be far off
    assert abs(np.exp(tau * e @ q - 2 * delta).mean() - 1.0) > 10 * z.std() / np.sqrt(n)


def test_psac_projection_removes_the_compensated_direction():
    """U = the first axis: the query's first channel sees no remaining error."""
    d, tau = 8, 0.5
    v = np.arange(1, d + 1, dtype=np.float64)
    U = np.zeros((d, 1))
    U[0, 0] = 1.0
    e0, e1 = np.eye(d)[0], np.eye(d)[1]
    assert A.codebook_jensen(e0[None], v, tau, A.JENSEN_TAYLOR2, U)[0] == 0.0
    assert A.codebook_jensen(e0[None], v, tau, A.JENSEN_TAYLOR2)[0] == 0.5 * tau * tau * 1.0
    assert A.codebook_jensen(e1[None], v, tau, A.JENSEN_TAYLOR2, U)[0] == 0.5 * tau * tau * 2.0
    with pytest.raises(ValueError):
        A.codebook_jensen(e0[None], v, tau, A.JENSEN_EXACT)


@pytest.mark.parametrize("psac", [False, True])
def test_codebook_attention_shifts_lse_only(psac):
    """Without a current chunk the codebook term lowers every logit of a row by the same
    delta_i: the output is unchanged and the lse drops by exactly delta_i."""
    c = synth.codebook_case(seed=8, H=1, d=32, n_cache=100, n_cur=4, n_hist=32)
    cent = C.fit_centroids(c["K_cache"][0, 0])[None, None]
    v = C.residual_var(c["K_cache"][0, 0], cent[0, 0]).astype(np.float32)[None, None]
    U = None
    if psac:
        from oracle import psac as P
        U = P.psac_basis(c["Q_hist"][0], 4)[0].astype(np.float32)[None, None]
    cache = C.build_codebook(c["K_cache"], c["V_cache"], cent, U, 4, resid_var=v)
    none = np.zeros((1, 1, 0, 32), np.float32)
    o0, l0 = A.attention_over_cache(cache, c["Q"], none, none, "bf16", psac_U=U)
    o1, l1 = A.attention_over_cache(cache, c["Q"], none, none, "bf16", jensen=A.JENSEN_TAYLOR2, psac_U=U)
    tau = 1 / np.sqrt(32)
    delta = A.codebook_jensen(c["Q"][0, 0], v[0, 0], tau, A.JENSEN_TAYLOR2, None if U is None else U[0, 0])
    assert np.abs(o1 - o0).max() < 1e-12
    assert np.abs((l0 - l1)[0, 0] - delta).max() < 1e-12
    assert delta.min() > 0
    # without residual variances the codebook keys carry no term
    plain = C.build_codebook(c["K_cache"], c["V_cache"], cent, U, 4)
    o2, l2 = A.attention_over_cache(plain, c["Q"], none, none, "bf16", jensen=A.JENSEN_TAYLOR2, psac_U=U)
    assert np.array_equal(l2, l0)
