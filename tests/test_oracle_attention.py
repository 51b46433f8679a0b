"""Pins for the oracle's attention, Jensen correction and split merge."""

import numpy as np
import pytest
from scipy import integrate

from oracle import attention as A
from oracle import layout, window
from bit_kv_cache_28_b300 import synth


def brute_attention(Q, Kall, Vall, tau, bias=None):
    """Direct definition: w_ij = exp(l_ij) / sum_j exp(l_ij), no max shift (small inputs)."""
    out = np.zeros((Q.shape[0], Vall.shape[1]))
    for i in range(Q.shape[0]):
        ws = []
        for j in range(Kall.shape[0]):
            l = tau * sum(float(Q[i, c]) * float(Kall[j, c]) for c in range(Q.shape[1]))
            if bias is not None:
                l += bias[i, j]
            ws.append(np.exp(l))
        tot = sum(ws)
        for j in range(Kall.shape[0]):
            out[i] += ws[j] / tot * Vall[j]
    return out


def test_softmax_matches_brute_force():
    rng = np.random.default_rng(0)
    Q = rng.standard_normal((3, 5))
    Kc, Vc = rng.standard_normal((4, 5)), rng.standard_normal((4, 5))
    Kn, Vn = rng.standard_normal((2, 5)), rng.standard_normal((2, 5))
    delta = rng.uniform(0, 0.3, (3, 4))
    o, lse = A.attention_rows(Q, Kc, Vc, Kn, Vn, 0.7, delta_keys=delta)
    bias = np.concatenate([-delta, np.zeros((3, 2))], 1)
    ref = brute_attention(Q, np.concatenate([Kc, Kn]), np.concatenate([Vc, Vn]), 0.7, bias)
    assert np.abs(o - ref).max() < 1e-13
    # lse is log of the partition function
    Z = np.exp(0.7 * Q @ np.concatenate([Kc, Kn]).T + bias).sum(1)
    assert np.abs(lse - np.log(Z)).max() < 1e-13


def test_equal_keys_give_mean_of_values():
    rng = np.random.default_rng(1)
    k = rng.standard_normal(8)
    K = np.tile(k, (6, 1))
    V = rng.standard_normal((6, 8))
    o, _ = A.attention_rows(rng.standard_normal((2, 8)), K[:4], V[:4], K[4:], V[4:], 0.35)
    assert np.abs(o - V.mean(0)).max() < 1e-14


def test_unquantised_cache_equals_exact_attention():
    """A cache whose windows are all 16-bit is exact attention over cache + chunk."""
    c = synth.decode_case(seed=11, B=2, Hq=4, Hkv=2, d=64, n_cache=200)
    W = (200 + 31) // 32
    bits = np.full((2, W), 16)
    cache = layout.build_mixed(c["K_cache"], c["V_cache"], bits, [W, 0, 0], "f16")
    Q = synth.to_dtype_values(np.random.default_rng(2).standard_normal((2, 4, 5, 64)), "f16")
    Kn = c["K_cache"][:, :, :3] * 0.5
    Vn = c["V_cache"][:, :, :3] * 0.5
    o, lse = A.attention_over_cache(cache, Q, Kn, Vn, "f16", jensen=A.JENSEN_TAYLOR2)
    tau = 1 / 8
    for b in range(2):
        for h in range(4):
            kv = h // 2
            Kall = np.concatenate([c["K_cache"][b, kv], Kn[b, kv]]).astype(np.float64)
            Vall = np.concatenate([c["V_cache"][b, kv], Vn[b, kv]]).astype(np.float64)
            lg = tau * Q[b, h].astype(np.float64) @ Kall.T
            p = np.exp(lg - lg.max(1, keepdims=True))
            ref = p @ Vall / p.sum(1, keepdims=True)
            assert np.abs(o[b, h] - ref).max() < 1e-12


def test_gqa_equals_repeated_heads():
    c = synth.chunk_case(5, B=1, Hkv=2, Hq=6, d=64, chunks=[70], n_cur=9, n_q=4, dtype="bf16")
    cache = layout.build_uniform(c["K_cache"], c["V_cache"], 2, c["chunks"], 8)
    o, lse = A.attention_over_cache(cache, c["Q"], c["K_cur"], c["V_cur"], "bf16", jensen=1)
    rep = lambda a: np.repeat(a, 3, axis=1)
    cache_mha = layout.build_uniform(rep(c["K_cache"]), rep(c["V_cache"]), 2, c["chunks"], 8)
    o2, lse2 = A.attention_over_cache(cache_mha, c["Q"], rep(c["K_cur"]), rep(c["V_cur"]), "bf16", jensen=1)
    assert np.abs(o - o2).max() == 0 and np.abs(lse - lse2).max() == 0


@pytest.mark.parametrize("splits", [1, 2, 3, 7])
def test_lse_merge_equals_unsplit(splits):
    rng = np.random.default_rng(splits)
    Q = rng.standard_normal((5, 16))
    K = rng.standard_normal((40, 16)) * 2
    V = rng.standard_normal((40, 16))
    o_ref, lse_ref = A.attention_rows(Q, K, V, K[:0], V[:0], 0.25)
    edges = np.linspace(0, 40, splits + 1).astype(int)
    ms, ls, os_ = [], [], []
    for s0, s1 in zip(edges[:-1], edges[1:]):
        lg = 0.25 * Q @ K[s0:s1].T
        m = lg.max(1)
        p = np.exp(lg - m[:, None])
        l = p.sum(1)
        ms.append(m)
        ls.append(l)
        os_.append(p @ V[s0:s1] / l[:, None])
    # an empty split is skipped
    ms.append(np.full(5, -np.inf))
    ls.append(np.zeros(5))
    os_.append(np.zeros((5, 16)))
    o, lse = A.lse_merge(ms, ls, os_)
    assert np.abs(o - o_ref).max() < 1e-13 and np.abs(lse - lse_ref).max() < 1e-13


# ---------------------------------------------------------------- Jensen -----

def test_single_channel_closed_form():
    """E[exp(a eps)] for eps ~ U(-s/2, s/2) equals sinh(a s/2) / (a s/2) (numerical integral)."""
    for a, s in [(0.3, 1.0), (2.0, 1.5), (-1.2, 0.7), (5.0, 2.0)]:
        val, _ = integrate.quad(lambda e: np.exp(a * e) / s, -s / 2, s / 2)
        x = a * s / 2
        assert abs(np.log(val) - A.log_sinhc(x)) < 1e-12
        # and the per-score delta for one channel
        d = A.jensen_delta(np.array([[a / 0.5]]), np.array([[s]]), 0.5, A.JENSEN_EXACT)
        assert abs(d[0, 0] - np.log(val)) < 1e-12


def test_taylor2_is_second_order_of_exact():
    rng = np.random.default_rng(3)
    Q = rng.standard_normal((4, 32)) * 0.2
    S = rng.uniform(0, 0.5, (6, 32))
    tau = 1 / np.sqrt(32)
    ex = A.jensen_delta(Q, S, tau, A.JENSEN_EXACT)
    t2 = A.jensen_delta(Q, S, tau, A.JENSEN_TAYLOR2)
    x = 0.5 * tau * Q[:, None, :] * S[None]
    bound = (x ** 4 / 180).sum(-1) * 1.01 + 1e-15      # next term of the series
    assert (np.abs(ex - t2) <= bound).all()
    # direct restatement: (tau^2/24) sum_c q_c^2 s_c^2 for one pair
    assert abs(t2[1, 2] - tau * tau / 24 * np.sum(Q[1] ** 2 * S[2] ** 2)) < 1e-15


def test_isotropic_jensen_pins():
    """The query-norm form (tau^2/24)|q|^2 mean_c s_c^2: a hand value, equality with TAYLOR2
    whenever a group's steps are equal, and a difference from it when they are not."""
    # hand value: q = (1, 2, 0, 0), s = (2, 0, 4, 2), tau = 1/2: |q|^2 = 5, mean s^2 = 24/4 = 6,
    # delta = (1/4)/24 * 30 = 0.3125
    d = A.jensen_delta(np.array([[1.0, 2.0, 0.0, 0.0]]), np.array([[2.0, 0.0, 4.0, 2.0]]), 0.5,
                       A.JENSEN_ISOTROPIC)
    assert abs(d[0, 0] - 0.3125) < 1e-15
    rng = np.random.default_rng(7)
    Q = rng.standard_normal((5, 32))
    S = np.repeat(rng.uniform(0.1, 2.0, (6, 1)), 32, axis=1)     # equal steps within each group
    tau = 1 / np.sqrt(32)
    iso = A.jensen_delta(Q, S, tau, A.JENSEN_ISOTROPIC)
    t2 = A.jensen_delta(Q, S, tau, A.JENSEN_TAYLOR2)
    assert np.abs(iso - t2).max() < 1e-12 * np.abs(t2).max()
    S2 = rng.uniform(0.1, 2.0, (6, 32))
    assert np.abs(A.jensen_delta(Q, S2, tau, A.JENSEN_ISOTROPIC) - A.jensen_delta(Q, S2, tau, A.JENSEN_TAYLOR2)).max() > 1e-3


def test_jensen_special_cases():
    Q = np.zeros((2, 8))
    S = np.ones((3, 8))
    for mode in (A.JENSEN_TAYLOR2, A.JENSEN_EXACT, A.JENSEN_ISOTROPIC):
        assert np.abs(A.jensen_delta(Q, S, 0.3, mode)).max() == 0
        assert np.abs(A.jensen_delta(np.ones((2, 8)), np.zeros((3, 8)), 0.3, mode)).max() == 0
        assert (A.jensen_delta(np.ones((1, 8)), S, 0.3, mode) > 0).all()


def test_monte_carlo_exact_removes_bias():
    """Mean over noise draws of exp(tau q.k_hat - delta_exact) equals exp(tau q.k)."""
    rng = np.random.default_rng(4)
    d, n_keys, draws = 16, 12, 200000
    tau = 1 / np.sqrt(d)
    q = rng.standard_normal(d) * 1.5
    K = rng.standard_normal((n_keys, d))
    s = rng.uniform(0.1, 1.5, d)                       # one group: per-channel steps
    delta = A.jensen_delta(q[None], s[None], tau, A.JENSEN_EXACT)[0, 0]
    for j in range(3):
        eps = rng.uniform(-0.5, 0.5, (draws, d)) * s
        vals = np.exp(tau * (K[j] + eps) @ q - delta)
        mean, se = vals.mean(), vals.std() / np.sqrt(draws)
        target = np.exp(tau * K[j] @ q)
        assert abs(mean - target) < 3.5 * se + 1e-12


def test_monte_carlo_attention_mass_bias_reduced():
    """Cached keys steal mass from the current chunk under noise; Taylor2 removes >= 90% of it (x <= 0.5)."""
    rng = np.random.default_rng(5)
    d, nc, nn, draws = 32, 24, 8, 4000
    tau = 1 / np.sqrt(d)
    q = rng.standard_normal(d)
    Kc = rng.standard_normal((nc, d))
    Kn = rng.standard_normal((nn, d))
    s = np.full(d, 2 * 0.5 / (tau * np.abs(q).max()))   # makes max_c x_c = 0.5
    x = 0.5 * tau * np.abs(q) * s
    assert x.max() <= 0.5 + 1e-12
    delta = A.jensen_delta(q[None], s[None], tau, A.JENSEN_TAYLOR2)[0, 0]

    def mass(logit_c, logit_n):
        m = max(logit_c.max(), logit_n.max())
        ec, en = np.exp(logit_c - m).sum(), np.exp(logit_n - m).sum()
        return ec / (ec + en)

    true = mass(tau * Kc @ q, tau * Kn @ q)
    # the mass is a nonlinear function of the noisy sum, so compare the
    # expected cache partition sums (what the correction targets)
    unc, cor = [], []
    ref_sum = np.exp(tau * Kc @ q).sum()
    for _ in range(draws):
        eps = rng.uniform(-0.5, 0.5, (nc, d)) * s
        lc = tau * (Kc + eps) @ q
        unc.append(np.exp(lc).sum())
        cor.append(np.exp(lc - delta).sum())
    bias_unc = np.mean(unc) - ref_sum
    bias_cor = np.mean(cor) - ref_sum
    assert bias_unc > 0                                   # noise inflates the cached share
    assert abs(bias_cor) <= 0.1 * bias_unc + 3 * np.std(cor) / np.sqrt(draws)
    assert 0 < true < 1


def test_planted_sign_error_is_caught(monkeypatch):
    """A sign flip in the correction makes the Monte Carlo pin fail."""
    orig = A.jensen_delta
    monkeypatch.setattr(A, "jensen_delta", lambda *a, **k: -orig(*a, **k))
    with pytest.raises(AssertionError):
        test_monte_carlo_exact_removes_bias()


def test_jensen_applies_only_to_quantised_keys():
    """RAW16 windows and the current chunk carry no correction."""
    c = synth.decode_case(seed=12, B=1, Hq=2, Hkv=1, d=64, n_cache=96)
    bits = np.array([[16, 2, 16]])
    cache = layout.build_mixed(c["K_cache"], c["V_cache"], bits, [2, 0, 1], "f16")
    Q = c["Q"]
    o0, l0 = A.attention_over_cache(cache, Q, c["K_cur"], c["V_cur"], "f16", jensen=0)
    o1, l1 = A.attention_over_cache(cache, Q, c["K_cur"], c["V_cur"], "f16", jensen=1)
    lg = cache.logical(0, 0)
    assert lg["quantised"].tolist() == [False, True, False]
    assert (l1 < l0).all()            # the INT2 window's logits were lowered
    bits_raw = np.array([[16, 16, 16]])
    cache_raw = layout.build_mixed(c["K_cache"], c["V_cache"], bits_raw, [3, 0, 0], "f16")
    a0, _ = A.attention_over_cache(cache_raw, Q, c["K_cur"], c["V_cur"], "f16", jensen=0)
    a1, _ = A.attention_over_cache(cache_raw, Q, c["K_cur"], c["V_cur"], "f16", jensen=1)
    assert np.abs(a0 - a1).max() == 0


def test_one_precision_model_and_operand_storage():
    """The oracle has one precision model: the exact dequantised entries, fp64 arithmetic, the
    same whatever the inputs' dtype.  Hand case: 32 cached tokens whose key channel 0 and value
    channel 0 are the constant 1 + 2^-10 (a constant group quantises to itself: s = 0, z = x),
    everything else 0, one query e_0, no current chunk.  All logits are tau x, so
    lse = tau x + ln 32 and o_0 = x.  x is exact in fp32 and fp16 (10 fraction bits) but rounds
    to 1 in bf16 (7 fraction bits): the definition and fp16 operand storage keep it, bf16
    storage gives lse = tau + ln 32 and o_0 = 1."""
    x = 1.0 + 2.0 ** -10
    d = 32
    K = np.zeros((1, 1, 32, d), np.float32)
    V = np.zeros((1, 1, 32, d), np.float32)
    K[..., 0] = x
    V[..., 0] = x
    Q = np.zeros((1, 1, 1, d), np.float32)
    Q[..., 0] = 1.0
    none = np.zeros((1, 1, 0, d), np.float32)
    cache = layout.build_uniform(K, V, 2, [32], 1)
    tau = 1.0 / np.sqrt(d)
    for io in ("f32", "f16", "bf16"):
        o, l = A.attention_over_cache(cache, Q, none, none, io)
        assert o[0, 0, 0, 0] == x and l[0, 0, 0] == tau * x + np.log(32.0)
    o, l = A.attention_over_cache(cache, Q, none, none, "bf16", operand_dtype="f16")
    assert o[0, 0, 0, 0] == x and l[0, 0, 0] == tau * x + np.log(32.0)
    o, l = A.attention_over_cache(cache, Q, none, none, "bf16", operand_dtype="bf16")
    assert o[0, 0, 0, 0] == 1.0 and l[0, 0, 0] == tau + np.log(32.0)


def test_operand_storage_stays_within_its_rounding_bound():
    """Storing the operands in bf16 moves each cached logit by at most tau sum_c |q_c| |k_c| 2^-8
    (the relative rounding of a key entry), so the lse moves by at most the largest such bound."""
    c = synth.chunk_case(9, Hkv=1, d=64, chunks=[64], n_cur=8, n_q=4, dtype="bf16")
    cache = layout.build_uniform(c["K_cache"], c["V_cache"], 2, [64], 2)
    ex = A.attention_over_cache(cache, c["Q"], c["K_cur"], c["V_cur"], "bf16")
    rb = A.attention_over_cache(cache, c["Q"], c["K_cur"], c["V_cur"], "bf16", operand_dtype="bf16")
    assert not np.array_equal(rb[0], ex[0])
    kh = cache.logical(0, 0)["khat"]
    tau = 1 / 8
    bound = tau * np.abs(c["Q"][0, 0]).astype(np.float64) @ np.abs(kh).T.astype(np.float64) * 2.0 ** -8
    assert np.abs(rb[1] - ex[1]).max() <= bound.max()
