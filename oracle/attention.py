"""Softmax attention over a quantised cache plus the current chunk (oracle, test infrastructure only).

"Quantized Keys Steal Attention" (abstract): in chunk-wise autoregressive video
diffusion the queries of the current chunk attend to the cache of earlier
chunks and to the current, unquantised chunk.  Quantisation noise on cached
keys inflates their expected softmax weight through the convexity of exp (the
Jensen bias); a per-score correction computed from the cached keys' step sizes
and the query removes it in expectation, with a second-order Taylor form.

Reading (no formula is printed): with k_hat = k + eps, eps_c ~ U(-s_c/2, s_c/2)
independent,

    E[exp(tau q.k_hat)] = exp(tau q.k) * prod_c sinh(x_c) / x_c,   x_c = tau q_c s_c / 2

so the corrected cached logit is  tau q.k_hat - delta  with

    delta_exact   = sum_c log(sinh(x_c) / x_c)
    delta_taylor2 = sum_c x_c^2 / 6 = (tau^2 / 24) sum_c q_c^2 s_c^2

and, in the abstract's "query norm" form that treats the noise as isotropic (one
step for every channel, the group's mean square step),

    delta_isotropic = (tau^2 / 24) |q|^2 mean_c s_c^2,

which equals delta_taylor2 whenever a group's steps are all equal.

applied to quantised cached keys only (zero for RAW16 windows and the current
chunk).  All sums and the softmax are fp64; the output is returned in fp64.

Codebook keys (QuantWM) have no step size.  Their second-order form follows the
same expansion, log E[exp(X)] = Var(X) / 2 for a zero-mean logit error X =
tau q.e, with the channels' residuals e_c independent of variance v_c (measured
on the fitted keys):

    delta_taylor2 = (tau^2 / 2) sum_c q'_c^2 v_c,
    delta_isotropic = (tau^2 / 2) |q'|^2 mean_c v_c,

where q' = q - U (U^T q) when the PSAC term is on (PSAC restores the error
component along U, so only the query's part outside that subspace sees the
remaining error) and q' = q otherwise.  For uniform steps v_c = s_c^2 / 12 this is
delta_taylor2 above.  EXACT has no closed form for an empirical residual and is
not defined for codebook keys.  The term is one value per query row, the same for
every cached key.
"""

from __future__ import annotations

import numpy as np

from .quant import round_to

F64 = np.float64

JENSEN_OFF, JENSEN_TAYLOR2, JENSEN_EXACT, JENSEN_ISOTROPIC = 0, 1, 2, 3


def log_sinhc(x):
    """log(sinh(x)/x) in fp64, stable near 0 (series x^2/6 - x^4/180 + x^6/2835)."""
    x = np.abs(np.asarray(x, F64))
    small = x < 1e-3
    xs = np.where(small, 1.0, x)
    # log(sinh x / x) = x + log1p(-exp(-2x)) - log(2x)
    big = xs + np.log1p(-np.exp(-2.0 * xs)) - np.log(2.0 * xs)
    x2 = x * x
    ser = x2 / 6.0 - x2 * x2 / 180.0 + x2 * x2 * x2 / 2835.0
    return np.where(small, ser, big)


def jensen_delta(Q, s_groups, tau, mode):
    """Per (query, key group) Jensen correction.

    Q: [nq, d] queries (fp64 values), s_groups: [G, d] key step sizes per group.
    Returns delta [nq, G] (fp64).
    """
    Q = np.asarray(Q, F64)
    S = np.asarray(s_groups, F64)
    if mode == JENSEN_OFF or S.shape[0] == 0:
        return np.zeros((Q.shape[0], S.shape[0]), F64)
    if mode == JENSEN_TAYLOR2:
        return (tau * tau / 24.0) * ((Q * Q) @ (S * S).T)
    if mode == JENSEN_EXACT:
        x = 0.5 * tau * Q[:, None, :] * S[None, :, :]
        return log_sinhc(x).sum(-1)
    if mode == JENSEN_ISOTROPIC:
        qn2 = (Q * Q).sum(-1)                      # |q|^2
        ms2 = (S * S).mean(-1)                     # mean_c s_c^2 of each group
        return (tau * tau / 24.0) * qn2[:, None] * ms2[None, :]
    raise ValueError(mode)


def codebook_jensen(Q, v, tau, mode, U=None):
    """Per-query Jensen correction for codebook keys: Q [nq, d], v [d] residual variances,
    U [d, r] PSAC basis (None: PSAC off).  Returns delta [nq] (fp64)."""
    Q = np.asarray(Q, F64)
    v = np.asarray(v, F64)
    if U is not None:
        U = np.asarray(U, F64)
        Q = Q - (Q @ U) @ U.T
    if mode == JENSEN_OFF:
        return np.zeros(Q.shape[0], F64)
    if mode == JENSEN_TAYLOR2:
        return 0.5 * tau * tau * ((Q * Q) @ v)
    if mode == JENSEN_ISOTROPIC:
        return 0.5 * tau * tau * (Q * Q).sum(-1) * v.mean()
    raise ValueError("the EXACT Jensen form is not defined for codebook keys")


def softmax_attend(logits, Vall):
    """Row softmax of fp64 logits [nq, n] against values [n, d] -> (o [nq, d], lse [nq]).

    Uses the max-shifted form; pinned against the direct exp/sum definition on
    small inputs in the oracle tests.
    """
    logits = np.asarray(logits, F64)
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    l = p.sum(axis=1, keepdims=True)
    o = (p @ np.asarray(Vall, F64)) / l
    lse = (m + np.log(l))[:, 0]
    return o, lse


def attention_rows(Q, Kc, Vc, Kn, Vn, tau, delta_keys=None, extra_keys=None):
    """Attention of queries Q [nq, d] over cached (Kc, Vc) [nc, d] and current (Kn, Vn) [nn, d].

    delta_keys [nq, nc] is subtracted from and extra_keys [nq, nc] added to the
    cached logits.  All inputs are used as given, in fp64.
    """
    Q = np.asarray(Q, F64)
    lc = tau * (Q @ np.asarray(Kc, F64).T)
    if delta_keys is not None:
        lc = lc - delta_keys
    if extra_keys is not None:
        lc = lc + extra_keys
    ln = tau * (Q @ np.asarray(Kn, F64).T)
    logits = np.concatenate([lc, ln], axis=1)
    Vall = np.concatenate([np.asarray(Vc, F64), np.asarray(Vn, F64)], axis=0)
    return softmax_attend(logits, Vall)


def lse_merge(ms, ls, os_):
    """Merge split partials (m_p, l_p, o_p) with o_p already normalised by l_p.

    m = max m_p; l = sum l_p exp(m_p - m); o = sum l_p exp(m_p - m) o_p / l.
    Splits with l_p == 0 (empty) are skipped.  Returns (o, lse).
    """
    ms = np.asarray(ms, F64)
    ls = np.asarray(ls, F64)
    os_ = np.asarray(os_, F64)
    keep = ls > 0
    m = np.max(np.where(keep, ms, -np.inf), axis=0)
    w = np.where(keep, ls * np.exp(np.where(keep, ms, 0.0) - m), 0.0)
    l = w.sum(axis=0)
    o = (w[..., None] * os_).sum(axis=0) / l[..., None]
    return o, m + np.log(l)


def attention_over_cache(cache, Q, Kcur, Vcur, io_dtype, tau=None, jensen=JENSEN_OFF,
                         psac_U=None, rows=None, operand_dtype=None):
    """Reference attention for every (b, q-head): the plain definition.

    The precision model (one, for every path): the queries and the current chunk
    are the exact values given (16-bit inputs are exact in fp32), the cached keys
    and values are the dequantised entries x_hat = fmaf(code, s, z) exactly as
    the fp32 values they are, and every product, sum and the softmax run in fp64.
    Nothing is rounded on the way; the output is returned in fp64.

    cache : oracle.layout.Cache (or codebook cache) holding the dequantised view.
    Q     : fp32 [B, Hq, nq, d]; Kcur, Vcur: fp32 [B, Hkv, nn, d] (may have nn = 0).
    io_dtype: 'f32' | 'f16' | 'bf16' -- the inputs' dtype (informational: the
              inputs already hold values exact in it).
    psac_U: optional fp32 [B, Hkv, d, r]; adds tau (U^T q) . coeff for cached keys.
    rows  : optional index array of query rows to evaluate (all if None).
    operand_dtype: None for the definition above.  'f16' | 'bf16' | 'f32'
              evaluates the same definition after storing every operand of the two
              products -- Q, the dequantised cached keys and values and the
              current chunk -- in that dtype (round to nearest even), for paths
              documented to hold their operands in 16 bits.  It is a diagnostic
              with a tighter tolerance, never a replacement for the definition.
    GQA: q-head h reads kv-head h // (Hq // Hkv).
    Returns (o [B, Hq, nrows, d], lse [B, Hq, nrows]) in fp64.
    """
    Q = np.asarray(Q, np.float32)
    B, Hq, nq, d = Q.shape
    Hkv = cache.H
    assert Hq % Hkv == 0
    grp = Hq // Hkv
    if tau is None:
        tau = 1.0 / np.sqrt(d)
    if rows is None:
        rows = np.arange(nq)
    store = (lambda x: np.asarray(x, np.float32)) if operand_dtype is None else \
        (lambda x: round_to(x, operand_dtype))
    cb_var = getattr(cache, "resid_var", None)     # codebook caches with residual variances
    o = np.zeros((B, Hq, len(rows), d), F64)
    lse = np.zeros((B, Hq, len(rows)), F64)
    for b in range(B):
        for hk in range(Hkv):
            lg = cache.logical(b, hk)
            Kc = store(lg["khat"])
            Vc = store(lg["vhat"])
            kn = store(Kcur[b, hk]) if Kcur is not None else np.zeros((0, d), np.float32)
            vn = store(Vcur[b, hk]) if Vcur is not None else np.zeros((0, d), np.float32)
            for hq in range(hk * grp, (hk + 1) * grp):
                # the Jensen term and the PSAC product use the query as given
                q_in = Q[b, hq, rows].astype(F64)
                q = store(Q[b, hq, rows]).astype(F64)
                delta = None
                if jensen != JENSEN_OFF and Kc.shape[0] > 0 and cb_var is not None:
                    U = None if psac_U is None else psac_U[b, hk]
                    dq = codebook_jensen(q_in, cb_var[b, hk], tau, jensen, U)
                    delta = np.repeat(dq[:, None], Kc.shape[0], axis=1)
                elif jensen != JENSEN_OFF and Kc.shape[0] > 0:
                    dg = jensen_delta(q_in, lg["ks"], tau, jensen)
                    dg = dg * lg["quantised"][None, :]
                    delta = dg[:, lg["kgroup"]]
                extra = None
                if psac_U is not None and lg["coeff"] is not None and Kc.shape[0] > 0:
                    U = np.asarray(psac_U[b, hk], F64)
                    uq = q_in @ U                                # [nrows, r]
                    extra = tau * (uq @ np.asarray(lg["coeff"], F64).T)
                o[b, hq], lse[b, hq] = attention_rows(q, Kc, Vc, kn, vn, tau, delta, extra)
    return o, lse
