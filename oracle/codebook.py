"""QSAC-style codebook keys and the codebook cache (oracle, test infrastructure only).

"QuantWM" (Innovations, item 2; Methodology): INT2 key centroids chosen per
channel with quantisation-sensitivity-aware clustering that weighs channels by
the historical queries' sensitivity.  The pages give no algorithm, so the
reading is a per-(head, channel) 1-D Lloyd k-means with 4 centroids:

* sensitivity weight w_c = mean over historical queries of q_c^2.  It is one
  constant per channel, so inside that channel's 1-D k-means it cancels from
  every weighted mean and every assignment: the weighted algorithm equals the
  unweighted one.  It is computed and reported, and changes nothing.
* init at quantiles: sort the n values, mu_k = x_(floor((2k+1) n / 8)).
* 20 iterations: assign each value to the nearest centroid by |x - mu_k| in
  fp64 (ties to the lower k); mu_k = (exact sum of members) / n_k rounded
  once to fp64; an empty cluster keeps its centroid.
* centroids are stored as fp32; the stored index of a value is its nearest
  fp32 centroid, again by fp64 |x - mu_k| with ties to the lower k.

The exact member sum (``math.fsum``) equals any-order fp64 summation whenever
that summation is exact, which holds for bf16 inputs of magnitude >= 2^-30 at
these sizes.

QSAC with residual ranges.  The pages say QSAC weighs the historical queries'
sensitivity together with the range of the residuals, protecting the channels
that matter more for attention.  A per-channel weight cannot do that inside a
1-D mean-squared k-means (it cancels), so the reading that lets it act is a
per-channel choice of objective:

* relative sensitivity rho_c = w_c / max_c' w_c' (fp64 of the fp32 weights), in
  [0, 1]; rho = 0 when every weight is 0;
* the same quantile initialisation and nearest-centroid assignment, and the
  update mu_k = mean_k + rho_c (mid_k - mean_k): mean_k the members' mean (the
  mean-squared centroid) and mid_k = (min_k + max_k) / 2 the members' mid-range
  (the centroid that minimises the cluster's largest residual |x - mu|), each
  operation one fp64 rounding in that order.

rho = 0 is Lloyd; the most sensitive channel (rho = 1) iterates towards the
smallest residual range; channels in between blend the two.

Residual variance (for the Jensen term of codebook keys): v_c = (1/n) sum_t
(x_t - mu_a(t))^2 over the fitted keys with the stored fp32 centroids and the
stored nearest index a(t), summed in fp64.
"""

from __future__ import annotations

import math

import numpy as np

from .quant import quantize_groups, dequantize, pack_codes, F32
from .layout import BLOCK, CB2, Cache, block_bytes, ceil8

F64 = np.float64


def nearest(x, mu):
    """Index of the nearest centroid by fp64 |x - mu_k|, ties to the lower k."""
    x = np.asarray(x, F64)
    mu = np.asarray(mu, F64)
    dist = np.abs(x[:, None] - mu[None, :])
    return np.argmin(dist, axis=1)          # argmin returns the first minimum


def kmeans_1d(x, k=4, iters=20):
    """1-D Lloyd k-means of one channel; returns fp64 centroids [k]."""
    x = np.asarray(x, F64)
    n = x.shape[0]
    xs = np.sort(x)
    mu = np.array([xs[(2 * j + 1) * n // (2 * k)] for j in range(k)], F64)
    for _ in range(iters):
        a = nearest(x, mu)
        for j in range(k):
            mem = x[a == j]
            if mem.shape[0] > 0:
                mu[j] = math.fsum(mem.tolist()) / mem.shape[0]
    return mu


def sensitivity(Qhist):
    """w_c = mean_t q_{t,c}^2 over historical queries Qhist [n, d] (fp64)."""
    Q = np.asarray(Qhist, F64)
    return (Q * Q).mean(axis=0)


def sensitivity_f32(Qhist):
    """The stored weight: fp32 of (sum_t q_{t,c}^2, summed in token order in fp64) / n."""
    Q = np.asarray(Qhist, F64)
    return (np.cumsum(Q * Q, axis=0)[-1] / Q.shape[0]).astype(F32)


def relative_sensitivity(w32):
    """rho_c = w_c / max_c' w_c' in fp64 from the fp32 weights (0 when all are 0)."""
    w = np.asarray(w32, F32).astype(F64)
    m = w.max()
    return np.zeros_like(w) if m == 0.0 else w / m


def kmeans_1d_range(x, rho, k=4, iters=20):
    """QSAC with residual range of one channel: quantile init, nearest assignment, and
    mu_k = mean_k + rho (mid_k - mean_k); returns fp64 centroids [k]."""
    x = np.asarray(x, F64)
    n = x.shape[0]
    xs = np.sort(x)
    mu = np.array([xs[(2 * j + 1) * n // (2 * k)] for j in range(k)], F64)
    rho = F64(rho)
    for _ in range(iters):
        a = nearest(x, mu)
        new = mu.copy()
        for j in range(k):
            mem = x[a == j]
            if mem.shape[0] > 0:
                mean = F64(math.fsum(mem.tolist()) / mem.shape[0])
                mid = (F64(mem.min()) + F64(mem.max())) * 0.5
                new[j] = mean + rho * (mid - mean)
        mu = new
    return mu


def fit_centroids_range(Kh, w32, iters=20):
    """QSAC-with-residual-range centroids fp32 [d, 4] of one head's keys Kh [n, d], given the
    channels' fp32 sensitivity weights w32 [d]."""
    Kh = np.asarray(Kh, F64)
    rho = relative_sensitivity(w32)
    return np.stack([kmeans_1d_range(Kh[:, c], rho[c], 4, iters) for c in range(Kh.shape[1])]).astype(F32)


def residual_var(Kh, cent):
    """v_c = mean_t (x_t - mu_a(t))^2 of one head's keys Kh [n, d] against fp32 centroids [d, 4]."""
    Kh = np.asarray(Kh, F64)
    v = np.zeros(Kh.shape[1], F64)
    for c in range(Kh.shape[1]):
        mu = np.asarray(cent[c], F32).astype(F64)
        e = Kh[:, c] - mu[nearest(Kh[:, c], mu)]
        v[c] = (e * e).sum() / Kh.shape[0]
    return v


def fit_centroids(Kh, iters=20):
    """Centroids fp32 [d, 4] of one head's cached keys Kh [n, d]."""
    Kh = np.asarray(Kh, F64)
    return np.stack([kmeans_1d(Kh[:, c], 4, iters) for c in range(Kh.shape[1])]).astype(F32)


def encode_cb_blocks(Kb, Vb, cent, coeff, nvalid, r):
    """Pack N codebook blocks of one head.

    Kb, Vb: fp32 [N, 32, d]; cent fp32 [d, 4]; coeff fp16 [N, 32, r] or None.
    """
    Kb = np.asarray(Kb, F32)
    Vb = np.asarray(Vb, F32)
    N, T, d = Kb.shape
    idx = np.zeros((N, T, d), np.uint8)
    for c in range(d):
        idx[:, :, c] = nearest(Kb[:, :, c].reshape(-1), cent[c]).reshape(N, T)
    idx[:, nvalid:] = 0
    vc, vs, vz = quantize_groups(Vb.reshape(N, T, d // 32, 32), 2)
    vc[:, nvalid:] = 0
    vs[:, nvalid:] = 0
    vz[:, nvalid:] = 0
    rp = ceil8(r)
    cq = np.zeros((N, T, rp), np.float16)
    if r:
        cq[:, :nvalid, :r] = coeff[:, :nvalid]
    raw = np.concatenate([pack_codes(idx, 2).reshape(N, -1).view(np.uint8),
                          pack_codes(vc.reshape(N, T, d).transpose(0, 2, 1), 2).reshape(N, -1).view(np.uint8),
                          np.ascontiguousarray(np.stack([vs, vz], -1).astype(F32).transpose(0, 2, 1, 3))
                          .reshape(N, -1).view(np.uint8),
                          cq.reshape(N, -1).view(np.uint8)], axis=1)
    khat = cent[np.arange(d)[None, None, :], idx].astype(F32)
    vhat = dequantize(vc, vs[..., None], vz[..., None]).reshape(N, T, d)
    assert raw.shape[1] == block_bytes(CB2, d, r)
    return dict(bytes=raw, idx=idx, khat=khat, vhat=vhat, coeff=cq[..., :r])


def build_codebook(K, V, cent, U, cap_blocks, resid_var=None):
    """Codebook cache of one prefill of n tokens per (b, head).

    K, V: fp32 [B, H, n, d] (bf16 values); cent fp32 [B, H, d, 4];
    U: fp32 [B, H, d, r] PSAC basis or None (r = 0).
    resid_var: fp32 [B, H, d] per-channel residual variances, or None.  Codebook
    keys have no step sizes: without residual variances no Jensen term applies;
    with them, the attention applies the codebook form (attention.codebook_jensen).
    """
    from .psac import psac_coeff
    K = np.asarray(K, F32)
    V = np.asarray(V, F32)
    B, H, n, d = K.shape
    r = 0 if U is None else U.shape[-1]
    c = Cache(B, H, d, [CB2], [cap_blocks], r)
    nb = (n + BLOCK - 1) // BLOCK
    assert nb <= cap_blocks
    npad = nb * BLOCK
    for b in range(B):
        for h in range(H):
            Kp = np.zeros((npad, d), F32)
            Vp = np.zeros((npad, d), F32)
            Kp[:n] = K[b, h]
            Vp[:n] = V[b, h]
            for j in range(nb):
                nv = min(BLOCK, n - j * BLOCK)
                Kb = Kp[j * BLOCK:(j + 1) * BLOCK][None]
                Vb = Vp[j * BLOCK:(j + 1) * BLOCK][None]
                co = None
                if r:
                    idx = np.stack([nearest(Kb[0, :, ch], cent[b, h, ch]) for ch in range(d)], 1)
                    khat = cent[b, h][np.arange(d)[None, :], idx]
                    co = psac_coeff(Kb[0], khat, U[b, h])[None]
                enc = encode_cb_blocks(Kb, Vb, cent[b, h], co, nv, r)
                c._put(b, h, 0, j, enc["bytes"][0])
                rec = dict(pos=j * BLOCK, len=nv, khat=enc["khat"][0], vhat=enc["vhat"][0],
                           ks=np.zeros(d, F32), quantised=False, seg=0, slot=j)
                rec["coeff"] = enc["coeff"][0].astype(F64) if r else np.zeros((BLOCK, 0))
                c.blocks[b][h].append(rec)
                if h == 0:
                    c.blk_len[b, j] = nv
                    c.blk_pos[b, j] = j * BLOCK
    c.n_blocks = [nb]
    c.n_tokens = n
    c.resid_var = None if resid_var is None else np.asarray(resid_var, F32)
    return c
