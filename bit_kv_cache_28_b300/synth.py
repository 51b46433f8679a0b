"""Seeded synthetic workloads.

This module only draws random inputs and rounds them to the I/O dtype; it holds
none of the quantisation, attention or clustering arithmetic.  Tests feed the
same arrays to the CUDA path and to the oracle; the benchmark feeds them to the
CUDA path.

Every generator uses ``numpy.random.Generator(PCG64(seed))`` and draws in the
order documented on each function.  Arrays are fp32 holding values that are
exact in the workload's dtype (bf16 / fp16 values are rounded with
round-to-nearest-even before being returned).

Workloads (the shapes of the video-diffusion and video-VLM settings on the
source pages; no public dataset is involved):

* ``tiny``     1 head, d 64, 1024 cached + 64 current tokens, fp32, 4 outlier key
               channels x8.
* ``chunk``    24 heads, d 128, current chunk 1560 (3 latent frames x 520), cache of
               3 prior chunks, bf16; keys N(0,1) x per-channel lognormal(0, 0.5)
               with 8 outlier channels per head x10.
* ``rollout``  as ``chunk`` with 40 heads and 21 cached chunks (32760 tokens).
* ``decode``   batch 8, 28 query heads over 4 kv heads, d 64, 100 frames x 196 =
               19600 cached tokens, one query, fp16, window similarity U(-1, 1).
* ``codebook`` 24 heads, d 128, 8192 cached tokens, 1560 current tokens, 256
               historical queries per head; queries x per-channel lognormal(0, 0.7).
"""

from __future__ import annotations

import numpy as np


def to_bf16_values(x):
    """Round fp32 to the nearest bf16 (ties to even); return fp32 holding the bf16 values."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = ((u + 0x7FFF + lsb) & 0xFFFF0000).astype(np.uint32)
    return u.view(np.float32)


def to_dtype_values(x, dtype):
    if dtype == "f32":
        return np.asarray(x, np.float32)
    if dtype == "f16":
        return np.asarray(x, np.float32).astype(np.float16).astype(np.float32)
    if dtype == "bf16":
        return to_bf16_values(x)
    raise ValueError(dtype)


def _normal(rng, shape):
    return rng.standard_normal(size=shape, dtype=np.float32)


def chunk_case(seed, *, B=1, Hkv=24, Hq=None, d=128, chunks=(1560, 1560, 1560), n_cur=1560,
               n_q=None, dtype="bf16", sigma=0.5, n_outlier=8, outlier_scale=10.0, q_sigma=0.0):
    """Chunk-wise cache workload.

    Draw order: per-(head, channel) key scale lognormal(0, sigma) [Hkv, d]; for
    each kv head the outlier channels (without replacement); K_cache, K_cur,
    V_cache, V_cur ~ N(0,1); Q ~ N(0,1) [B, Hq, n_q, d]; if q_sigma > 0, a
    per-(kv head, channel) query scale lognormal(0, q_sigma).
    """
    Hq = Hkv if Hq is None else Hq
    n_q = n_cur if n_q is None else n_q
    rng = np.random.Generator(np.random.PCG64(seed))
    n_cache = int(sum(chunks))
    kscale = np.exp(sigma * _normal(rng, (Hkv, d))) if sigma > 0 else np.ones((Hkv, d), np.float32)
    for h in range(Hkv):
        if n_outlier:
            ch = rng.choice(d, size=n_outlier, replace=False)
            kscale[h, ch] *= outlier_scale
    Kc = _normal(rng, (B, Hkv, n_cache, d)) * kscale[None, :, None, :]
    Kn = _normal(rng, (B, Hkv, n_cur, d)) * kscale[None, :, None, :]
    Vc = _normal(rng, (B, Hkv, n_cache, d))
    Vn = _normal(rng, (B, Hkv, n_cur, d))
    Q = _normal(rng, (B, Hq, n_q, d))
    if q_sigma > 0:
        qscale = np.exp(q_sigma * _normal(rng, (Hkv, d)))
        Q = Q * np.repeat(qscale, Hq // Hkv, axis=0)[None, :, None, :]
    cv = lambda a: to_dtype_values(a, dtype)
    return dict(K_cache=cv(Kc), V_cache=cv(Vc), K_cur=cv(Kn), V_cur=cv(Vn), Q=cv(Q),
                chunks=list(chunks), dtype=dtype, B=B, Hkv=Hkv, Hq=Hq, d=d)


def tiny(seed=1):
    """1 head, d 64, cache 1024 (one append), chunk 64, fp32, 4 outlier key channels x8."""
    rng = np.random.Generator(np.random.PCG64(seed))
    d = 64
    ch = rng.choice(d, size=4, replace=False)
    Kc = _normal(rng, (1, 1, 1024, d))
    Vc = _normal(rng, (1, 1, 1024, d))
    Kn = _normal(rng, (1, 1, 64, d))
    Vn = _normal(rng, (1, 1, 64, d))
    Q = _normal(rng, (1, 1, 64, d))
    Kc[..., ch] *= 8.0
    Kn[..., ch] *= 8.0
    return dict(K_cache=Kc, V_cache=Vc, K_cur=Kn, V_cur=Vn, Q=Q, chunks=[1024], dtype="f32",
                B=1, Hkv=1, Hq=1, d=d, outliers=np.sort(ch))


def chunk(seed=2, n_heads=24, n_chunks=3):
    """24 heads, d 128, chunk 1560, cache of 3 chunks, bf16."""
    return chunk_case(seed, Hkv=n_heads, chunks=[1560] * n_chunks)


def rollout(seed=3):
    """40 heads, d 128, chunk 1560, cache of 21 chunks (32760 tokens), bf16."""
    return chunk_case(seed, Hkv=40, chunks=[1560] * 21)


def decode_case(seed=4, *, B=8, Hq=28, Hkv=4, d=64, n_cache=19600, dtype="f16"):
    """Windowed decode workload.

    Draw order: K_cache, V_cache [B, Hkv, n, d]; K_cur, V_cur [B, Hkv, 1, d];
    Q [B, Hq, 1, d]; window similarity U(-1, 1) [B, ceil(n/32)].
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    W = (n_cache + 31) // 32
    Kc = _normal(rng, (B, Hkv, n_cache, d))
    Vc = _normal(rng, (B, Hkv, n_cache, d))
    Kn = _normal(rng, (B, Hkv, 1, d))
    Vn = _normal(rng, (B, Hkv, 1, d))
    Q = _normal(rng, (B, Hq, 1, d))
    sim = rng.uniform(-1.0, 1.0, size=(B, W)).astype(np.float32)
    cv = lambda a: to_dtype_values(a, dtype)
    return dict(K_cache=cv(Kc), V_cache=cv(Vc), K_cur=cv(Kn), V_cur=cv(Vn), Q=cv(Q), sim=sim,
                dtype=dtype, B=B, Hkv=Hkv, Hq=Hq, d=d)


def codebook_case(seed=5, *, H=24, d=128, n_cache=8192, n_cur=1560, n_hist=256, dtype="bf16",
                  q_sigma=0.7):
    """QuantWM-style workload.

    Draw order: query scale lognormal(0, q_sigma) [H, d]; K_cache, V_cache
    [1, H, n_cache, d]; K_cur, V_cur [1, H, n_cur, d]; Q [1, H, n_cur, d];
    Q_hist [H, n_hist, d]; Q and Q_hist carry the query scale.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    qscale = np.exp(q_sigma * _normal(rng, (H, d)))
    Kc = _normal(rng, (1, H, n_cache, d))
    Vc = _normal(rng, (1, H, n_cache, d))
    Kn = _normal(rng, (1, H, n_cur, d))
    Vn = _normal(rng, (1, H, n_cur, d))
    Q = _normal(rng, (1, H, n_cur, d)) * qscale[None, :, None, :]
    Qh = _normal(rng, (H, n_hist, d)) * qscale[:, None, :]
    cv = lambda a: to_dtype_values(a, dtype)
    return dict(K_cache=cv(Kc), V_cache=cv(Vc), K_cur=cv(Kn), V_cur=cv(Vn), Q=cv(Q), Q_hist=cv(Qh),
                dtype=dtype, B=1, Hkv=H, Hq=H, d=d)
