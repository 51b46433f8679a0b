"""Window-level mixed-precision plan (oracle, test infrastructure only).

WindowQuant note, sections 何が新しいのか (table: high relevance -> FP16,
middle -> INT4, low -> INT2), 技術的に面白い点 (the first window is always FP16;
windows of one bit-width are stored together) and 実装者視点で気になった点
(window size 32, one bit-width per window).

Reading: windows 1..W-1 are ranked by similarity, descending, ties to the
lower window index.  With n = W - 1 (or W when the first window is not forced):

    n16 = floor(f16 * n),  n_hi = floor((f16 + f4) * n)     (fp64 arithmetic)
    ranks [0, n16) -> FP16, [n16, n_hi) -> INT4, [n_hi, n) -> INT2

The physical order is FP16 windows, then INT4, then INT2, each in ascending
window index; ``perm[i]`` is the window stored at physical block i.

The similarity that feeds the plan (``window_similarity``) is the cosine
similarity of each window to the question (section 何が新しいのか: each window's
similarity to the text question is computed, by cosine similarity, and picks
the window's bit-width).  The pages do not say which vectors are compared.
Reading: in key space, a window is the mean of its valid tokens' keys and the
question the mean of its tokens' keys, each with every kv head's d channels
concatenated; a zero vector on either side gives similarity 0.
"""

from __future__ import annotations

import math

import numpy as np


def window_plan(sim, frac16=0.2, frac4=0.3, force_first=True):
    sim = np.asarray(sim, dtype=np.float32)
    W = int(sim.shape[0])
    bits = np.full(W, 2, dtype=np.int8)
    if W == 0:
        return bits, np.zeros(0, np.int32)
    first = 1 if force_first else 0
    if force_first:
        bits[0] = 16
    rest = list(range(first, W))
    # rank by similarity (as fp32), descending; equal similarities -> lower index first
    order = sorted(rest, key=lambda w: (-float(sim[w]), w))
    n = len(rest)
    n16 = int(math.floor(float(frac16) * n))
    nhi = int(math.floor((float(frac16) + float(frac4)) * n))
    nhi = max(nhi, n16)
    for rank, w in enumerate(order):
        if rank < n16:
            bits[w] = 16
        elif rank < nhi:
            bits[w] = 4
        else:
            bits[w] = 2
    perm = [w for cls in (16, 4, 2) for w in range(W) if bits[w] == cls]
    return bits, np.asarray(perm, dtype=np.int32)


def window_similarity(K, Kq, window=32):
    """Cosine similarity of every window of K to the question Kq, fp64.

    K: [B, Hkv, n, d] keys of the windows (window w holds tokens 32 w .. 32 w + 31,
    the last one possibly partial); Kq: [B, Hkv, m, d] keys of the question
    tokens.  Returns [B, ceil(n / 32)]: cos(u_w, v) with u_w the mean of window
    w's keys and v the mean of the question's keys, both over all kv heads'
    channels; 0 where either mean is the zero vector (or m == 0).
    """
    K = np.asarray(K, dtype=np.float64)
    Kq = np.asarray(Kq, dtype=np.float64)
    B, H, n, d = K.shape
    m = Kq.shape[2]
    W = (n + window - 1) // window
    sim = np.zeros((B, W))
    for b in range(B):
        v = Kq[b].mean(axis=1).reshape(-1) if m > 0 else np.zeros(H * d)
        nv = math.sqrt(float(v @ v))
        for w in range(W):
            u = K[b, :, window * w:min(n, window * (w + 1))].mean(axis=1).reshape(-1)
            nu = math.sqrt(float(u @ u))
            sim[b, w] = float(u @ v) / (nu * nv) if nu > 0 and nv > 0 else 0.0
    return sim
