"""kv_window_similarity (CUDA) against the oracle's window_similarity, and the window
plan built from it (WindowQuant note, 何が新しいのか: per-window cosine similarity to
the question picks the bit-width)."""

import numpy as np
import pytest

from bit_kv_cache_28_b300 import bitkv as B
from oracle import window as OW
from helpers import DT, to_dev

pytestmark = pytest.mark.gpu

# fp32 sums of <= 32 tokens and dot products over <= 8192 channels: the cosine is
# within about 1e-6 of the fp64 value; 2e-5 leaves room for the outlier channels
TOL = 2e-5


def keys(rng, B_, H, n, d, dtype, outliers=4):
    K = rng.normal(size=(B_, H, n, d)).astype(np.float32)
    ch = rng.choice(d, size=min(outliers, d), replace=False)
    K[..., ch] *= 8.0
    if dtype == "bf16":
        import torch
        K = torch.from_numpy(K).to(torch.bfloat16).float().numpy()
    elif dtype == "f16":
        K = K.astype(np.float16).astype(np.float32)
    return K


def run(K, Kq, dtype):
    import torch
    B_, H, n, d = K.shape
    m = Kq.shape[2]
    W = (n + 31) // 32
    sim = torch.full((B_, max(W, 1)), 7.0, dtype=torch.float32, device="cuda")
    kd = to_dev(K, dtype)
    qd = to_dev(Kq, dtype) if m > 0 else None
    B.kv_window_similarity(kd, qd, DT[dtype], B_, H, n, m, d, sim)
    torch.cuda.synchronize()
    return sim.cpu().numpy().astype(np.float64)[:, :W]


@pytest.mark.parametrize("B_,H,n,m,d,dtype", [
    (8, 4, 19600, 32, 64, "f16"),     # the decode workload's cache: 613 windows, the last of 16
    (2, 8, 1000, 7, 128, "bf16"),     # 128 threads per CTA (4 warps), last window of 8
    (1, 2, 33, 1, 64, "f32"),         # one full window and one of a single token
    (3, 1, 100, 2, 64, "f16"),        # 8 of a warp's 32 lanes own channels
    (1, 16, 70, 3, 512, "bf16"),      # 1024 threads per CTA, the largest head block
])
def test_window_similarity_matches_oracle(B_, H, n, m, d, dtype):
    rng = np.random.default_rng(n + d)
    K = keys(rng, B_, H, n, d, dtype)
    Kq = keys(rng, B_, H, m, d, dtype)
    # some windows aligned with / against the question, so the extremes are covered
    v = Kq.mean(axis=2, keepdims=True)
    K[:, :, 0:min(32, n)] = v
    if n > 64:
        K[:, :, 32:64] = -2.0 * v
    if dtype == "f16":
        K = K.astype(np.float16).astype(np.float32)
    elif dtype == "bf16":
        import torch
        K = torch.from_numpy(K).to(torch.bfloat16).float().numpy()
    got = run(K, Kq, dtype)
    ref = OW.window_similarity(K, Kq)
    assert got.shape == ref.shape
    err = np.abs(got - ref)
    assert err.max() <= TOL, f"max err {err.max():.3e} at {np.unravel_index(np.argmax(err), err.shape)}"


def test_window_similarity_empty_question_and_zero_windows():
    import torch
    rng = np.random.default_rng(5)
    K = keys(rng, 2, 4, 100, 64, "f16")
    K[:, :, 32:64] = 0.0
    got = run(K, np.zeros((2, 4, 0, 64), np.float32), "f16")
    assert np.all(got == 0.0)
    Kq = keys(rng, 2, 4, 5, 64, "f16")
    got = run(K, Kq, "f16")
    assert np.all(got[:, 1] == 0.0)
    # n == 0 launches nothing and leaves sim as it was
    sim = torch.full((1, 4), 7.0, dtype=torch.float32, device="cuda")
    B.kv_window_similarity(to_dev(K[:, :, :0], "f16"), to_dev(Kq, "f16"), B.KV_F16, 2, 4, 0, 5, 64, sim)
    torch.cuda.synchronize()
    assert np.all(sim.cpu().numpy() == 7.0)


def test_window_plan_from_device_similarity():
    """The decode workload's plan made from the device similarity: where the oracle's
    similarities are further apart than the tolerance at the rank cut-offs, the plan
    (bit-widths and physical order) equals the plan from the oracle's values."""
    rng = np.random.default_rng(4)
    B_, H, n, m, d = 8, 4, 19600, 32, 64
    K = keys(rng, B_, H, n, d, "f16")
    Kq = keys(rng, B_, H, m, d, "f16")
    got = run(K, Kq, "f16")
    ref = OW.window_similarity(K, Kq)
    checked = 0
    for b in range(B_):
        W = got.shape[1]
        bits_ref, perm_ref = OW.window_plan(ref[b].astype(np.float32))
        srt = np.sort(ref[b, 1:].astype(np.float64))[::-1]
        n_rest = W - 1
        cuts = [int(np.floor(0.2 * n_rest)), int(np.floor(0.5 * n_rest))]
        if min(srt[c - 1] - srt[c] for c in cuts) <= 2 * TOL:
            continue                     # a near-tie at a cut-off: either plan is valid
        bits = np.zeros(W, np.int8)
        perm = np.zeros(W, np.int32)
        B.kv_window_plan(np.ascontiguousarray(got[b], dtype=np.float32), W, None, bits, perm)
        assert np.array_equal(bits, bits_ref) and np.array_equal(perm, perm_ref)
        checked += 1
    assert checked >= 4
