"""Pins for the oracle's window plan, layout builders, k-means codebook and PSAC basis."""

import itertools
import json
import os

import numpy as np
import pytest
from scipy.cluster.vq import kmeans2

from oracle import window, layout, codebook, psac, quant
from oracle import attention as A
from bit_kv_cache_28_b300 import synth

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")))


@pytest.mark.parametrize("case", GOLD["window_plan"])
def test_window_plan_hand(case):
    bits, perm = window.window_plan(case["sim"], case["frac16"], case["frac4"])
    assert bits.tolist() == case["bits"] and perm.tolist() == case["perm"]


def test_window_plan_counts_decode_workload():
    c = synth.decode_case()
    W = c["sim"].shape[1]
    assert W == 613
    for b in range(8):
        bits, perm = window.window_plan(c["sim"][b])
        assert bits[0] == 16
        assert [(bits == k).sum() for k in (16, 4, 2)] == [123, 184, 306]
        assert sorted(perm.tolist()) == list(range(W))
        # relevance order: every FP16 window (except 0) has sim >= every INT4 >= every INT2
        s = c["sim"][b]
        f16 = [w for w in range(1, W) if bits[w] == 16]
        assert s[f16].min() >= s[bits == 4].max() >= s[bits == 2].max()


def test_window_plan_unforced_and_degenerate():
    bits, perm = window.window_plan([0.1, 0.9], 0.5, 0.5, force_first=False)
    assert bits.tolist() == [4, 16]
    bits, _ = window.window_plan([0.3], 0.2, 0.3)
    assert bits.tolist() == [16]
    bits, perm = window.window_plan([], 0.2, 0.3)
    assert bits.size == 0 and perm.size == 0


def test_window_similarity_closed_forms():
    """Cosine of window means to the question mean (WindowQuant note, 何が新しいのか):
    a window along the question gives 1, against it -1, orthogonal to it 0; a zero
    window or an empty question gives 0."""
    rng = np.random.default_rng(11)
    H, d, m = 2, 4, 3
    Kq = rng.normal(size=(1, H, m, d))
    v = Kq[0].mean(axis=1)                                   # [H, d]
    vf = v.reshape(-1)
    r = rng.normal(size=H * d)
    orth = (r - (r @ vf) / (vf @ vf) * vf).reshape(H, d)     # Gram-Schmidt: orth . v = 0
    n = 5 * 32 + 7
    K = rng.normal(size=(1, H, n, d))
    K[0, :, 0:32] = 2.5 * v[:, None, :]
    K[0, :, 32:64] = -0.1 * v[:, None, :]
    K[0, :, 64:96] = orth[:, None, :]
    K[0, :, 96:128] = 0.0
    # window 4: tokens whose deviations from 3 v cancel over the window
    dev = rng.normal(size=(H, 16, d))
    K[0, :, 128:160] = 3.0 * v[:, None, :] + np.concatenate([dev, -dev], axis=1)
    K[0, :, 160:] = -v[:, None, :] + 0.0                      # partial window of 7 tokens
    sim = window.window_similarity(K, Kq)
    assert sim.shape == (1, 6)
    assert abs(sim[0, 0] - 1.0) < 1e-12 and abs(sim[0, 1] + 1.0) < 1e-12
    assert abs(sim[0, 2]) < 1e-12 and sim[0, 3] == 0.0
    assert abs(sim[0, 4] - 1.0) < 1e-12 and abs(sim[0, 5] + 1.0) < 1e-12
    assert np.all(window.window_similarity(K, Kq[:, :, :0]) == 0.0)


def test_window_similarity_library_and_symmetries():
    """Against scipy's cosine distance on the concatenated means; invariant to positive
    scalings, token order inside a window and a common permutation of the kv heads;
    odd in the question."""
    from scipy.spatial.distance import cosine
    rng = np.random.default_rng(12)
    B, H, n, m, d = 2, 3, 3 * 32 + 10, 5, 8
    K = rng.normal(size=(B, H, n, d))
    K[:, :, :, 2] *= 8.0                                      # an outlier channel
    Kq = rng.normal(size=(B, H, m, d))
    sim = window.window_similarity(K, Kq)
    for b in range(B):
        v = Kq[b].mean(axis=1).reshape(-1)
        for w in range(sim.shape[1]):
            u = K[b, :, 32 * w:32 * w + 32].mean(axis=1).reshape(-1)
            assert abs(sim[b, w] - (1.0 - cosine(u, v))) < 1e-12
    assert np.allclose(window.window_similarity(3.0 * K, 0.5 * Kq), sim, atol=1e-12)
    assert np.allclose(window.window_similarity(K, -Kq), -sim, atol=1e-12)
    Kp = K.copy()
    Kp[:, :, 32:64] = K[:, :, 32:64][:, :, rng.permutation(32)]
    assert np.allclose(window.window_similarity(Kp, Kq), sim, atol=1e-12)
    hp = [2, 0, 1]
    assert np.allclose(window.window_similarity(K[:, hp], Kq[:, hp]), sim, atol=1e-12)


def test_block_bytes():
    assert layout.block_bytes(layout.INT2, 128) == 4096
    assert layout.block_bytes(layout.INT4, 128) == 6144
    assert layout.block_bytes(layout.RAW16, 64) == 8192
    assert layout.block_bytes(layout.INT2, 64) == 2048
    assert layout.block_bytes(layout.INT4, 64) == 3072
    assert layout.block_bytes(layout.CB2, 128, 8) == 1024 + 1024 + 1024 + 512


def test_uniform_builder_chunk_alignment_and_bytes():
    c = synth.chunk_case(7, Hkv=2, d=64, chunks=[50, 40], n_cur=8, n_q=8)
    cache = layout.build_uniform(c["K_cache"], c["V_cache"], 2, [50, 40], 8)
    assert cache.n_blocks == [4]
    assert cache.blk_len[0, :4].tolist() == [32, 18, 32, 8]
    assert cache.blk_pos[0, :4].tolist() == [0, 32, 50, 82]
    # the block of tokens 50..81 is quantised on its own (chunk-aligned group)
    bb = layout.block_bytes(layout.INT2, 64)
    raw = cache.data[0, 1, 2 * bb:3 * bb]
    kc = quant.unpack_codes(raw[:512].view(np.uint32).reshape(32, 4), 2, 64)
    km = raw[512:1024].view(np.float32).reshape(64, 2)
    K = c["K_cache"][0, 1, 50:82]
    codes, s, z = quant.quantize_groups(K.T, 2)
    assert (kc == codes.T).all() and (km[:, 0] == s).all() and (km[:, 1] == z).all()
    # pad slots of the 18-token block are zero
    raw1 = cache.data[0, 0, bb:2 * bb]
    vm = raw1[1536:2048].view(np.float32).reshape(2, 32, 2)     # [group][token][s,z]
    assert (vm[:, 18:] == 0).all() and (vm[:, :18, 0] > 0).all()
    vc = quant.unpack_codes(raw1[1024:1536].view(np.uint32).reshape(64, 2), 2, 32)   # [channel][token]
    V = c["V_cache"][0, 0, 32:50]
    codes_v, _, _ = quant.quantize_groups(V.reshape(18, 2, 32), 2)
    assert (vc[:, :18] == codes_v.reshape(18, 64).T).all() and (vc[:, 18:] == 0).all()
    lg = cache.logical(0, 1)
    assert lg["khat"].shape == (90, 64)


@pytest.mark.parametrize("d", [32, 64, 128])
def test_raw16_chunk_permutation(d):
    """RAW16 rows: element (t, c) sits at 16-bit slot t*d + 8*((c//8) ^ (t % m)) + c % 8, m = min(8, d/8),
    written out element by element from the format definition."""
    rng = np.random.default_rng(5)
    K = synth.to_dtype_values(rng.standard_normal((1, 32, d)), "f16")
    V = synth.to_dtype_values(rng.standard_normal((1, 32, d)), "f16")
    enc = layout.encode_raw_blocks(K, V, 30, "f16")
    words = enc["bytes"][0].view(np.float16)
    m = min(8, d // 8)
    for part, X in ((0, K[0]), (1, V[0])):
        for t in range(32):
            for c in range(d):
                slot = part * 32 * d + t * d + 8 * ((c // 8) ^ (t % m)) + c % 8
                want = X[t, c] if t < 30 else 0.0
                assert float(words[slot]) == want
    # for d >= 64, eight consecutive rows of one chunk column land in eight distinct
    # 16-byte bank groups of a 128-byte bank line
    if d >= 64:
        order = layout.raw16_chunk_order(d)
        for j in range(d // 8):
            banks = {((t * 2 * d + 16 * order[t, j]) % 128) // 16 for t in range(8)}
            assert len(banks) == 8


def test_bytes_of_workloads():
    """Algorithmic cache bytes (codes of valid tokens + all metadata) of the chunk workload."""
    H, d, n = 24, 128, 4680
    codes = H * n * d * 2 * 2 / 8
    meta = H * (3 * 49) * d * 8 + H * n * (d // 32) * 8
    assert abs((codes + meta) / 1e6 - 14.40) < 0.01


# ---------------------------------------------------------------- k-means -----

def test_kmeans_hand():
    case = GOLD["kmeans"][0]
    mu = codebook.kmeans_1d(np.array(case["x"], float))
    assert mu.tolist() == case["centroids"]


def test_kmeans_fixed_point_and_library():
    rng = np.random.default_rng(0)
    x = synth.to_bf16_values(rng.standard_normal(4096)).astype(np.float64)
    mu = codebook.kmeans_1d(x, 4, 50)
    a = codebook.nearest(x, mu)
    for j in range(4):
        assert mu[j] == pytest.approx(x[a == j].mean(), abs=1e-15)
    # scipy's Lloyd from the same start agrees on data without ties
    xs = np.sort(x)
    init = np.array([xs[(2 * j + 1) * 4096 // 8] for j in range(4)])
    cen, lab = kmeans2(x[:, None], init[:, None], iter=20, minit="matrix")
    mu20 = codebook.kmeans_1d(x, 4, 20)
    assert np.abs(cen[:, 0] - mu20).max() < 1e-12


def test_kmeans_brute_force_small():
    """For n <= 10 the Lloyd result's objective is >= the best contiguous partition and
    satisfies the local optimality conditions exactly."""
    rng = np.random.default_rng(1)
    for trial in range(20):
        n = int(rng.integers(5, 11))
        x = np.round(rng.standard_normal(n) * 4, 2)
        mu = codebook.kmeans_1d(x, 4, 20)
        a = codebook.nearest(x, mu)
        obj = ((x - mu[a]) ** 2).sum()
        xs = np.sort(x)
        best = np.inf
        for cuts in itertools.combinations(range(1, n), 3):
            parts = np.split(xs, cuts)
            best = min(best, sum(((p - p.mean()) ** 2).sum() for p in parts))
        assert obj >= best - 1e-12
        for j in range(4):
            if (a == j).any():
                assert abs(mu[j] - x[a == j].mean()) < 1e-12


def test_sensitivity_weight_cancels():
    """A per-channel constant weight changes no weighted mean: weighted Lloyd equals plain Lloyd."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal(300)
    w = 3.7
    mu = codebook.kmeans_1d(x)
    a = codebook.nearest(x, mu)
    for j in range(4):
        m = x[a == j]
        assert abs((w * m).sum() / (w * len(m)) - mu[j]) < 1e-12
    Qh = rng.standard_normal((256, 8))
    assert np.allclose(codebook.sensitivity(Qh), (Qh ** 2).mean(0))


# ---------------------------------------------------------------- PSAC --------

def test_psac_full_rank_reproduces_keys():
    rng = np.random.default_rng(3)
    d = 16
    Qh = rng.standard_normal((256, d)) * np.exp(rng.standard_normal(d))
    U, w = psac.psac_basis(Qh, d)
    assert np.abs(U.T @ U - np.eye(d)).max() < 1e-12
    K = rng.standard_normal((10, d))
    cent = codebook.fit_centroids(K, 5)
    idx = np.stack([codebook.nearest(K[:, c], cent[c]) for c in range(d)], 1)
    Khat = cent[np.arange(d)[None], idx]
    coeff64 = (K - Khat) @ U
    comp = Khat + coeff64 @ U.T
    assert np.abs(comp - K).max() < 1e-12
    q = rng.standard_normal(d)
    tau = 0.25
    lg = tau * Khat @ q + tau * coeff64 @ (U.T @ q)
    assert np.abs(lg - tau * K @ q).max() < 1e-10
    # with fp16 coefficients the error is bounded by the fp16 rounding
    c16 = psac.psac_coeff(K, Khat, U).astype(np.float64)
    lg16 = tau * Khat @ q + tau * c16 @ (U.T @ q)
    bound = tau * np.abs(U.T @ q).sum() * np.abs(coeff64).max() * 2 ** -11
    assert np.abs(lg16 - tau * K @ q).max() <= bound


def test_psac_eigen_and_signs():
    rng = np.random.default_rng(4)
    d = 12
    scales = np.array([5, 1, 7, 0.5, 3, 2, 0.1, 4, 6, 0.2, 0.3, 8.0])
    Qh = rng.standard_normal((20000, d)) * scales
    C = psac.second_moment(Qh)
    U, w = psac.psac_basis(Qh, 4)
    assert np.abs(C @ U - U * w).max() < 1e-9 * w.max()
    assert (np.diff(w) <= 0).all()
    for j in range(4):
        assert U[np.argmax(np.abs(U[:, j])), j] > 0
    # nearly diagonal covariance: the top vectors are the largest-scale axes
    axes = [int(np.argmax(np.abs(U[:, j]))) for j in range(4)]
    assert axes == [11, 2, 8, 0]


def test_psac_rank_zero_is_plain_codebook():
    c = synth.codebook_case(seed=9, H=1, d=32, n_cache=70, n_cur=5, n_hist=16)
    cent = codebook.fit_centroids(c["K_cache"][0, 0])[None, None]
    cache0 = codebook.build_codebook(c["K_cache"], c["V_cache"], cent, None, 4)
    o0, _ = A.attention_over_cache(cache0, c["Q"], c["K_cur"], c["V_cur"], "bf16")
    lg = cache0.logical(0, 0)
    Kc = np.asarray(lg["khat"], np.float64)
    Vc = np.asarray(lg["vhat"], np.float64)
    o_ref, _ = A.attention_rows(c["Q"][0, 0], Kc, Vc, c["K_cur"][0, 0], c["V_cur"][0, 0], 1 / np.sqrt(32))
    assert np.abs(o0[0, 0] - o_ref).max() == 0
    U, _ = psac.psac_basis(c["Q_hist"][0], 4)
    U32 = U.astype(np.float32)[None, None]
    cache4 = codebook.build_codebook(c["K_cache"], c["V_cache"], cent, U32, 4)
    o4, _ = A.attention_over_cache(cache4, c["Q"], c["K_cur"], c["V_cur"], "bf16", psac_U=U32)
    assert np.abs(o4 - o0).max() > 0
