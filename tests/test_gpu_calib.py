"""GPU parity of the codebook-cache calibration calls against the oracle.

kv_codebook_fit: per-(head, channel) 1-D Lloyd k-means of the cached keys (QSAC
reading) -- centroids bit-exact, sensitivity weights bit-exact.
kv_psac_basis: top-r eigenvectors of the historical queries' second moment (PSAC
reading) -- same vectors and signs up to fp64 round-off, eigenvalues to fp32.
"""

import numpy as np
import pytest

from bit_kv_cache_28_b300 import bitkv as B
from bit_kv_cache_28_b300 import synth
from oracle import codebook as OC, psac as OP, attention as OA
from helpers import to_dev, run_attention, assert_close, TIGHT

pytestmark = pytest.mark.gpu


def fit_on_device(case, n, r=0, n_hist=None):
    import torch
    H, d = case["Hkv"], case["d"]
    nb = (n + 31) // 32
    tc = B.TorchCache(1, H, d, B.KV_CODEBOOK2, (0, 0, nb), raw_dtype=B.KV_BF16, psac_rank=r)
    K = to_dev(case["K_cache"][:, :, :n], "bf16")
    Qh = to_dev(case["Q_hist"][None], "bf16") if n_hist else None
    w = torch.zeros((1, H, d), dtype=torch.float32, device="cuda")
    B.kv_codebook_fit(K, B.KV_BF16, n, tc.c, 20, Qh, n_hist or 0, w if n_hist else None)
    eig = None
    if r:
        eig = torch.zeros((1, H, r), dtype=torch.float32, device="cuda")
        wsb = B.kv_psac_workspace(tc.layout)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        B.kv_psac_basis(Qh, B.KV_BF16, n_hist, tc.c, eig, ws, wsb)
    torch.cuda.synchronize()
    return tc, w, eig


def test_codebook_fit_bit_exact_small():
    case = synth.codebook_case(seed=91, H=3, d=128, n_cache=700, n_cur=8, n_hist=64)
    tc, w, _ = fit_on_device(case, 700, n_hist=64)
    cent = tc.centroids.cpu().numpy().reshape(3, 128, 4)
    for h in range(3):
        ref = OC.fit_centroids(case["K_cache"][0, h])
        assert np.array_equal(cent[h], ref), f"head {h}: {np.abs(cent[h] - ref).max()}"
    ref_w = np.stack([OC.sensitivity(case["Q_hist"][h]) for h in range(3)]).astype(np.float32)
    assert np.array_equal(w.cpu().numpy()[0], ref_w)


def test_codebook_fit_workload_sampled():
    """24 heads x 8192 cached keys: every head's centroids on the device, a sample against the oracle."""
    case = synth.codebook_case()
    tc, _, _ = fit_on_device(case, 8192)
    cent = tc.centroids.cpu().numpy().reshape(24, 128, 4)
    rng = np.random.default_rng(0)
    for h, c in zip(rng.choice(24, 6, replace=False), rng.choice(128, 6, replace=False)):
        ref = OC.kmeans_1d(case["K_cache"][0, h, :, c]).astype(np.float32)
        assert np.array_equal(cent[h, c], ref), (h, c, cent[h, c], ref)


@pytest.mark.parametrize("r", [8, 32])
def test_psac_basis_matches_oracle(r):
    case = synth.codebook_case(seed=92, H=2, d=128, n_cache=64, n_cur=8, n_hist=256)
    tc, _, eig = fit_on_device(case, 64, r=r, n_hist=256)
    U = tc.psac_u.cpu().numpy().reshape(2, 128, r).astype(np.float64)
    for h in range(2):
        Ur, wr = OP.psac_basis(case["Q_hist"][h], r)
        dots = np.einsum("dk,dk->k", U[h], Ur)
        assert (dots > 1 - 1e-5).all(), dots.min()
        assert np.allclose(eig.cpu().numpy()[0, h], wr, rtol=1e-6, atol=1e-7)
        # orthonormal columns
        assert np.abs(U[h].T @ U[h] - np.eye(r)).max() < 1e-5


def test_codebook_calibration_chain():
    """Centroids and PSAC basis fitted on the device, then append and attention with PSAC,
    against the oracle given the same calibration."""
    import torch
    case = synth.codebook_case(seed=93, H=2, d=128, n_cache=300, n_cur=40, n_hist=128)
    tc, _, _ = fit_on_device(case, 300, r=8, n_hist=128)
    B.kv_quantize_append(to_dev(case["K_cache"], "bf16"), to_dev(case["V_cache"], "bf16"), B.KV_BF16, 300, tc.c)
    cent = tc.centroids.cpu().numpy().reshape(1, 2, 128, 4)
    U = tc.psac_u.cpu().numpy().reshape(1, 2, 128, 8)
    oc = OC.build_codebook(case["K_cache"], case["V_cache"], cent, U, 10)
    assert np.array_equal(tc.data.cpu().numpy().reshape(oc.data.shape), oc.data)
    ro, rl = OA.attention_over_cache(oc, case["Q"], case["K_cur"], case["V_cur"], "bf16", psac_U=U)
    o, l = run_attention(tc, case, psac=1, out_f32=True, path=B.KV_PATH_SIMT)
    assert_close(o, l, ro, rl, TIGHT)      # the CUDA-core path computes the definition
