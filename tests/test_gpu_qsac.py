"""GPU parity of the QSAC-with-residual-range fit, the residual variances and the Jensen term of
codebook keys (with and without PSAC) against the oracle.

QuantWM (Innovations 2, 3): the clustering weighs the historical queries' sensitivity with the
range of the residuals; PSAC restores the key error along the dominant query subspace.  The
fit's centroids and weights must be bit-exact; the residual variances within fp32 rounding
of a different summation order; attention within the bounds of the other attention tests."""

import numpy as np
import pytest

from bit_kv_cache_28_b300 import bitkv as B
from bit_kv_cache_28_b300 import synth
from oracle import codebook as OC, psac as OP, attention as OA
from helpers import to_dev, attention_checked, run_attention, assert_close, tol, TIGHT

pytestmark = pytest.mark.gpu


def calibrated(case, n, r, n_hist, range_fit=True):
    """Device calibration of a codebook cache: fit (residual-range or Lloyd), PSAC basis,
    residual variances, then the append of the n cached tokens."""
    import torch
    H, d = case["Hkv"], case["d"]
    nb = (n + 31) // 32
    tc = B.TorchCache(1, H, d, B.KV_CODEBOOK2, (0, 0, nb), raw_dtype=B.KV_BF16, psac_rank=r, resid_var=True)
    K = to_dev(case["K_cache"][:, :, :n], "bf16")
    Qh = to_dev(case["Q_hist"][None], "bf16")
    w = torch.zeros((1, H, d), dtype=torch.float32, device="cuda")
    if range_fit:
        B.kv_codebook_fit_range(K, B.KV_BF16, n, tc.c, 20, Qh, n_hist, w)
    else:
        B.kv_codebook_fit(K, B.KV_BF16, n, tc.c, 20, Qh, n_hist, w)
    if r:
        wsb = B.kv_psac_workspace(tc.layout)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        B.kv_psac_basis(Qh, B.KV_BF16, n_hist, tc.c, None, ws, wsb)
    B.kv_codebook_residual_var(K, B.KV_BF16, n, tc.c)
    B.kv_quantize_append(K, to_dev(case["V_cache"][:, :, :n], "bf16"), B.KV_BF16, n, tc.c)
    torch.cuda.synchronize()
    cent = tc.centroids.cpu().numpy().reshape(1, H, d, 4)
    U = tc.psac_u.cpu().numpy().reshape(1, H, d, r) if r else None
    var = tc.resid_var.cpu().numpy().reshape(1, H, d)
    return tc, w.cpu().numpy().reshape(1, H, d), cent, U, var


def test_range_fit_bit_exact_and_weights_act():
    case = synth.codebook_case(seed=101, H=3, d=128, n_cache=700, n_cur=8, n_hist=64)
    _, w, cent, _, var = calibrated(case, 700, 0, 64)
    changed = 0
    for h in range(3):
        w32 = OC.sensitivity_f32(case["Q_hist"][h])
        assert np.array_equal(w[0, h], w32)
        ref = OC.fit_centroids_range(case["K_cache"][0, h], w32)
        assert np.array_equal(cent[0, h], ref), f"head {h}: {np.abs(cent[0, h] - ref).max()}"
        changed += int((ref != OC.fit_centroids(case["K_cache"][0, h])).any(axis=1).sum())
        v = OC.residual_var(case["K_cache"][0, h], cent[0, h])
        assert np.allclose(var[0, h], v, rtol=1e-6, atol=0)
    assert changed > 100           # the sensitivity moves most channels' centroids


def test_range_fit_workload_sampled():
    """The codebook workload (24 heads x 8192 keys, 256 historical queries): sampled channels."""
    case = synth.codebook_case()
    _, w, cent, _, _ = calibrated(case, 8192, 0, 256)
    rng = np.random.default_rng(1)
    for h in rng.choice(24, 4, replace=False):
        w32 = OC.sensitivity_f32(case["Q_hist"][h])
        assert np.array_equal(w[0, h], w32)
        rho = OC.relative_sensitivity(w32)
        for c in rng.choice(128, 4, replace=False):
            ref = OC.kmeans_1d_range(case["K_cache"][0, h, :, c], rho[c]).astype(np.float32)
            assert np.array_equal(cent[0, h, c], ref), (h, c)


@pytest.mark.parametrize("r", [0, 8])
@pytest.mark.parametrize("jensen", [1, 3])
def test_codebook_jensen_tc_and_simt(r, jensen):
    """Ragged cache (450 tokens: tiles of 4, 4, 4, 3 blocks), ragged current tile, partial query
    tile; the Jensen term of codebook keys with and without the PSAC projection."""
    case = synth.codebook_case(seed=102, H=2, d=128, n_cache=450, n_cur=150, n_hist=128)
    tc, _, cent, U, var = calibrated(case, 450, r, 128)
    oc = OC.build_codebook(case["K_cache"], case["V_cache"], cent, U, 15, resid_var=var)
    for psac in ((0, 1) if r else (0,)):
        args = (oc, case["Q"], case["K_cur"], case["V_cur"], "bf16")
        kw = dict(jensen=jensen, psac_U=U if psac else None)
        ref = OA.attention_over_cache(*args, **kw)
        tight = OA.attention_over_cache(*args, operand_dtype="f16", **kw)
        for splits in (1, 3):
            attention_checked(tc, case, ref, "bf16", tight, jensen=jensen, psac=psac, path=B.KV_PATH_TC,
                              splits=splits)
        attention_checked(tc, case, ref, "bf16", ref, jensen=jensen, psac=psac, path=B.KV_PATH_SIMT, splits=2)
        # the term is there: without it the lse is higher
        off = OA.attention_over_cache(*args, psac_U=U if psac else None)
        assert (off[1] > ref[1]).all()


def test_codebook_exact_jensen_is_rejected():
    case = synth.codebook_case(seed=103, H=1, d=128, n_cache=64, n_cur=16, n_hist=32)
    tc, _, _, _, _ = calibrated(case, 64, 0, 32)
    with pytest.raises(B.BitKVError) as e:
        run_attention(tc, case, jensen=2, out_f32=True, path=B.KV_PATH_TC)
    assert e.value.status == B.KV_ERR_UNSUPPORTED


def test_codebook_workload_range_fit_jensen_psac_sampled():
    """The codebook workload calibrated on the device with the residual-range fit, rank-8 PSAC
    and the Jensen term, through the dispatch the benchmark uses: sampled rows of two heads
    against the oracle given the device calibration, every row against the CUDA-core kernel."""
    case = synth.codebook_case()
    tc, _, cent, U, var = calibrated(case, 8192, 8, 256)
    path, _ = B.kv_attention_plan(tc.c, B.KV_BF16, 1560, 1560, 24, B.kv_attn_opts(0.0, 1, 1, 0, 0, B.KV_PATH_AUTO))
    assert path == B.KV_PATH_TC
    o_tc, l_tc = run_attention(tc, case, jensen=1, psac=1, out_f32=True)
    o_si, l_si = run_attention(tc, case, jensen=1, psac=1, out_f32=True, path=B.KV_PATH_SIMT)
    assert_close(o_tc, l_tc, o_si, l_si, tol("bf16"))
    rows = np.random.default_rng(3).choice(1560, 32, replace=False)
    for h in [4, 17]:
        sl = slice(h, h + 1)
        oc = OC.build_codebook(case["K_cache"][:, sl], case["V_cache"][:, sl], cent[:, sl], U[:, sl], 256,
                               resid_var=var[:, sl])
        args = (oc, case["Q"][:, sl], case["K_cur"][:, sl], case["V_cur"][:, sl], "bf16")
        ref = OA.attention_over_cache(*args, jensen=1, psac_U=U[:, sl], rows=rows)
        tight = OA.attention_over_cache(*args, jensen=1, psac_U=U[:, sl], rows=rows, operand_dtype="f16")
        assert_close(o_tc[:, sl], l_tc[:, sl], ref[0], ref[1], tol("bf16"), rows=rows)
        assert_close(o_tc[:, sl], l_tc[:, sl], tight[0], tight[1], TIGHT, rows=rows)
        assert_close(o_si[:, sl], l_si[:, sl], ref[0], ref[1], TIGHT, rows=rows)
