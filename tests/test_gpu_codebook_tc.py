"""GPU parity of the tensor-core kernel on codebook (CODEBOOK2) caches against the oracle:
centroid-lookup keys, INT2 values and the rank-r PSAC logit term."""

import numpy as np
import pytest

from bit_kv_cache_28_b300 import bitkv as B
from bit_kv_cache_28_b300 import synth
from oracle import codebook as OC, psac as OP
from oracle import attention as OA
from helpers import run_attention, to_dev, attention_checked, assert_close, tol, TIGHT

pytestmark = pytest.mark.gpu


def oracle_calibrated_cache(case, n, r):
    """Cache on the device with the oracle's centroids and (rank r) PSAC basis, plus the
    oracle's view of the same cache."""
    import torch
    H, d = case["Hkv"], case["d"]
    nb = (n + 31) // 32
    cent = np.stack([OC.fit_centroids(case["K_cache"][0, h, :n]) for h in range(H)])[None]
    U = (np.stack([OP.psac_basis(case["Q_hist"][h], r)[0] for h in range(H)]).astype(np.float32)[None]
         if r else None)
    tc = B.TorchCache(1, H, d, B.KV_CODEBOOK2, (0, 0, nb), raw_dtype=B.KV_BF16, psac_rank=r)
    tc.centroids.copy_(torch.from_numpy(cent.astype(np.float32).reshape(-1)).cuda())
    if r:
        tc.psac_u.copy_(torch.from_numpy(U.reshape(-1)).cuda())
    K, V = case["K_cache"][:, :, :n], case["V_cache"][:, :, :n]
    B.kv_quantize_append(to_dev(K, "bf16"), to_dev(V, "bf16"), B.KV_BF16, n, tc.c)
    oc = OC.build_codebook(K, V, cent, U, nb)
    return tc, oc, U


@pytest.mark.parametrize("path", [B.KV_PATH_TC, B.KV_PATH_TC_SINGLE])
@pytest.mark.parametrize("r", [0, 8, 24, 32])
def test_codebook_tc_small(r, path):
    """Ragged cache (15 blocks, the last partial: tiles of 4, 4, 4, 3 blocks), ragged current
    tile, partial query tile; rank 24 leaves a zero 8-wide chunk in the 32-wide PSAC operand."""
    case = synth.codebook_case(seed=71, H=2, d=128, n_cache=450, n_cur=150, n_hist=128)
    tc, oc, U = oracle_calibrated_cache(case, 450, r)
    for psac in ((0, 1) if r else (0,)):
        args = (oc, case["Q"], case["K_cur"], case["V_cur"], "bf16")
        ref = OA.attention_over_cache(*args, psac_U=U if psac else None)
        tight = OA.attention_over_cache(*args, psac_U=U if psac else None, operand_dtype="f16")
        for splits in (1, 3):
            attention_checked(tc, case, ref, "bf16", tight, psac=psac, path=path, splits=splits)


def test_codebook_tc_matches_simt_and_jensen_has_no_effect():
    """Codebook keys have no step sizes: the Jensen option changes nothing; the tensor-core and
    CUDA-core kernels agree on every row."""
    case = synth.codebook_case(seed=72, H=2, d=128, n_cache=700, n_cur=64, n_hist=64)
    tc, _, _ = oracle_calibrated_cache(case, 700, 8)
    o0, l0 = run_attention(tc, case, psac=1, out_f32=True, path=B.KV_PATH_TC)
    o1, l1 = run_attention(tc, case, psac=1, jensen=1, out_f32=True, path=B.KV_PATH_TC)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    o2, l2 = run_attention(tc, case, psac=1, out_f32=True, path=B.KV_PATH_SIMT)
    assert_close(o0, l0, o2, l2, tol("bf16"))


def test_codebook_workload_tc_sampled():
    """The codebook workload (24 heads, 8192 cached + 1560 current tokens, rank 8) calibrated
    on the device and attended through the dispatch the benchmark uses: sampled rows against
    the oracle given the device calibration, every row against the CUDA-core kernel."""
    import torch
    case = synth.codebook_case()
    H, d, n, r = 24, 128, 8192, 8
    nb = n // 32
    tc = B.TorchCache(1, H, d, B.KV_CODEBOOK2, (0, 0, nb), raw_dtype=B.KV_BF16, psac_rank=r)
    K = to_dev(case["K_cache"], "bf16")
    Qh = to_dev(case["Q_hist"][None], "bf16")
    w = torch.zeros((1, H, d), dtype=torch.float32, device="cuda")
    B.kv_codebook_fit(K, B.KV_BF16, n, tc.c, 20, Qh, 256, w)
    wsb = B.kv_psac_workspace(tc.layout)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    B.kv_psac_basis(Qh, B.KV_BF16, 256, tc.c, None, ws, wsb)
    B.kv_quantize_append(K, to_dev(case["V_cache"], "bf16"), B.KV_BF16, n, tc.c)
    path, _ = B.kv_attention_plan(tc.c, B.KV_BF16, 1560, 1560, H, B.kv_attn_opts(0.0, 0, 1, 0, 0, B.KV_PATH_AUTO))
    assert path == B.KV_PATH_TC
    o_tc, l_tc = run_attention(tc, case, psac=1, out_f32=True)
    o_si, l_si = run_attention(tc, case, psac=1, out_f32=True, path=B.KV_PATH_SIMT)
    assert_close(o_tc, l_tc, o_si, l_si, tol("bf16"))
    cent = tc.centroids.cpu().numpy().reshape(1, H, d, 4)
    U = tc.psac_u.cpu().numpy().reshape(1, H, d, r)
    rows = np.random.default_rng(2).choice(1560, 32, replace=False)
    for h in [0, 13]:
        sl = slice(h, h + 1)
        oc = OC.build_codebook(case["K_cache"][:, sl], case["V_cache"][:, sl], cent[:, sl], U[:, sl], nb)
        args = (oc, case["Q"][:, sl], case["K_cur"][:, sl], case["V_cur"][:, sl], "bf16")
        ref = OA.attention_over_cache(*args, psac_U=U[:, sl], rows=rows)
        tight = OA.attention_over_cache(*args, psac_U=U[:, sl], rows=rows, operand_dtype="f16")
        assert_close(o_tc[:, sl], l_tc[:, sl], ref[0], ref[1], tol("bf16"), rows=rows)
        assert_close(o_tc[:, sl], l_tc[:, sl], tight[0], tight[1], TIGHT, rows=rows)
        assert_close(o_si[:, sl], l_si[:, sl], ref[0], ref[1], TIGHT, rows=rows)
