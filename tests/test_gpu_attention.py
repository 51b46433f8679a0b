"""GPU parity of kv_attention against the oracle (CUDA-core path and dispatch)."""

import numpy as np
import pytest

from bit_kv_cache_28_b300 import bitkv as B
from bit_kv_cache_28_b300 import synth
from oracle import layout as OL, window as OW, codebook as OC, psac as OP
from oracle import attention as OA
from helpers import gpu_uniform, gpu_mixed, run_attention, out_tol, to_dev

pytestmark = pytest.mark.gpu


def check(out, lse, ref_o, ref_lse, dtype, out_f32, rows=None):
    if rows is not None:
        out = out[:, :, rows]
        lse = lse[:, :, rows]
    err = np.abs(out - ref_o)
    tol = out_tol(dtype, out_f32, ref_o)
    worst = np.unravel_index(np.argmax(err - tol), err.shape)
    assert (err <= tol).all(), f"max err {err.max():.3e} at {worst} (tol {tol[worst]:.3e})"
    assert np.abs(lse - ref_lse).max() < 2e-3


def oracle_uniform(case, bits):
    return OL.build_uniform(case["K_cache"], case["V_cache"], bits, case["chunks"],
                            sum((n + 31) // 32 for n in case["chunks"]))


@pytest.mark.parametrize("jensen", [0, 1, 2, 3])
def test_tiny_workload(jensen):
    case = synth.tiny()
    tc = gpu_uniform(case, 2)
    oc = oracle_uniform(case, 2)
    ro, rl = OA.attention_over_cache(oc, case["Q"], case["K_cur"], case["V_cur"], "f32", jensen=jensen)
    for splits in (1, 4):
        o, l = run_attention(tc, case, jensen=jensen, path=B.KV_PATH_SIMT, splits=splits)
        check(o, l, ro, rl, "f32", True)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("jensen", [0, 1, 2, 3])
@pytest.mark.parametrize("out_f32", [True, False])
def test_chunk_small_simt(bits, jensen, out_f32):
    case = synth.chunk_case(51, B=2, Hkv=2, Hq=4, d=128, chunks=[100, 77], n_cur=45, dtype="bf16")
    tc = gpu_uniform(case, bits)
    oc = oracle_uniform(case, bits)
    ro, rl = OA.attention_over_cache(oc, case["Q"], case["K_cur"], case["V_cur"], "bf16", jensen=jensen)
    for splits in (1, 3):
        o, l = run_attention(tc, case, jensen=jensen, out_f32=out_f32, path=B.KV_PATH_SIMT, splits=splits)
        check(o, l, ro, rl, "bf16", out_f32)


@pytest.mark.parametrize("dtype,d", [("f16", 64), ("f32", 32), ("bf16", 256)])
def test_chunk_other_shapes_simt(dtype, d):
    case = synth.chunk_case(52, B=1, Hkv=1, Hq=3, d=d, chunks=[33], n_cur=31, n_q=40, dtype=dtype, sigma=0.3,
                            n_outlier=2, outlier_scale=4.0)
    tc = gpu_uniform(case, 2)
    oc = oracle_uniform(case, 2)
    ro, rl = OA.attention_over_cache(oc, case["Q"], case["K_cur"], case["V_cur"], dtype, jensen=1)
    o, l = run_attention(tc, case, jensen=1, out_f32=True, path=B.KV_PATH_SIMT)
    check(o, l, ro, rl, dtype, True)


def test_empty_cache_and_no_current():
    case = synth.chunk_case(53, B=1, Hkv=2, d=64, chunks=[64], n_cur=20, n_q=7, dtype="f16")
    empty = B.TorchCache(1, 2, 64, B.KV_UNIFORM2, (0, 0, 2))
    o, l = run_attention(empty, case, out_f32=True, path=B.KV_PATH_SIMT)
    oc0 = OL.build_uniform(case["K_cache"][:, :, :0], case["V_cache"][:, :, :0], 2, [], 2)
    ro, rl = OA.attention_over_cache(oc0, case["Q"], case["K_cur"], case["V_cur"], "f16")
    check(o, l, ro, rl, "f16", True)
    tc = gpu_uniform(case, 2)
    oc = oracle_uniform(case, 2)
    z = np.zeros((1, 2, 0, 64), np.float32)
    o, l = run_attention(tc, case, out_f32=True, path=B.KV_PATH_SIMT, Kcur=z, Vcur=z)
    ro, rl = OA.attention_over_cache(oc, case["Q"], z, z, "f16")
    check(o, l, ro, rl, "f16", True)


@pytest.mark.parametrize("n_q", [1, 5])
def test_mixed_simt(n_q):
    case = synth.decode_case(seed=54, B=2, Hq=14, Hkv=2, d=64, n_cache=1000)
    rng = np.random.default_rng(3)
    if n_q > 1:
        case["Q"] = synth.to_dtype_values(rng.standard_normal((2, 14, n_q, 64)), "f16")
    bits = np.stack([OW.window_plan(case["sim"][b])[0] for b in range(2)])
    caps = [int((bits[0] == k).sum()) for k in (16, 4, 2)]
    tc = gpu_mixed(case, bits, caps)
    oc = OL.build_mixed(case["K_cache"], case["V_cache"], bits, caps, "f16")
    for jensen in (0, 1):
        ro, rl = OA.attention_over_cache(oc, case["Q"], case["K_cur"], case["V_cur"], "f16", jensen=jensen)
        o, l = run_attention(tc, case, jensen=jensen, out_f32=True, path=B.KV_PATH_SIMT, splits=3)
        check(o, l, ro, rl, "f16", True)
        o, l = run_attention(tc, case, jensen=jensen, out_f32=False, path=B.KV_PATH_SIMT)
        check(o, l, ro, rl, "f16", False)


def test_codebook_psac_simt():
    import torch
    case = synth.codebook_case(seed=55, H=2, d=128, n_cache=150, n_cur=40, n_hist=64)
    H, d, r = 2, 128, 8
    cent = np.stack([OC.fit_centroids(case["K_cache"][0, h]) for h in range(H)])[None]
    U = np.stack([OP.psac_basis(case["Q_hist"][h], r)[0] for h in range(H)]).astype(np.float32)[None]
    nb = 5
    tc = B.TorchCache(1, H, d, B.KV_CODEBOOK2, (0, 0, nb), raw_dtype=B.KV_BF16, psac_rank=r)
    tc.centroids.copy_(torch.from_numpy(cent.reshape(-1)).cuda())
    tc.psac_u.copy_(torch.from_numpy(U.reshape(-1)).cuda())
    B.kv_quantize_append(to_dev(case["K_cache"], "bf16"), to_dev(case["V_cache"], "bf16"), B.KV_BF16, 150, tc.c)
    oc = OC.build_codebook(case["K_cache"], case["V_cache"], cent, U, nb)
    for psac in (0, 1):
        ro, rl = OA.attention_over_cache(oc, case["Q"], case["K_cur"], case["V_cur"], "bf16",
                                         psac_U=U if psac else None)
        o, l = run_attention(tc, case, psac=psac, out_f32=True, path=B.KV_PATH_SIMT, splits=2)
        check(o, l, ro, rl, "bf16", True)


def test_chunk_workload_simt_sampled():
    """Full chunk workload (24 heads, 4680 cached + 1560 current), sampled rows vs the oracle."""
    case = synth.chunk()
    tc = gpu_uniform(case, 2)
    oc = oracle_uniform(case, 2)
    rows = np.random.default_rng(0).choice(1560, 48, replace=False)
    heads = [0, 7, 23]
    o, l = run_attention(tc, case, jensen=1, out_f32=True, path=B.KV_PATH_SIMT)
    # evaluate the oracle per head through a one-head view of the cache
    for h in heads:
        view = OL.Cache(1, 1, 128, oc.classes, oc.caps)
        view.blocks = [[oc.blocks[0][h]]]
        ro, rl = OA.attention_over_cache(view, case["Q"][:, h:h + 1], case["K_cur"][:, h:h + 1],
                                         case["V_cur"][:, h:h + 1], "bf16", jensen=1, rows=rows)
        check(o[:, h:h + 1], l[:, h:h + 1], ro, rl, "bf16", True, rows=rows)


# ------------------------------------------------------ tensor-core path -----

@pytest.mark.parametrize("jensen", [2, 1])
def test_tc_repeated_runs_identical(jensen):
    """tcgen05 kernel: 200 repeated calls on one input give bit-identical outputs within the
    oracle's tolerance.  The EXACT softmax is slow, so Q K^T of tile j and P V of tile j - 2
    (which share TMEM columns) are issued back to back; an ordering race between them showed
    as an occasional wrong output here."""
    case = synth.chunk_case(61, B=2, Hkv=2, Hq=4, d=128, chunks=[300, 77], n_cur=150, n_q=150, dtype="bf16")
    tc = gpu_uniform(case, 2)
    oc = oracle_uniform(case, 2)
    ro, rl = OA.attention_over_cache(oc, case["Q"], case["K_cur"], case["V_cur"], "bf16", jensen=jensen)
    for splits in (3, 1):
        first = None
        for _ in range(200):
            o, l = run_attention(tc, case, jensen=jensen, out_f32=True, path=B.KV_PATH_TC, splits=splits)
            if first is None:
                check(o, l, ro, rl, "bf16", True)
                first = (o, l)
            else:
                assert np.array_equal(o, first[0]) and np.array_equal(l, first[1])


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("jensen", [0, 1, 2, 3])
def test_chunk_small_tc(bits, jensen):
    """tcgen05 kernel: ragged cache blocks, ragged current tile, partial query tile, GQA."""
    case = synth.chunk_case(61, B=2, Hkv=2, Hq=4, d=128, chunks=[300, 77], n_cur=150, n_q=150, dtype="bf16")
    tc = gpu_uniform(case, bits)
    oc = oracle_uniform(case, bits)
    ro, rl = OA.attention_over_cache(oc, case["Q"], case["K_cur"], case["V_cur"], "bf16", jensen=jensen)
    for splits in (1, 3):
        for out_f32 in (True, False):
            o, l = run_attention(tc, case, jensen=jensen, out_f32=out_f32, path=B.KV_PATH_TC, splits=splits)
            check(o, l, ro, rl, "bf16", out_f32)


def test_tc_only_current_or_only_cache():
    case = synth.chunk_case(62, B=1, Hkv=2, d=128, chunks=[200], n_cur=130, n_q=64, dtype="bf16")
    empty = B.TorchCache(1, 2, 128, B.KV_UNIFORM2, (0, 0, 8))
    oc0 = OL.build_uniform(case["K_cache"][:, :, :0], case["V_cache"][:, :, :0], 2, [], 8)
    ro, rl = OA.attention_over_cache(oc0, case["Q"], case["K_cur"], case["V_cur"], "bf16")
    o, l = run_attention(empty, case, out_f32=True, path=B.KV_PATH_TC)
    check(o, l, ro, rl, "bf16", True)
    tc = gpu_uniform(case, 2)
    oc = oracle_uniform(case, 2)
    z = np.zeros((1, 2, 0, 128), np.float32)
    ro, rl = OA.attention_over_cache(oc, case["Q"], z, z, "bf16", jensen=1)
    o, l = run_attention(tc, case, out_f32=True, jensen=1, path=B.KV_PATH_TC, Kcur=z, Vcur=z)
    check(o, l, ro, rl, "bf16", True)


@pytest.mark.parametrize("jensen", [0, 1])
def test_chunk_workload_tc_sampled(jensen):
    """Full chunk workload through the dispatch the benchmark uses: sampled rows vs the oracle,
    and every row vs the CUDA-core kernel."""
    case = synth.chunk()
    tc = gpu_uniform(case, 2)
    oc = oracle_uniform(case, 2)
    o_tc, l_tc = run_attention(tc, case, jensen=jensen, out_f32=True)              # auto path
    o_bf, _ = run_attention(tc, case, jensen=jensen, out_f32=False)
    o_si, l_si = run_attention(tc, case, jensen=jensen, out_f32=True, path=B.KV_PATH_SIMT)
    assert np.abs(o_tc - o_si).max() < 2e-3 and np.abs(l_tc - l_si).max() < 2e-3
    rows = np.random.default_rng(1).choice(1560, 40, replace=False)
    for h in [0, 11, 23]:
        view = OL.Cache(1, 1, 128, oc.classes, oc.caps)
        view.blocks = [[oc.blocks[0][h]]]
        ro, rl = OA.attention_over_cache(view, case["Q"][:, h:h + 1], case["K_cur"][:, h:h + 1],
                                         case["V_cur"][:, h:h + 1], "bf16", jensen=jensen, rows=rows)
        check(o_tc[:, h:h + 1], l_tc[:, h:h + 1], ro, rl, "bf16", True, rows=rows)
        check(o_bf[:, h:h + 1], l_tc[:, h:h + 1], ro, rl, "bf16", False, rows=rows)
