"""GPU parity of the split-K decode kernel (one query per sequence) against the oracle.

The decode kernel never forms dequantised 16-bit key or value tiles: it folds the
step sizes and zero points into the query (fp16 high + low parts, ~22 bits) and the
attention weights, so it is held to 2e-3 against the oracle's definition itself (inside
the required 1e-2 for its 16-bit I/O); its 16-bit outputs must be the rounding of the
fp32 result.
"""

import numpy as np
import pytest

from bit_kv_cache_28_b300 import bitkv as B
from bit_kv_cache_28_b300 import synth
from oracle import layout as OL, window as OW
from oracle import attention as OA
from helpers import gpu_mixed, gpu_uniform, run_attention, assert_close, assert_rounding_of, TIGHT

pytestmark = pytest.mark.gpu


def check(out, lse, ref_o, ref_lse):
    assert_close(out, lse, ref_o, ref_lse, TIGHT)


def mixed_case(case, frac16=0.2, frac4=0.3):
    bits = np.stack([OW.window_plan(case["sim"][b], frac16, frac4)[0] for b in range(case["B"])])
    caps = [int((bits[0] == k).sum()) for k in (16, 4, 2)]
    tc = gpu_mixed(case, bits, caps)
    oc = OL.build_mixed(case["K_cache"], case["V_cache"], bits, caps, case["dtype"])
    return tc, oc


def test_decode_workload_full():
    """Batch 8, 28 query heads over 4 kv heads, d 64, 19600 cached tokens in 613 windows
    (FP16 / INT4 / INT2 by similarity), fp16: every output row against the oracle.  The
    automatic split count spreads one wave of resident CTAs over the 32 streams, so streams
    take different split counts; the two uniform counts around it are checked as well."""
    case = synth.decode_case()
    tc, oc = mixed_case(case)
    path, splits = B.kv_attention_plan(tc.c, B.KV_F16, 1, 1, 28)
    assert path == B.KV_PATH_DECODE and splits > 1
    for jensen in (0, 1, 3):
        ro, rl = OA.attention_over_cache(oc, case["Q"], case["K_cur"], case["V_cur"], "f16", jensen=jensen)
        o, l = run_attention(tc, case, jensen=jensen, out_f32=True)
        check(o, l, ro, rl)
        o16, l16 = run_attention(tc, case, jensen=jensen, out_f32=False)
        assert_rounding_of(o16, o, "f16")
        if jensen == 1:
            for sp in (splits - 1, splits):
                o, l = run_attention(tc, case, jensen=jensen, out_f32=True, path=B.KV_PATH_DECODE, splits=sp)
                check(o, l, ro, rl)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("n_cur", [0, 1, 5])
def test_decode_mixed_ragged(dtype, n_cur):
    """1000 cached tokens (last window 8 tokens), GQA 3:1, explicit split counts."""
    case = synth.decode_case(seed=81, B=3, Hq=6, Hkv=2, d=64, n_cache=1000, dtype=dtype)
    if n_cur != 1:
        rng = np.random.default_rng(n_cur)
        case["K_cur"] = synth.to_dtype_values(rng.standard_normal((3, 2, n_cur, 64)), dtype)
        case["V_cur"] = synth.to_dtype_values(rng.standard_normal((3, 2, n_cur, 64)), dtype)
    tc, oc = mixed_case(case)
    for jensen in (0, 1, 2, 3):
        ro, rl = OA.attention_over_cache(oc, case["Q"], case["K_cur"], case["V_cur"], dtype, jensen=jensen)
        for splits in (1, 3, 7):
            o, l = run_attention(tc, case, jensen=jensen, out_f32=True, path=B.KV_PATH_DECODE, splits=splits)
            check(o, l, ro, rl)


def test_decode_many_splits():
    """The split merge past 16 splits: 24 splits (weights through shared memory) and 300 splits
    over the 32 blocks (plain loops; most splits empty), 16 query heads per kv head."""
    case = synth.decode_case(seed=85, B=1, Hq=16, Hkv=1, d=64, n_cache=1000)
    tc, oc = mixed_case(case)
    ro, rl = OA.attention_over_cache(oc, case["Q"], case["K_cur"], case["V_cur"], "f16", jensen=1)
    for splits in (24, 300):
        o, l = run_attention(tc, case, jensen=1, out_f32=True, path=B.KV_PATH_DECODE, splits=splits)
        check(o, l, ro, rl)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("d,Hq,Hkv", [(128, 3, 3), (64, 32, 2), (128, 16, 1)])
def test_decode_uniform(bits, d, Hq, Hkv):
    """Uniform INT2 / INT4 chunk caches (ragged chunk ends), bf16, including 16 heads per kv head."""
    case = synth.chunk_case(82, B=2, Hkv=Hkv, Hq=Hq, d=d, chunks=[300, 77, 5], n_cur=1, n_q=1, dtype="bf16")
    tc = gpu_uniform(case, bits)
    oc = OL.build_uniform(case["K_cache"], case["V_cache"], bits, case["chunks"],
                          sum((n + 31) // 32 for n in case["chunks"]))
    for jensen in (0, 1, 3):
        ro, rl = OA.attention_over_cache(oc, case["Q"], case["K_cur"], case["V_cur"], "bf16", jensen=jensen)
        for splits in (0, 2):
            o, l = run_attention(tc, case, jensen=jensen, out_f32=True, path=B.KV_PATH_DECODE, splits=splits)
            check(o, l, ro, rl)
        o16, _ = run_attention(tc, case, jensen=jensen, out_f32=False, path=B.KV_PATH_DECODE, splits=2)
        assert_rounding_of(o16, o, "bf16")


def test_decode_mixed_d128_f16():
    case = synth.decode_case(seed=83, B=2, Hq=8, Hkv=2, d=128, n_cache=700)
    tc, oc = mixed_case(case)
    ro, rl = OA.attention_over_cache(oc, case["Q"], case["K_cur"], case["V_cur"], "f16", jensen=1)
    o, l = run_attention(tc, case, jensen=1, out_f32=True)
    check(o, l, ro, rl)


def test_decode_empty_cache_and_single_block():
    case = synth.decode_case(seed=84, B=1, Hq=4, Hkv=1, d=64, n_cache=20)
    empty = B.TorchCache(1, 1, 64, B.KV_MIXED, (1, 1, 1), raw_dtype=B.KV_F16)
    oc0 = OL.build_mixed(case["K_cache"][:, :, :0], case["V_cache"][:, :, :0], np.zeros((1, 0), int),
                         [1, 1, 1], "f16")
    ro, rl = OA.attention_over_cache(oc0, case["Q"], case["K_cur"], case["V_cur"], "f16")
    o, l = run_attention(empty, case, out_f32=True, path=B.KV_PATH_DECODE)
    check(o, l, ro, rl)
    tc, oc = mixed_case(case)          # one window of 20 tokens, FP16 (window 0)
    ro, rl = OA.attention_over_cache(oc, case["Q"], case["K_cur"], case["V_cur"], "f16")
    o, l = run_attention(tc, case, out_f32=True, path=B.KV_PATH_DECODE, splits=4)
    check(o, l, ro, rl)


def test_decode_matches_simt_path():
    """Same cache through the decode kernel and the CUDA-core kernel."""
    case = synth.decode_case(seed=85, B=2, Hq=14, Hkv=2, d=64, n_cache=3000)
    tc, _ = mixed_case(case, 0.1, 0.4)
    o_d, l_d = run_attention(tc, case, jensen=1, out_f32=True, path=B.KV_PATH_DECODE)
    o_s, l_s = run_attention(tc, case, jensen=1, out_f32=True, path=B.KV_PATH_SIMT)
    assert_close(o_d, l_d, o_s, l_s, TIGHT)


def test_decode_over_rollout_cache_sampled():
    """The streaming path over a video-diffusion cache at full size: one query per head over
    the rollout cache (40 heads, 21 INT2 chunks = 32760 tokens, d 128, bf16) plus its own
    token, Jensen TAYLOR2, automatic split-K; sampled heads against the oracle."""
    chunks = [1560] * 21
    case = synth.chunk_case(3, Hkv=40, chunks=chunks, n_cur=1, n_q=1)
    tc = gpu_uniform(case, 2)
    path, splits = B.kv_attention_plan(tc.c, B.KV_BF16, 1, 1, 40, B.kv_attn_opts(0.0, 1, 0, 1, 0, B.KV_PATH_AUTO))
    assert path == B.KV_PATH_DECODE and splits > 1
    o, l = run_attention(tc, case, jensen=1, out_f32=True)
    nb = sum((n + 31) // 32 for n in chunks)
    for h in [0, 17, 39]:
        sl = slice(h, h + 1)
        oc = OL.build_uniform(case["K_cache"][:, sl], case["V_cache"][:, sl], 2, chunks, nb)
        ro, rl = OA.attention_over_cache(oc, case["Q"][:, sl], case["K_cur"][:, sl], case["V_cur"][:, sl], "bf16",
                                         jensen=1)
        check(o[:, sl], l[:, sl], ro, rl)
