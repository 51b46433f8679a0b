"""GPU parity of caches with fp16 (s, z) metadata: the append bit for bit, the kernels' own
operands bit for bit, and attention on every path against the oracle's definition.

The WindowQuant note (主な結果) and the QuantWM card (Key Results) report caches far smaller
than fp32 step and zero-point metadata allows; this cache variant stores each pair as two
fp16 values (3072 instead of 4096 bytes per INT2 block at head dim 128) and takes its codes
against the stored pair (oracle/quant.py).  The tolerances are the other attention tests'."""

import numpy as np
import pytest

from bit_kv_cache_28_b300 import bitkv as B
from bit_kv_cache_28_b300 import synth
from oracle import layout as OL, window as OW
from oracle import attention as OA
from helpers import (gpu_uniform, gpu_mixed, cache_bytes, run_attention, attention_checked, assert_close,
                     assert_rounding_of, tol, TIGHT)

pytestmark = pytest.mark.gpu

TC_PATHS = [B.KV_PATH_TC, B.KV_PATH_TC_SINGLE]


def assert_same_cache(tc, oc):
    data, blen, bpos = cache_bytes(tc)
    assert data.shape == oc.data.shape
    bad = np.nonzero(data != oc.data)
    assert bad[0].size == 0, f"{bad[0].size} bytes differ, first at {[x[0] for x in bad]}"
    assert (blen == oc.blk_len).all() and (bpos == oc.blk_pos).all()


def oracle_uniform(case, bits, heads=None):
    sl = slice(None) if heads is None else heads
    return OL.build_uniform(case["K_cache"][:, sl], case["V_cache"][:, sl], bits, case["chunks"],
                            sum((n + 31) // 32 for n in case["chunks"]), meta16=True)


def mixed_pair(case):
    bits = np.stack([OW.window_plan(case["sim"][b])[0] for b in range(case["B"])])
    caps = [int((bits[0] == k).sum()) for k in (16, 4, 2)]
    tc = gpu_mixed(case, bits, caps, meta16=True)
    oc = OL.build_mixed(case["K_cache"], case["V_cache"], bits, caps, case["dtype"], meta16=True)
    return tc, oc


# ---- append ------------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 128), ("f16", 64), ("f32", 32), ("bf16", 256)])
def test_uniform_append_bit_exact(bits, dtype, d):
    """16-bit rows at head dim 128 take the fast append kernel, the rest the general one."""
    case = synth.chunk_case(131, B=2, Hkv=3, d=d, chunks=[100, 77, 32, 1], n_cur=5, dtype=dtype)
    tc = gpu_uniform(case, bits, meta16=True)
    assert tc.layout.block_bytes[2 if bits == 2 else 1] == OL.block_bytes(OL.INT2 if bits == 2 else OL.INT4, d,
                                                                          meta16=True)
    assert_same_cache(tc, oracle_uniform(case, bits))


def test_degenerate_groups_bit_exact():
    """Constant groups, signed zeros, a step that rounds to a subnormal fp16 and one that
    underflows to zero (every code 0), a minimum whose fp16 rounding lies above it."""
    case = synth.chunk_case(132, B=1, Hkv=2, d=128, chunks=[40, 1], n_cur=1, dtype="f32")
    K, V = case["K_cache"], case["V_cache"]
    K[:, 0, :32, 5] = 2.5
    K[:, 1, :32, 7] = -0.0
    K[:, 1, 3, 7] = 0.0
    K[:, 0, :32, 9] = 1.0
    K[:, 0, 4, 9] = 1.0 + 2.0 ** -20            # subnormal fp16 step
    K[:, 0, :32, 10] = 1.0
    K[:, 0, 4, 10] = 1.0 + 2.0 ** -23           # step underflows to zero
    K[:, 1, :32, 11] = np.float32(1.000732421875)
    K[:, 1, 6, 11] = 4.0                        # zero point rounds up past the minimum
    V[:, 0, 10, :32] = -1.25
    for bits in (2, 4):
        tc = gpu_uniform(case, bits, meta16=True)
        assert_same_cache(tc, oracle_uniform(case, bits))


def test_mixed_append_and_dequantize_bit_exact():
    import torch
    case = synth.decode_case(seed=133, B=3, Hq=6, Hkv=2, d=64, n_cache=1000, dtype="f16")
    tc, oc = mixed_pair(case)
    assert_same_cache(tc, oc)
    Ko = torch.zeros((3, 2, 1000, 64), dtype=torch.float32, device="cuda")
    Vo = torch.zeros_like(Ko)
    B.kv_dequantize(tc.c, Ko, Vo)
    Ko, Vo = Ko.cpu().numpy(), Vo.cpu().numpy()
    for b in range(3):
        for h in range(2):
            lg = oc.logical(b, h)
            assert np.array_equal(Ko[b, h], lg["khat"]) and np.array_equal(Vo[b, h], lg["vhat"])


def test_decode_workload_append_full():
    """The decode workload's mixed cache (batch 8, 4 kv heads, 19600 tokens) at fp16 metadata:
    every byte, and the algorithmic cache bytes against the fp32-metadata cache."""
    case = synth.decode_case()
    tc, oc = mixed_pair(case)
    assert_same_cache(tc, oc)
    assert tc.layout.block_bytes[1] == 2560 and tc.layout.block_bytes[2] == 1536


# ---- the kernels' own operands -------------------------------------------------------------

def _f16_bits(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float16).view(torch.int16).numpy()


def _dump(tc, path):
    import torch
    L = tc.layout
    n = sum(tc.c.n_blocks) * 32
    K = torch.full((L.B, L.Hkv, n, L.d), float("nan"), dtype=torch.float16, device="cuda")
    V = torch.full_like(K, float("nan"))
    B.kv_debug_operands(tc.c, path, K, V)
    torch.cuda.synchronize()
    return K.cpu().view(torch.int16).numpy(), V.cpu().view(torch.int16).numpy()


@pytest.mark.parametrize("bits", [2, 4])
def test_tc_operands(bits):
    """K_hat and V_hat of the tensor-core producers: the fp16 rounding of fmaf(code, s16, z16)."""
    case = synth.chunk_case(134, B=2, Hkv=2, Hq=4, d=128, chunks=[300, 77], n_cur=1, n_q=1, dtype="bf16")
    tc = gpu_uniform(case, bits, meta16=True)
    oc = oracle_uniform(case, bits)
    Kd, Vd = _dump(tc, B.KV_PATH_TC)
    for b in range(2):
        for h in range(2):
            for rec in oc.blocks[b][h]:
                n, s = rec["len"], 32 * rec["slot"]
                assert np.array_equal(Kd[b, h, s:s + n], _f16_bits(rec["khat"][:n])), (b, h, rec["pos"])
                assert np.array_equal(Vd[b, h, s:s + n], _f16_bits(rec["vhat"][:n])), (b, h, rec["pos"])


@pytest.mark.parametrize("d", [64, 128])
def test_decode_operands_mixed(d):
    """The decode kernel's A operands for fp16-metadata blocks: the fp16 entries themselves,
    bit for bit, pad slots included (code 0: a key pad holds its channel's zero point, a
    value pad +0; the kernel masks them by the block length)."""
    case = synth.decode_case(seed=135, B=2, Hq=4, Hkv=2, d=d, n_cache=700, dtype="bf16")
    tc, oc = mixed_pair(case)
    Kd, Vd = _dump(tc, B.KV_PATH_DECODE)
    for b in range(2):
        for h in range(2):
            for rec in oc.blocks[b][h]:
                if not rec["quantised"]:
                    continue
                s = 32 * (int(sum(oc.n_blocks[:rec["seg"]])) + rec["slot"])
                assert np.array_equal(Kd[b, h, s:s + 32], _f16_bits(rec["khat"]))
                assert np.array_equal(Vd[b, h, s:s + 32], _f16_bits(rec["vhat"]))
                assert (Vd[b, h, s + rec["len"]:s + 32] == 0).all()


def test_decode_range_flag_for_bf16_queries_beyond_fp16():
    """The decode kernel takes the queries of fp16-metadata blocks as fp16: a bf16 query entry
    of 70144 raises the range flag; in-range queries on a fresh workspace report KV_OK."""
    import torch
    case = synth.decode_case(seed=139, B=1, Hq=2, Hkv=1, d=64, n_cache=100, dtype="bf16")
    tc, _ = mixed_pair(case)
    for big, want in ((True, B.KV_ERR_RANGE), (False, B.KV_OK)):
        Q = case["Q"].copy()
        if big:
            Q[0, 1, 0, 9] = synth.to_bf16_values(np.array([70000.0], np.float32))[0]
        q = torch.from_numpy(Q).cuda().to(torch.bfloat16)
        k = torch.from_numpy(case["K_cur"]).cuda().to(torch.bfloat16)
        v = torch.from_numpy(case["V_cur"]).cuda().to(torch.bfloat16)
        opts = B.kv_attn_opts(0.0, 0, 0, 1, 0, B.KV_PATH_DECODE)
        wsb = B.kv_attention_workspace(tc.c, B.KV_BF16, 1, 1, 2, opts)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        out = torch.empty((1, 2, 1, 64), dtype=torch.float32, device="cuda")
        lse = torch.empty((1, 2, 1), dtype=torch.float32, device="cuda")
        B.kv_attention(q, k, v, B.KV_BF16, 1, 1, 2, tc.c, opts, out, lse, ws, wsb)
        if want == B.KV_OK:
            B.kv_attention_status(ws)
        else:
            with pytest.raises(B.BitKVError) as e:
                B.kv_attention_status(ws)
            assert e.value.status == want


# ---- attention -----------------------------------------------------------------------------

@pytest.mark.parametrize("path", TC_PATHS)
@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("jensen", [0, 1, 2, 3])
def test_tc_attention(bits, jensen, path):
    """Ragged blocks, ragged current tile, partial query tile, GQA, 150 queries (a pair with an
    empty odd CTA in the single-tile case), split counts 1 and 3."""
    case = synth.chunk_case(136, B=2, Hkv=2, Hq=4, d=128, chunks=[300, 77], n_cur=150, n_q=150, dtype="bf16")
    tc = gpu_uniform(case, bits, meta16=True)
    oc = oracle_uniform(case, bits)
    args = (oc, case["Q"], case["K_cur"], case["V_cur"], "bf16")
    ref = OA.attention_over_cache(*args, jensen=jensen)
    tight = OA.attention_over_cache(*args, jensen=jensen, operand_dtype="f16")
    for splits in (1, 3):
        attention_checked(tc, case, ref, "bf16", tight, jensen=jensen, path=path, splits=splits)


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("f16", 128)])
@pytest.mark.parametrize("jensen", [1, 2])
def test_simt_attention(dtype, d, jensen):
    case = synth.chunk_case(137, B=1, Hkv=2, Hq=4, d=d, chunks=[130, 45], n_cur=40, n_q=33, dtype=dtype)
    tc = gpu_uniform(case, 2, meta16=True)
    ref = OA.attention_over_cache(oracle_uniform(case, 2), case["Q"], case["K_cur"], case["V_cur"], dtype,
                                  jensen=jensen)
    attention_checked(tc, case, ref, dtype, ref, jensen=jensen, path=B.KV_PATH_SIMT, splits=2)


@pytest.mark.parametrize("dtype,d", [("f16", 64), ("bf16", 128)])
def test_decode_attention_mixed(dtype, d):
    case = synth.decode_case(seed=138, B=3, Hq=6, Hkv=2, d=d, n_cache=1000, dtype=dtype)
    tc, oc = mixed_pair(case)
    for jensen in (0, 1, 2, 3):
        ro, rl = OA.attention_over_cache(oc, case["Q"], case["K_cur"], case["V_cur"], dtype, jensen=jensen)
        for splits in (0, 5):
            o, l = run_attention(tc, case, jensen=jensen, out_f32=True, path=B.KV_PATH_DECODE, splits=splits)
            assert_close(o, l, ro, rl, TIGHT)
            o16, _ = run_attention(tc, case, jensen=jensen, out_f32=False, path=B.KV_PATH_DECODE, splits=splits)
            assert_rounding_of(o16, o, dtype)


def test_decode_workload_full():
    """The decode workload on the fp16-metadata cache: every output row against the oracle."""
    case = synth.decode_case()
    tc, oc = mixed_pair(case)
    path, splits = B.kv_attention_plan(tc.c, B.KV_F16, 1, 1, 28)
    assert path == B.KV_PATH_DECODE and splits > 1
    ro, rl = OA.attention_over_cache(oc, case["Q"], case["K_cur"], case["V_cur"], "f16", jensen=1)
    o, l = run_attention(tc, case, jensen=1, out_f32=True)
    assert_close(o, l, ro, rl, TIGHT)


def test_rollout_workload_tc_sampled():
    """The rollout workload (40 heads, 21 cached chunks of 1560 tokens, 1560 queries) on an
    fp16-metadata INT2 cache through the benchmark's dispatch: 2 heads x 24 sampled rows
    against the oracle, every row against the CUDA-core kernel."""
    case = synth.rollout()
    tc = gpu_uniform(case, 2, meta16=True)
    path, _ = B.kv_attention_plan(tc.c, B.KV_BF16, 1560, 1560, 40, B.kv_attn_opts(0.0, 1, 0, 0, 0, B.KV_PATH_AUTO))
    assert path == B.KV_PATH_TC
    o_tc, l_tc = run_attention(tc, case, jensen=1, out_f32=True)
    o_si, l_si = run_attention(tc, case, jensen=1, out_f32=True, path=B.KV_PATH_SIMT)
    assert_close(o_tc, l_tc, o_si, l_si, tol("bf16"))
    rows = np.random.default_rng(4).choice(1560, 24, replace=False)
    heads = [3, 36]
    oc = oracle_uniform(case, 2, heads)
    for i, h in enumerate(heads):
        view = OL.Cache(1, 1, oc.d, oc.classes, oc.caps, meta16=True)
        view.blocks = [[oc.blocks[0][i]]]
        args = (view, case["Q"][:, h:h + 1], case["K_cur"][:, h:h + 1], case["V_cur"][:, h:h + 1], "bf16")
        ref = OA.attention_over_cache(*args, jensen=1, rows=rows)
        tight = OA.attention_over_cache(*args, jensen=1, rows=rows, operand_dtype="f16")
        assert_close(o_tc[:, h:h + 1], l_tc[:, h:h + 1], ref[0], ref[1], tol("bf16"), rows=rows)
        assert_close(o_tc[:, h:h + 1], l_tc[:, h:h + 1], tight[0], tight[1], TIGHT, rows=rows)
        assert_close(o_si[:, h:h + 1], l_si[:, h:h + 1], ref[0], ref[1], TIGHT, rows=rows)

