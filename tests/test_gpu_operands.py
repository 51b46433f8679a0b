"""The attention kernels' own cache operands against the oracle (kv_debug_operands).

The tensor-core kernel's producers expand packed blocks into fp16 K_hat and V_hat tiles;
the dump runs those same device routines on a staged tile.  Each operand must be the fp16
round-to-nearest-even of the oracle's dequantised entry fmaf(code, s, z) (codebook keys: of
the centroid), bit for bit -- which also bounds the kernel's fp32 value before the
rounding to half an fp16 step.  The decode kernel forms no dequantised entry: its operands
are the codes, as exact fp16 integers, which must equal the oracle's codes bit for bit
(pad slots: code 0)."""

import numpy as np
import pytest

from bit_kv_cache_28_b300 import bitkv as B
from bit_kv_cache_28_b300 import synth
from oracle import layout as OL, window as OW, codebook as OC
from helpers import gpu_uniform, gpu_mixed, to_dev

pytestmark = pytest.mark.gpu


def dump(tc, path):
    import torch
    L = tc.layout
    n = sum(tc.c.n_blocks) * 32
    K = torch.full((L.B, L.Hkv, n, L.d), float("nan"), dtype=torch.float16, device="cuda")
    V = torch.full_like(K, float("nan"))
    B.kv_debug_operands(tc.c, path, K, V)
    torch.cuda.synchronize()
    return K.cpu().view(torch.int16).numpy(), V.cpu().view(torch.int16).numpy()


def f16_bits(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float16).view(torch.int16).numpy()


def slot0(oc, seg):
    return int(sum(oc.n_blocks[:seg]))


def check_tc(Kd, Vd, oc, pairs):
    """pairs: (b, h of the dump, h of the oracle cache)."""
    for b, h, ho in pairs:
        for rec in oc.blocks[b][ho]:
            n, s = rec["len"], 32 * (slot0(oc, rec["seg"]) + rec["slot"])
            assert np.array_equal(Kd[b, h, s:s + n], f16_bits(rec["khat"][:n])), (b, h, rec["pos"])
            assert np.array_equal(Vd[b, h, s:s + n], f16_bits(rec["vhat"][:n])), (b, h, rec["pos"])


def check_dec(Kd, Vd, oc, pairs):
    for b, h, ho in pairs:
        for rec in oc.blocks[b][ho]:
            if not rec["quantised"]:
                continue
            n, s = rec["len"], 32 * (slot0(oc, rec["seg"]) + rec["slot"])
            assert np.array_equal(Kd[b, h, s:s + n], f16_bits(rec["kcode"][:n])), (b, h, rec["pos"])
            assert np.array_equal(Vd[b, h, s:s + n], f16_bits(rec["vcode"][:n])), (b, h, rec["pos"])
            assert (Kd[b, h, s + n:s + 32] == 0).all() and (Vd[b, h, s + n:s + 32] == 0).all()


@pytest.mark.parametrize("bits", [2, 4])
def test_tc_operands_ragged(bits):
    """Ragged chunk ends (300 = 9 blocks + 12 tokens, 77 = 2 blocks + 13): tiles of 4, 4, 4, 1
    blocks, two batch rows, two kv heads."""
    case = synth.chunk_case(61, B=2, Hkv=2, Hq=4, d=128, chunks=[300, 77], n_cur=1, n_q=1, dtype="bf16")
    tc = gpu_uniform(case, bits)
    oc = OL.build_uniform(case["K_cache"], case["V_cache"], bits, case["chunks"], sum(tc.c.n_blocks))
    Kd, Vd = dump(tc, B.KV_PATH_TC)
    check_tc(Kd, Vd, oc, [(b, h, h) for b in range(2) for h in range(2)])


def test_tc_operands_codebook():
    import torch
    case = synth.codebook_case(seed=71, H=2, d=128, n_cache=450, n_cur=8, n_hist=64)
    cent = np.stack([OC.fit_centroids(case["K_cache"][0, h]) for h in range(2)])[None].astype(np.float32)
    tc = B.TorchCache(1, 2, 128, B.KV_CODEBOOK2, (0, 0, 15), raw_dtype=B.KV_BF16)
    tc.centroids.copy_(torch.from_numpy(cent.reshape(-1)).cuda())
    B.kv_quantize_append(to_dev(case["K_cache"], "bf16"), to_dev(case["V_cache"], "bf16"), B.KV_BF16, 450, tc.c)
    oc = OC.build_codebook(case["K_cache"], case["V_cache"], cent, None, 15)
    Kd, Vd = dump(tc, B.KV_PATH_TC)
    check_tc(Kd, Vd, oc, [(0, 0, 0), (0, 1, 1)])


def test_tc_operands_rollout_workload():
    """The full rollout cache (40 heads, 21 chunks of 1560 tokens = 1092 blocks per head)."""
    case = synth.rollout()
    tc = gpu_uniform(case, 2)
    Kd, Vd = dump(tc, B.KV_PATH_TC)
    heads = [0, 21, 39]
    oc = OL.build_uniform(case["K_cache"][:, heads], case["V_cache"][:, heads], 2, case["chunks"],
                          sum(tc.c.n_blocks))
    check_tc(Kd, Vd, oc, [(0, h, i) for i, h in enumerate(heads)])


@pytest.mark.parametrize("dtype,d", [("f16", 64), ("bf16", 128)])
def test_decode_operands_mixed(dtype, d):
    """A mixed FP16 / INT4 / INT2 cache (1000 tokens, last window 8): every quantised slot's
    codes as the decode kernel's extraction routine produces them."""
    case = synth.decode_case(seed=81, B=3, Hq=6, Hkv=2, d=d, n_cache=1000, dtype=dtype)
    bits = np.stack([OW.window_plan(case["sim"][b])[0] for b in range(3)])
    caps = [int((bits[0] == k).sum()) for k in (16, 4, 2)]
    tc = gpu_mixed(case, bits, caps)
    oc = OL.build_mixed(case["K_cache"], case["V_cache"], bits, caps, dtype)
    Kd, Vd = dump(tc, B.KV_PATH_DECODE)
    check_dec(Kd, Vd, oc, [(b, h, h) for b in range(3) for h in range(2)])


def test_decode_operands_rollout_workload():
    case = synth.chunk_case(3, Hkv=40, chunks=[1560] * 21, n_cur=1, n_q=1)
    tc = gpu_uniform(case, 2)
    Kd, Vd = dump(tc, B.KV_PATH_DECODE)
    heads = [0, 27]
    oc = OL.build_uniform(case["K_cache"][:, heads], case["V_cache"][:, heads], 2, case["chunks"],
                          sum(tc.c.n_blocks))
    check_dec(Kd, Vd, oc, [(0, h, i) for i, h in enumerate(heads)])
