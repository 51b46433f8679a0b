"""GPU parity of kv_quantize_append and kv_dequantize against the oracle: bit-exact bytes."""

import numpy as np
import pytest

from bit_kv_cache_28_b300 import bitkv as B
from bit_kv_cache_28_b300 import synth
from oracle import layout as OL, window as OW, codebook as OC, psac as OP
from helpers import gpu_uniform, gpu_mixed, cache_bytes, to_dev, DT

pytestmark = pytest.mark.gpu


def assert_same_cache(tc, oc):
    data, blen, bpos = cache_bytes(tc)
    assert data.shape == oc.data.shape
    bad = np.nonzero(data != oc.data)
    assert bad[0].size == 0, f"{bad[0].size} bytes differ, first at {[x[0] for x in bad]}"
    assert (blen == oc.blk_len).all() and (bpos == oc.blk_pos).all()
    assert sum(tc.n_blocks) == sum(oc.n_blocks) and tc.n_tokens == oc.n_tokens


def uniform_pair(case, bits):
    tc = gpu_uniform(case, bits)
    oc = OL.build_uniform(case["K_cache"], case["V_cache"], bits, case["chunks"], sum((n + 31) // 32 for n in case["chunks"]))
    return tc, oc


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 128), ("f16", 64), ("f32", 64), ("bf16", 256),
                                     ("f32", 32), ("f32", 128)])
def test_uniform_append_ragged(bits, dtype, d):
    """Ragged chunk ends (100 = 3 blocks + 4 tokens, 77, a full block, one token), every input
    dtype, head dims 32 to 256."""
    case = synth.chunk_case(21, B=2, Hkv=3, d=d, chunks=[100, 77, 32, 1], n_cur=5, dtype=dtype)
    tc, oc = uniform_pair(case, bits)
    assert_same_cache(tc, oc)
    assert tc.n_tokens == 210 and tc.n_blocks[2 if bits == 2 else 1] == 4 + 3 + 1 + 1


def test_tiny_workload_append():
    case = synth.tiny()
    tc, oc = uniform_pair(case, 2)
    assert_same_cache(tc, oc)


def test_chunk_workload_append_full():
    case = synth.chunk()
    tc, oc = uniform_pair(case, 2)
    assert_same_cache(tc, oc)


@pytest.mark.slow
def test_rollout_workload_append_full():
    case = synth.rollout()
    tc, oc = uniform_pair(case, 2)
    assert_same_cache(tc, oc)


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128), ("f16", 128)])
def test_degenerate_groups(dtype, d):
    """Constant groups (s = 0), signed zeros, and a 1-token chunk."""
    case = synth.chunk_case(22, B=1, Hkv=2, d=d, chunks=[40, 1], n_cur=1, dtype=dtype)
    K = case["K_cache"]
    K[:, 0, :32, 5] = 2.5                  # constant key channel group
    K[:, 1, :32, 7] = -0.0
    K[:, 1, 3, 7] = 0.0
    case["V_cache"][:, 0, 10, :32] = -1.25  # constant value group
    for bits in (2, 4):
        tc, oc = uniform_pair(case, bits)
        assert_same_cache(tc, oc)


def test_dequantize_matches_oracle():
    import torch
    case = synth.chunk_case(23, B=2, Hkv=2, d=128, chunks=[70, 45], n_cur=3, dtype="bf16")
    tc, oc = uniform_pair(case, 2)
    n = tc.n_tokens
    Ko = torch.zeros((2, 2, n, 128), dtype=torch.float32, device="cuda")
    Vo = torch.zeros_like(Ko)
    B.kv_dequantize(tc.c, Ko, Vo)
    torch.cuda.synchronize()
    for b in range(2):
        for h in range(2):
            lg = oc.logical(b, h)
            assert np.abs(Ko[b, h].cpu().numpy() - lg["khat"]).max() <= 1e-6
            assert np.abs(Vo[b, h].cpu().numpy() - lg["vhat"]).max() <= 1e-6
            assert (Ko[b, h].cpu().numpy() == lg["khat"]).all()     # same fma rule: identical


def mixed_pair(case, frac16=0.2, frac4=0.3):
    n = case["K_cache"].shape[2]
    W = (n + 31) // 32
    bits = np.stack([OW.window_plan(case["sim"][b], frac16, frac4)[0] for b in range(case["B"])])
    caps = [int((bits[0] == k).sum()) for k in (16, 4, 2)]
    tc = gpu_mixed(case, bits, caps)
    oc = OL.build_mixed(case["K_cache"], case["V_cache"], bits, caps, case["dtype"])
    return tc, oc, bits


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_mixed_append_small(dtype):
    case = synth.decode_case(seed=31, B=3, Hq=6, Hkv=2, d=64, n_cache=1000, dtype=dtype)
    tc, oc, bits = mixed_pair(case)
    assert_same_cache(tc, oc)
    assert list(tc.c.n_blocks) == oc.n_blocks


def test_decode_workload_append_full():
    case = synth.decode_case()
    tc, oc, bits = mixed_pair(case)
    assert_same_cache(tc, oc)
    assert list(tc.c.n_blocks) == [123, 184, 306]


def test_codebook_append_with_oracle_calibration():
    """Codebook append given centroids and U (inputs): indices, values and fp16 coefficients."""
    import torch
    case = synth.codebook_case(seed=41, H=2, d=128, n_cache=150, n_cur=20, n_hist=64)
    H, d, r = 2, 128, 8
    cent = np.stack([OC.fit_centroids(case["K_cache"][0, h]) for h in range(H)])[None]
    U = np.stack([OP.psac_basis(case["Q_hist"][h], r)[0] for h in range(H)]).astype(np.float32)[None]
    nb = (150 + 31) // 32
    tc = B.TorchCache(1, H, d, B.KV_CODEBOOK2, (0, 0, nb), raw_dtype=B.KV_BF16, psac_rank=r)
    tc.centroids.copy_(torch.from_numpy(cent.reshape(-1)).cuda())
    tc.psac_u.copy_(torch.from_numpy(U.reshape(-1)).cuda())
    B.kv_quantize_append(to_dev(case["K_cache"], "bf16"), to_dev(case["V_cache"], "bf16"), B.KV_BF16, 150, tc.c)
    oc = OC.build_codebook(case["K_cache"], case["V_cache"], cent, U, nb)
    data, blen, bpos = cache_bytes(tc)
    # coefficients are fp16 roundings of an fp64 dot product: allow a differing last bit
    # only where the oracle's value sits on an fp16 rounding boundary (none expected)
    assert (data == oc.data).all()
    assert (blen == oc.blk_len).all() and (bpos == oc.blk_pos).all()


@pytest.mark.parametrize("r", [0, 24])
def test_codebook_append_adversarial_keys(r):
    """Nearest-centroid decisions at their edges, bit-exact against the oracle: duplicated
    centroids, keys exactly on midpoints (ties go to the lower index), keys next to midpoints,
    and keys far smaller than symmetric centroids (where fp64 |x - mu| rounds to a tie)."""
    import torch
    rng = np.random.default_rng(7)
    H, d, n = 1, 128, 96
    cent = rng.normal(size=(d, 4)).astype(np.float32)
    dup = rng.normal(size=(32, 2)).astype(np.float32)
    cent[32:64] = dup[:, [1, 0, 1, 0]]                                    # duplicates, higher index first
    cent[64:96] = rng.integers(-8, 8, size=(32, 4)) * 0.25                # bf16-exact midpoints
    b = np.abs(rng.normal(size=(32, 2))).astype(np.float32)
    cent[96:128] = np.stack([b[:, 0], -b[:, 0], -b[:, 1], b[:, 1]], 1)   # symmetric pairs
    K = synth.to_bf16_values(rng.normal(size=(1, H, n, d)).astype(np.float32))
    for c in range(64, 96):                                               # keys on and next to midpoints
        mids = (cent[c][:, None].astype(np.float64) + cent[c][None, :]) / 2
        pick = rng.choice(mids.reshape(-1), n)
        K[0, 0, :, c] = synth.to_bf16_values(pick.astype(np.float32))
        K[0, 0, ::3, c] = synth.to_bf16_values(np.nextafter(pick[::3].astype(np.float32), np.float32(9)))
    tiny = np.array([0.0, -0.0, 1e-30, -1e-30, 1e-38, -1e-38, 3e-39, 1e-20], np.float32)
    K[0, 0, :, 96:] = synth.to_bf16_values(rng.choice(tiny, (n, 32)))
    V = synth.to_bf16_values(rng.normal(size=(1, H, n, d)).astype(np.float32))
    nb = n // 32
    U = None
    if r:
        Qh = synth.to_bf16_values(rng.normal(size=(64, d)).astype(np.float32))
        U = OP.psac_basis(Qh, r)[0].astype(np.float32)[None, None]
    tc = B.TorchCache(1, H, d, B.KV_CODEBOOK2, (0, 0, nb), raw_dtype=B.KV_BF16, psac_rank=r)
    tc.centroids.copy_(torch.from_numpy(cent.reshape(-1)).cuda())
    if r:
        tc.psac_u.copy_(torch.from_numpy(U.reshape(-1)).cuda())
    B.kv_quantize_append(to_dev(K, "bf16"), to_dev(V, "bf16"), B.KV_BF16, n, tc.c)
    oc = OC.build_codebook(K, V, cent[None, None], U, nb)
    data, blen, _ = cache_bytes(tc)
    assert (data == oc.data).all(), np.argwhere(data != oc.data)[:8]
    assert (blen == oc.blk_len).all()
