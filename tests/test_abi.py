"""C-ABI checks that need no GPU: the library loads, exports every declared symbol,
and its host-side logic (layout sizes, window plan, argument checks) agrees with the oracle."""

import os
import re

import numpy as np
import pytest

from bit_kv_cache_28_b300 import bitkv as B
from oracle import layout as OL
from oracle import window as OW
from bit_kv_cache_28_b300 import synth

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "bitkv.h")


def declared_functions():
    src = open(HDR).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(kv_\w+)\s*\(", src, flags=re.M)))


def test_library_exports_every_declared_symbol():
    lib = B.lib()
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(B.EXPORTS) == names


def test_version():
    assert "sm_103a" in B.kv_version()


@pytest.mark.parametrize("d", [64, 128])
def test_layout_sizes_match_oracle(d):
    L = B.kv_layout_init(2, 3, d, B.KV_MIXED, B.KV_F16, (5, 7, 11))
    assert list(L.block_bytes) == [OL.block_bytes(OL.RAW16, d), OL.block_bytes(OL.INT4, d), OL.block_bytes(OL.INT2, d)]
    offs, stream = OL.stream_layout([OL.RAW16, OL.INT4, OL.INT2], [5, 7, 11], d)
    assert list(L.seg_offset) == offs and L.stream_bytes == stream
    assert B.kv_layout_bytes(L, B.KV_REGION_DATA) == 6 * stream
    assert B.kv_layout_bytes(L, B.KV_REGION_BLK_LEN) == 2 * 23 * 4
    Lc = B.kv_layout_init(1, 2, d, B.KV_CODEBOOK2, B.KV_BF16, (0, 0, 9), 8)
    assert Lc.block_bytes[2] == OL.block_bytes(OL.CB2, d, 8)
    assert B.kv_layout_bytes(Lc, B.KV_REGION_CENTROIDS) == 2 * d * 4 * 4
    assert B.kv_layout_bytes(Lc, B.KV_REGION_PSAC_U) == 2 * d * 8 * 4


@pytest.mark.parametrize("d", [64, 128])
def test_fp16_metadata_layout(d):
    """fp16 (s, z) pairs: the INT segments shrink by 8 d bytes per block, RAW16 stays."""
    L = B.kv_layout_init(2, 3, d, B.KV_MIXED, B.KV_F16, (5, 7, 11), 0, B.KV_F16)
    assert L.meta_dtype == B.KV_F16
    assert list(L.block_bytes) == [OL.block_bytes(OL.RAW16, d), OL.block_bytes(OL.INT4, d, meta16=True),
                                   OL.block_bytes(OL.INT2, d, meta16=True)]
    offs, stream = OL.stream_layout([OL.RAW16, OL.INT4, OL.INT2], [5, 7, 11], d, meta16=True)
    assert list(L.seg_offset) == offs and L.stream_bytes == stream
    L32 = B.kv_layout_init(2, 3, d, B.KV_MIXED, B.KV_F16, (5, 7, 11))
    assert L32.stream_bytes - L.stream_bytes == (7 + 11) * 8 * d
    with pytest.raises(B.BitKVError) as e:
        B.kv_layout_init(1, 1, d, B.KV_CODEBOOK2, B.KV_BF16, (0, 0, 4), 0, B.KV_F16)
    assert e.value.status == B.KV_ERR_UNSUPPORTED
    with pytest.raises(B.BitKVError) as e:
        B.kv_layout_init(1, 1, d, B.KV_UNIFORM2, B.KV_BF16, (0, 0, 4), 0, B.KV_BF16)
    assert e.value.status == B.KV_ERR_INVALID_ARG


def test_window_plan_matches_oracle():
    c = synth.decode_case()
    for b in range(8):
        bits = np.zeros(613, np.int8)
        perm = np.zeros(613, np.int32)
        B.kv_window_plan(c["sim"][b], 613, B.kv_thresholds(0.2, 0.3, 1), bits, perm)
        ob, op = OW.window_plan(c["sim"][b], 0.2, 0.3, True)
        assert (bits == ob).all() and (perm == op).all()
    rng = np.random.default_rng(0)
    for trial in range(50):
        W = int(rng.integers(1, 60))
        sim = np.round(rng.uniform(-1, 1, W), 1).astype(np.float32)   # many ties
        f16, f4 = float(rng.uniform(0, 0.5)), float(rng.uniform(0, 0.5))
        ff = int(rng.integers(0, 2))
        bits = np.zeros(W, np.int8)
        perm = np.zeros(W, np.int32)
        B.kv_window_plan(sim, W, B.kv_thresholds(f16, f4, ff), bits, perm)
        ob, op = OW.window_plan(sim, f16, f4, bool(ff))
        assert (bits == ob).all() and (perm == op).all()


def test_argument_errors_never_launch():
    with pytest.raises(B.BitKVError) as e:
        B.kv_layout_init(1, 1, 96 + 1, B.KV_UNIFORM2, B.KV_F16, (0, 0, 4))
    assert e.value.status == B.KV_ERR_UNSUPPORTED
    with pytest.raises(B.BitKVError) as e:
        B.kv_layout_init(1, 1, 64, B.KV_UNIFORM2, B.KV_F16, (1, 0, 4))
    assert e.value.status == B.KV_ERR_INVALID_ARG
    with pytest.raises(B.BitKVError) as e:
        B.kv_layout_init(1, 1, 64, B.KV_MIXED, B.KV_F32, (1, 1, 4))
    assert e.value.status == B.KV_ERR_INVALID_ARG
    L = B.kv_layout_init(1, 2, 64, B.KV_UNIFORM2, B.KV_F16, (0, 0, 4))
    with pytest.raises(B.BitKVError) as e:
        B.kv_cache_init(L, 0x1008, 0x2000, 0x3000)          # misaligned data pointer
    assert e.value.status == B.KV_ERR_ALIGNMENT
    # fake (never dereferenced) device addresses: every check below fails before a launch
    c = B.kv_cache_init(L, 0x10000, 0x20000, 0x30000)
    with pytest.raises(B.BitKVError) as e:
        B.kv_quantize_append(0x40000, 0x50000, B.KV_F16, 32 * 5, c, None, 0)
    assert e.value.status == B.KV_ERR_CAPACITY
    with pytest.raises(B.BitKVError) as e:
        B.kv_quantize_append(0x40008, 0x50000, B.KV_F16, 32, c, None, 0)
    assert e.value.status == B.KV_ERR_ALIGNMENT
    with pytest.raises(B.BitKVError) as e:
        B.kv_quantize_append(0x40000, 0x50000, B.KV_F16, 0, c, None, 0)
    assert e.value.status == B.KV_ERR_INVALID_ARG
    opts = B.kv_attn_opts(0.0, 0, 0, 0, 0, B.KV_PATH_SIMT)
    with pytest.raises(B.BitKVError) as e:
        B.kv_attention(0x40000, 0x50000, 0x60000, B.KV_F16, 4, 4, 3, c, opts, 0x70000, None, None, 0, 0)
    assert e.value.status == B.KV_ERR_INVALID_ARG        # Hq not a multiple of Hkv
    opts = B.kv_attn_opts(0.0, 0, 1, 0, 0, B.KV_PATH_SIMT)
    with pytest.raises(B.BitKVError) as e:
        B.kv_attention(0x40000, 0x50000, 0x60000, B.KV_F16, 4, 4, 2, c, opts, 0x70000, None, None, 0, 0)
    assert e.value.status == B.KV_ERR_INVALID_ARG        # PSAC on a uniform cache
    opts = B.kv_attn_opts(0.0, 0, 0, 0, 8, B.KV_PATH_SIMT)
    need = B.kv_attention_workspace(c, B.KV_F16, 4, 4, 2, opts)
    assert need > 0
    with pytest.raises(B.BitKVError) as e:
        B.kv_attention(0x40000, 0x50000, 0x60000, B.KV_F16, 4, 4, 2, c, opts, 0x70000, None, None, 0, 0)
    assert e.value.status == B.KV_ERR_WORKSPACE
    assert "workspace" in B.kv_last_error()


def test_window_similarity_argument_errors():
    """Rejected on the host before any launch (fake, never dereferenced addresses)."""
    sim = 0x30000
    cases = [((0x10000, 0x20000, B.KV_F16, 0, 4, 64, 8, 64, sim), B.KV_ERR_INVALID_ARG),   # B = 0
             ((0x10000, 0x20000, B.KV_F16, 1, 4, -1, 8, 64, sim), B.KV_ERR_INVALID_ARG),  # n < 0
             ((0x10000, None, B.KV_F16, 1, 4, 64, 8, 64, sim), B.KV_ERR_INVALID_ARG),     # Kq NULL, m > 0
             ((0x10000, 0x20000, B.KV_F16, 1, 4, 64, 8, 60, sim), B.KV_ERR_UNSUPPORTED),  # rows of 120 bytes
             ((0x10000, 0x20000, B.KV_F16, 1, 32, 64, 8, 512, sim), B.KV_ERR_UNSUPPORTED),  # 2048 groups
             ((0x10008, 0x20000, B.KV_F16, 1, 4, 64, 8, 64, sim), B.KV_ERR_ALIGNMENT)]
    for args, status in cases:
        with pytest.raises(B.BitKVError) as e:
            B.kv_window_similarity(*args, 0)
        assert e.value.status == status
    B.kv_window_similarity(0x10000, 0x20000, B.KV_F16, 1, 4, 0, 8, 64, sim, 0)   # n == 0: nothing to do
