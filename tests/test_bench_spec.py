"""The algorithmic bytes and FLOPs that bench.py divides by its kernel times (CPU only).

The roofline fractions rest on these counts, so each is rebuilt here from the oracle's
block layout (oracle/layout.py) and from the shapes of the two contractions, instead of
from bench.py's own closed forms:
- the cache bytes of a uniform INT2 cache are, block by block, the codes and value
  metadata of the valid tokens plus the block's key metadata; a full block's count must
  equal the oracle's block size;
- each appended chunk starts a new block, so a 1560-token chunk gives 48 full blocks and
  one of 24 tokens (the layout described in the "Quantized Keys Steal Attention" set-up:
  the cache of each finished chunk is packed);
- attention FLOPs are two matrix products per head, Q K^T and P V, 2 FLOPs per
  multiply-add.
"""

import pytest

import bench
from oracle import layout as OL


def blocks_of_chunk(n):
    return [OL.BLOCK] * (n // OL.BLOCK) + ([n % OL.BLOCK] if n % OL.BLOCK else [])


def int_block_algorithmic(v, d, bits, meta16):
    """Bytes of one INT block that carry information: codes and value (s, z) of the v valid
    tokens, and the block's per-channel key (s, z)."""
    pair = 4 if meta16 else 8
    return 2 * v * d * bits // 8 + d * pair + v * (d // 32) * pair


def matmul_flops(m, k, n):
    return 2 * m * k * n


@pytest.mark.parametrize("meta16", [False, True])
def test_full_int2_block_counts_as_the_oracle_block(meta16):
    for d in (64, 128):
        assert int_block_algorithmic(OL.BLOCK, d, 2, meta16) == OL.block_bytes(OL.INT2, d, meta16=meta16)
        assert int_block_algorithmic(OL.BLOCK, d, 4, meta16) == OL.block_bytes(OL.INT4, d, meta16=meta16)


@pytest.mark.parametrize("name,H,n_chunks", [("chunk", 24, 3), ("rollout", 40, 21)])
@pytest.mark.parametrize("meta16", [False, True])
def test_chunk_workload_cache_bytes(name, H, n_chunks, meta16):
    spec = bench.with_meta16(bench.workload_spec(name), meta16)
    d, n = spec["d"], spec["n_cur"]
    assert (d, n, spec["chunks"]) == (128, 1560, [1560] * n_chunks) and spec["Hkv"] == H
    blocks = blocks_of_chunk(n) * n_chunks
    assert len(blocks) == 49 * n_chunks and blocks[48] == 24
    want = H * sum(int_block_algorithmic(v, d, 2, meta16) for v in blocks)
    assert spec["cache_bytes"] == pytest.approx(want, rel=0, abs=0.5)


@pytest.mark.parametrize("meta16", [False, True])
def test_rollout_append_bytes(meta16):
    """A finished 1560-token chunk of 40 heads: bf16 K and V read once, 49 whole blocks
    (pad slots included) written per head."""
    spec = bench.with_meta16(bench.workload_spec("rollout"), meta16)
    H, d, n = spec["Hkv"], spec["d"], spec["n_cur"]
    read = 2 * H * n * d * 2
    written = H * len(blocks_of_chunk(n)) * OL.block_bytes(OL.INT2, d, meta16=meta16)
    assert spec["append_bytes"] == read + written


def test_codebook_workload_bytes():
    spec = bench.workload_spec("codebook")
    H, d, r = spec["Hkv"], spec["d"], spec["r"]
    nb = len(blocks_of_chunk(spec["chunks"][0]))
    assert nb == 256
    assert spec["cache_bytes"] == H * nb * OL.block_bytes(OL.CB2, d, r=r)


@pytest.mark.parametrize("name", ["chunk", "rollout", "tiny"])
def test_attention_flops(name):
    spec = bench.workload_spec(name)
    H, d, m = spec["Hq"], spec["d"], spec["n_q"]
    keys = sum(spec["chunks"]) + spec["n_cur"]
    want = H * (matmul_flops(m, d, keys) + matmul_flops(m, keys, d))
    assert spec["attn_flops"] == want


def test_rollout_flops_value():
    """40 heads, 1560 queries over 21 x 1560 cached + 1560 current tokens, d 128: 1096.5 GFLOP."""
    assert bench.workload_spec("rollout")["attn_flops"] / 1e9 == pytest.approx(1096.5, abs=0.05)


def test_codebook_flops_include_the_psac_term():
    """Q K^T and P V over all keys, plus the rank-r PSAC logits (U^T q) . coeff for the cached keys."""
    spec = bench.workload_spec("codebook")
    H, d, m, r = spec["Hq"], spec["d"], spec["n_q"], spec["r"]
    n_cache = spec["chunks"][0]
    keys = n_cache + spec["n_cur"]
    want = H * (matmul_flops(m, d, keys) + matmul_flops(m, keys, d) + matmul_flops(m, r, n_cache))
    assert spec["attn_flops"] == want


@pytest.mark.parametrize("name,H,B", [("decode", 28, 8), ("rollout_decode", 40, 1)])
def test_decode_flops(name, H, B):
    spec = bench.workload_spec(name)
    assert spec["Hq"] == H and spec["B"] == B and spec["n_q"] == 1
    keys = (spec["n_cache"] if name == "decode" else sum(spec["chunks"])) + 1
    d = spec["d"]
    assert spec["attn_flops"] == B * H * (matmul_flops(1, d, keys) + matmul_flops(1, keys, d))
