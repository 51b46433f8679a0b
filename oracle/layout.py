"""Packed-cache byte layout and cache builders (oracle, test infrastructure only).

The WindowQuant note (section 技術的に面白い点) stores windows of the same
bit-width together so that INT2, INT4 and FP16 blocks each stream well, and
(section 実装者視点で気になった点) uses 32-token windows whose tokens share one
bit-width.  "Quantized Keys Steal Attention" (abstract) packs the cache of each
finished chunk.  The byte format below is this library's own; the oracle
writes it independently of the CUDA packer so the two can be compared byte for
byte.

Block: 32 token slots of one (batch, kv-head).  Classes and their bytes, for
head dim d:

  INT2 / INT4 (b bits):  Kc  uint32[32][d*b/32]   key codes, token-major: channel c of
                                                  token t at word t*(d*b/32) + c/(32/b)
                         Km  float2[d]            per-channel (s, z) of the block
                         Vc  uint32[d][b]         value codes, channel-major: token t of
                                                  channel c at word c*b + t/(32/b)
                         Vm  float2[d/32][32]     per-(32-channel group, token) (s, z)
  RAW16:                 K   16-bit[32][d], then V 16-bit[32][d]  (fp16 or bf16),
                         each row's 16-byte chunks permuted: chunk j of token t's
                         row is stored at chunk position j XOR (t mod m), m = min(8, d/8)
  CODEBOOK2:             Kc  uint32[32][d/16]     2-bit centroid indices, token-major
                         Vc  uint32[d][2]         INT2 value codes, channel-major
                         Vm  float2[d/32][32]
                         Kq  fp16[32][rp]         PSAC coefficients, rp = ceil8(r)

fp16-metadata caches (a layout flag; INT2 / INT4 blocks only): Km is half2[d] and
Vm half2[d/32][32], each pair (s, z) as two fp16 values, so the block shrinks by
8 d bytes (d = 128 INT2: 4096 -> 3072 B); the quantiser then takes its codes
against the fp16 pair and dequantises in fp16 (oracle/quant.py).

Within a word, element i (channel for Kc, token for Vc) sits at bit
b*(i mod 32/b).  Keys are token-major because a key row feeds Q K^T;
values are channel-major because a value column feeds P V.  Pad slots
(a block's valid length < 32) hold code 0, zero value metadata and zero raw
entries.  Key groups are the blocks themselves: each appended chunk starts a
new block, so a 1560-token chunk gives 48 full blocks and one of 24 tokens.

Stream: for each (b, kv-head), segments in the order RAW16, INT4, INT2 (a
uniform cache has one INT segment; a codebook cache one CODEBOOK2 segment), each
holding ``cap[k]`` blocks.  Per-block valid lengths and logical start
positions are int32 arrays [B][sum(cap)], indexed segment-major.
"""

from __future__ import annotations

import numpy as np

from .quant import quantize_groups, dequantize, pack_codes, F32

BLOCK = 32
RAW16, INT4, INT2, CB2 = 0, 1, 2, 3
CLASS_BITS = {RAW16: 16, INT4: 4, INT2: 2, CB2: 2}


def ceil8(r):
    return (r + 7) // 8 * 8


def block_bytes(cls, d, r=0, meta16=False):
    if cls == RAW16:
        return 2 * BLOCK * d * 2
    if cls in (INT2, INT4):
        b = CLASS_BITS[cls]
        pair = 4 if meta16 else 8              # bytes of one (s, z)
        return 2 * (BLOCK * d * b // 8) + pair * d + BLOCK * (d // 32) * pair
    if cls == CB2:
        return 2 * (BLOCK * d * 2 // 8) + BLOCK * (d // 32) * 8 + BLOCK * ceil8(r) * 2
    raise ValueError(cls)


def stream_layout(classes, caps, d, r=0, meta16=False):
    """Segment byte offsets and stream bytes for segments ``classes`` with capacities ``caps``."""
    offs, o = [], 0
    for c, n in zip(classes, caps):
        offs.append(o)
        o += n * block_bytes(c, d, r, meta16)
    return offs, o


def _bits16(x, dtype):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(np.asarray(x, dtype=F32)))
    t = t.to(torch.float16 if dtype == "f16" else torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint8)


def _meta_bytes(sz, meta16):
    """(s, z) pairs [..., 2] as stored: fp32 pairs, or fp16 pairs under meta16."""
    if not meta16:
        return np.ascontiguousarray(sz, F32).view(np.uint8)
    return _bits16(sz, "f16")


def encode_int_blocks(Kb, Vb, bits, nvalid, meta16=False):
    """Quantise and pack N blocks that share one valid length.

    Kb, Vb: fp32 [N, 32, d].  Keys: one group per (block, channel) over the
    valid tokens.  Values: one group per (token, 32 consecutive channels).
    meta16: (s, z) stored as fp16 pairs (see oracle/quant.py).
    Returns a dict with the packed bytes [N, block_bytes] and the unpacked
    codes, steps and zero points, plus the dequantised fp32 entries.
    """
    Kb = np.asarray(Kb, F32)
    Vb = np.asarray(Vb, F32)
    N, T, d = Kb.shape
    assert T == BLOCK and d % 32 == 0
    kc, ks, kz = quantize_groups(Kb.transpose(0, 2, 1), bits, nvalid, meta16)   # [N,d,32]
    kc = np.ascontiguousarray(kc.transpose(0, 2, 1))                             # [N,32,d]
    vc, vs, vz = quantize_groups(Vb.reshape(N, T, d // 32, 32), bits, None, meta16)   # [N,32,d/32,32]
    vc[:, nvalid:] = 0
    vs[:, nvalid:] = 0
    vz[:, nvalid:] = 0
    kw = pack_codes(kc, bits)                                  # [N,32,d*b/32]
    vw = pack_codes(vc.reshape(N, T, d).transpose(0, 2, 1), bits)   # [N,d,b]
    km = np.stack([ks, kz], -1).astype(F32)                    # [N,d,2]
    vm = np.stack([vs, vz], -1).astype(F32).transpose(0, 2, 1, 3)   # [N,d/32,32,2]
    raw = np.concatenate([kw.reshape(N, -1).view(np.uint8), _meta_bytes(km, meta16).reshape(N, -1),
                          vw.reshape(N, -1).view(np.uint8), _meta_bytes(vm, meta16).reshape(N, -1)], axis=1)
    khat = dequantize(kc, ks[:, None, :], kz[:, None, :], meta16)
    vhat = dequantize(vc, vs[..., None], vz[..., None], meta16).reshape(N, T, d)
    return dict(bytes=raw, kcode=kc, ks=ks, kz=kz, vcode=vc.reshape(N, T, d), vs=vs, vz=vz,
                khat=khat, vhat=vhat)


def raw16_chunk_order(d):
    """Stored position of each 16-byte chunk of token t's row: ``order[t, j]`` for chunk j.

    The permutation is this library's own format choice: chunk j of row t goes
    to position j XOR (t mod m), m = min(8, d/8), so that eight consecutive rows
    of one chunk column fall into distinct shared-memory banks when a block is
    staged byte for byte.
    """
    nch = d // 8
    m = min(8, nch)
    t = np.arange(BLOCK)[:, None]
    j = np.arange(nch)[None, :]
    return j ^ (t % m)


def _swizzle_rows(rows16, d):
    """rows16: uint8 [N, 32, 2d] natural row bytes -> chunk-permuted rows."""
    N = rows16.shape[0]
    ch = rows16.reshape(N, BLOCK, d // 8, 16)
    out = np.empty_like(ch)
    order = raw16_chunk_order(d)
    for t in range(BLOCK):
        out[:, t, order[t]] = ch[:, t]
    return out.reshape(N, -1)


def encode_raw_blocks(Kb, Vb, nvalid, dtype):
    """RAW16 blocks: the 16-bit inputs unchanged (chunk-permuted per row), pad rows zero."""
    Kb = np.array(Kb, F32)
    Vb = np.array(Vb, F32)
    Kb[:, nvalid:] = 0
    Vb[:, nvalid:] = 0
    N, _, d = Kb.shape
    kr = _bits16(Kb, dtype).reshape(N, BLOCK, 2 * d)
    vr = _bits16(Vb, dtype).reshape(N, BLOCK, 2 * d)
    raw = np.concatenate([_swizzle_rows(kr, d), _swizzle_rows(vr, d)], axis=1)
    return dict(bytes=raw, khat=Kb, vhat=Vb)


class Cache:
    """Expected cache contents plus the logical (dequantised) view the attention oracle uses.

    data    : uint8 [B, H, stream_bytes]
    blk_len, blk_pos : int32 [B, sum(caps)]
    n_blocks: per-segment used blocks (equal across batch)
    tokens  : per (b, h) a dict of arrays over the valid cached tokens, in
              logical position order: khat, vhat (the exact dequantised fp32 entries),
              kgroup (block index of the token), quantised (bool: carries a
              key step size), and per block the key step sizes ks [nblk, d].
    """

    def __init__(self, B, H, d, classes, caps, r=0, meta16=False):
        self.B, self.H, self.d = B, H, d
        self.classes, self.caps, self.r, self.meta16 = list(classes), list(caps), r, meta16
        self.seg_off, self.stream_bytes = stream_layout(classes, caps, d, r, meta16)
        self.data = np.zeros((B, H, self.stream_bytes), np.uint8)
        ncap = int(sum(caps))
        self.blk_len = np.zeros((B, ncap), np.int32)
        self.blk_pos = np.zeros((B, ncap), np.int32)
        self.seg_base = np.concatenate([[0], np.cumsum(caps)[:-1]]).astype(int)
        self.n_blocks = [0] * len(classes)
        self.n_tokens = 0
        # logical view: list of block records per (b, h)
        self.blocks = [[[] for _ in range(H)] for _ in range(B)]

    def _put(self, b, h, seg, idx, raw):
        cls = self.classes[seg]
        bb = block_bytes(cls, self.d, self.r, self.meta16)
        o = self.seg_off[seg] + idx * bb
        self.data[b, h, o:o + bb] = raw

    def logical(self, b, h):
        """Valid cached tokens of (b, h) in logical order."""
        recs = sorted(self.blocks[b][h], key=lambda r: r["pos"])
        d = self.d
        kh = [r["khat"][:r["len"]] for r in recs]
        vh = [r["vhat"][:r["len"]] for r in recs]
        grp = [np.full(r["len"], i) for i, r in enumerate(recs)]
        out = dict(khat=np.concatenate(kh) if kh else np.zeros((0, d), F32),
                   vhat=np.concatenate(vh) if vh else np.zeros((0, d), F32),
                   kgroup=np.concatenate(grp) if grp else np.zeros(0, int),
                   ks=np.stack([r["ks"] for r in recs]) if recs else np.zeros((0, d), F32),
                   quantised=np.array([r["quantised"] for r in recs], bool),
                   coeff=(np.concatenate([r["coeff"][:r["len"]] for r in recs])
                          if recs and "coeff" in recs[0] else None))
        return out


def build_uniform(K, V, bits, appends, cap_blocks, meta16=False):
    """Cache of uniform INT{bits} blocks built by successive chunk appends.

    K, V: fp32 [B, H, n_total, d]; ``appends`` lists chunk lengths that sum to
    n_total.  Each chunk starts a new block (groups aligned to the chunk).
    meta16: blocks store their (s, z) as fp16.
    """
    K = np.asarray(K, F32)
    V = np.asarray(V, F32)
    B, H, n_total, d = K.shape
    assert sum(appends) == n_total
    cls = INT2 if bits == 2 else INT4
    c = Cache(B, H, d, [cls], [cap_blocks], meta16=meta16)
    t0 = 0
    for n in appends:
        nfull, tail = divmod(n, BLOCK)
        nb = nfull + (1 if tail else 0)
        assert c.n_blocks[0] + nb <= cap_blocks
        parts = []
        if nfull:
            parts.append((0, nfull, BLOCK))
        if tail:
            parts.append((nfull, 1, tail))
        for j0, cnt, nv in parts:
            Kb = np.zeros((B, H, cnt, BLOCK, d), F32)
            Vb = np.zeros((B, H, cnt, BLOCK, d), F32)
            a = t0 + j0 * BLOCK
            seg = K[:, :, a:a + cnt * nv]
            segv = V[:, :, a:a + cnt * nv]
            Kb[:, :, :, :nv] = seg.reshape(B, H, cnt, nv, d)
            Vb[:, :, :, :nv] = segv.reshape(B, H, cnt, nv, d)
            enc = encode_int_blocks(Kb.reshape(-1, BLOCK, d), Vb.reshape(-1, BLOCK, d), bits, nv, meta16)
            raw = enc["bytes"].reshape(B, H, cnt, -1)
            kh = enc["khat"].reshape(B, H, cnt, BLOCK, d)
            vh = enc["vhat"].reshape(B, H, cnt, BLOCK, d)
            ks = enc["ks"].reshape(B, H, cnt, d)
            kc = enc["kcode"].reshape(B, H, cnt, BLOCK, d)
            vcd = enc["vcode"].reshape(B, H, cnt, BLOCK, d)
            for b in range(B):
                for j in range(cnt):
                    idx = c.n_blocks[0] + j0 + j
                    c.blk_len[b, idx] = nv
                    c.blk_pos[b, idx] = c.n_tokens + (j0 + j) * BLOCK
                for h in range(H):
                    for j in range(cnt):
                        idx = c.n_blocks[0] + j0 + j
                        c._put(b, h, 0, idx, raw[b, h, j])
                        c.blocks[b][h].append(dict(pos=c.n_tokens + (j0 + j) * BLOCK, len=nv,
                                                   khat=kh[b, h, j], vhat=vh[b, h, j], ks=ks[b, h, j],
                                                   quantised=True, seg=0, slot=idx,
                                                   kcode=kc[b, h, j], vcode=vcd[b, h, j]))
        c.n_blocks[0] += nb
        c.n_tokens += n
        t0 += n
    return c


def build_mixed(K, V, window_bits, caps, dtype, meta16=False):
    """Mixed FP16/INT4/INT2 cache of one prefill, one class per 32-token window.

    K, V: fp32 [B, H, n, d] holding values exact in ``dtype`` ('f16'/'bf16').
    window_bits: int [B, W] with entries 16, 4 or 2; W = ceil(n / 32).
    Windows of one class are stored in ascending window order in their segment.
    meta16: INT blocks store their (s, z) as fp16.
    """
    K = np.asarray(K, F32)
    V = np.asarray(V, F32)
    B, H, n, d = K.shape
    W = (n + BLOCK - 1) // BLOCK
    window_bits = np.asarray(window_bits)
    assert window_bits.shape == (B, W)
    c = Cache(B, H, d, [RAW16, INT4, INT2], caps, meta16=meta16)
    cls_of = {16: 0, 4: 1, 2: 2}
    counts = None
    for b in range(B):
        cnt = [0, 0, 0]
        for w in range(W):
            seg = cls_of[int(window_bits[b, w])]
            t0, t1 = w * BLOCK, min(n, (w + 1) * BLOCK)
            nv = t1 - t0
            Kb = np.zeros((H, BLOCK, d), F32)
            Vb = np.zeros((H, BLOCK, d), F32)
            Kb[:, :nv] = K[b, :, t0:t1]
            Vb[:, :nv] = V[b, :, t0:t1]
            if seg == 0:
                enc = encode_raw_blocks(Kb, Vb, nv, dtype)
                ks = np.zeros((H, d), F32)
                kcd = vcd = [None] * H
            else:
                enc = encode_int_blocks(Kb, Vb, 4 if seg == 1 else 2, nv, meta16)
                ks = enc["ks"]
                kcd, vcd = enc["kcode"], enc["vcode"]
            idx = cnt[seg]
            cnt[seg] += 1
            assert idx < caps[seg]
            gidx = c.seg_base[seg] + idx
            c.blk_len[b, gidx] = nv
            c.blk_pos[b, gidx] = t0
            for h in range(H):
                c._put(b, h, seg, idx, enc["bytes"][h])
                c.blocks[b][h].append(dict(pos=t0, len=nv, khat=enc["khat"][h], vhat=enc["vhat"][h],
                                           ks=ks[h], quantised=seg != 0, seg=seg, slot=idx,
                                           kcode=kcd[h], vcode=vcd[h]))
        if counts is None:
            counts = cnt
        assert counts == cnt, "per-sequence segment counts must agree across the batch"
    c.n_blocks = counts
    c.n_tokens = n
    return c
