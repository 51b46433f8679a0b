"""Uniform asymmetric low-bit quantisation of one group (oracle, test infrastructure only).

Method: the cache stores keys and values at INT2 (and INT4) with a quantisation
step size per group ("Quantized Keys Steal Attention", abstract: the correction
is computed "from the quantization step sizes of the cached keys"; WindowQuant
note, table in 何が新しいのか: FP16 / INT4 / INT2 windows).  The pages give no
formula, so the scheme is the plain asymmetric min/max quantiser:

    m = min x_i,  M = max x_i           (valid members only)
    s = fl32(fl32(M - m) / (2^b - 1))   step size, fp32
    t_i = fl32(fl32(x_i - m) / s)
    code_i = clamp(rint_half_even(t_i), 0, 2^b - 1)   (code 0 everywhere if s == 0)
    z = m                                 zero point as an fp32 offset
    x_hat_i = fmaf(code_i, s, z)          one rounding

The decisions that produce integers (t_i and its rounding) are taken in fp32,
the precision the kernels use, so codes can be compared bit for bit.  ``-0.0``
as a minimum is canonicalised to ``+0.0`` (``m + 0.0``) so that stored bytes are
unique.

fp16 metadata (a cache variant that stores s and z as fp16, for the smaller
caches the WindowQuant note (主な結果) and the QuantWM card (Key Results) report):
s and z are the fp16 round-to-nearest-even of the fp32 s and m above (a ``-0``
zero point stored as ``+0``), and the codes are taken against the stored pair,

    t_i = fl32(fl32(x_i - z16) / s16),  code_i = clamp(rint(t_i), 0, 2^b - 1)
    (code 0 everywhere if s16 == 0),    x_hat_i = fmaf(code_i, s16, z16),

so that each code is the nearest level of the grid the cache actually holds,
and the dequantised entry is computed in fp16 arithmetic, one rounding of the
exact value (an fp16 fused multiply-add):

    x_hat_i = fp16_rne(code_i * s16 + z16).

The entry is then an fp16 number, as are the FP16 windows of a mixed cache
and the tensor-core operands.  Inputs stay within the fp16 range
(|x| <= 65504); beyond it s16 or z16 would be infinite.
"""

from __future__ import annotations

import numpy as np

F32 = np.float32
F64 = np.float64


def fma32(a, b, c):
    """Correctly rounded fp32 ``a*b + c`` (IEEE fusedMultiplyAdd, round to nearest even).

    Preconditions: a, b, c are fp32 values and ``a*b`` is exact in fp64, which
    holds when ``a`` is a small integer (a quantisation code, < 2^29).
    The fp64 sum ``p + c`` may be inexact; its rounding error is recovered with
    the TwoSum error-free transformation and used to settle the one case where
    rounding fp64 -> fp32 could differ from one correct rounding: an fp64 sum
    lying exactly half-way between two fp32 neighbours.
    """
    a64 = np.asarray(a, dtype=F32).astype(F64)
    b64 = np.asarray(b, dtype=F32).astype(F64)
    c64 = np.asarray(c, dtype=F32).astype(F64)
    p = a64 * b64                              # exact by precondition
    s = p + c64                                # one fp64 rounding
    bb = s - p                                 # TwoSum (Knuth): s + err == p + c exactly
    err = (p - (s - bb)) + (c64 - bb)
    r = s.astype(F32)                          # RNE fp64 -> fp32
    r64 = r.astype(F64)
    diff = s - r64                             # exact (r is a neighbour of s)
    toward = np.where(diff > 0, F32(np.inf), F32(-np.inf)).astype(F32)
    nb = np.nextafter(r, toward).astype(F32)
    half = (nb.astype(F64) - r64) / 2.0        # exact
    at_mid = (diff != 0) & (diff == half)
    # s is an fp32 midpoint and r was chosen by ties-to-even; the exact value
    # lies on the side of err, so move to the neighbour when err points to it.
    fix = at_mid & (err != 0) & (np.sign(err) == np.sign(diff))
    out = np.where(fix, nb, r).astype(F32)
    return out


def f16_round(x):
    """fp16 round-to-nearest-even of exact fp64 values, as fp64.

    Written from the format's definition: 11 significant bits, exponents down to
    -14 (below that the step stays 2^-24: subnormals), largest finite 65504;
    magnitudes that round beyond it become infinite.  The scaling by a power of
    two and np.rint (ties to even) are exact, so the result is one rounding.
    """
    x = np.asarray(x, dtype=F64)
    a = np.abs(x)
    _, e2 = np.frexp(np.where(a > 0, a, 1.0))          # a = m 2^e2, m in [0.5, 1)
    step = np.ldexp(1.0, np.maximum(e2 - 1, -14) - 10)
    y = np.rint(a / step) * step
    y = np.where(y > 65504.0, np.inf, y)
    return np.copysign(y, x)


def f16_rne(x):
    """fp16 round-to-nearest-even of fp32 values, returned as fp32 (exact widening)."""
    x = np.asarray(x, dtype=F32)
    return np.asarray(round_to(x, "f16"), dtype=F32).reshape(x.shape)


def quantize_groups(x, bits, n_valid=None, meta16=False):
    """Quantise groups laid out along the last axis.

    x       : fp32 array [..., n] (n <= 32 for the cache, any n here).
    bits    : 2 or 4.
    n_valid : members [0, n_valid) are real; the rest are padding (code 0,
              excluded from min/max).  ``None`` means all n are valid.
    meta16  : store s and z as fp16 and take the codes against them.

    Returns (codes uint8 [..., n], s fp32 [...], z fp32 [...]); with meta16
    s and z hold fp16 values.
    """
    x = np.asarray(x, dtype=F32)
    n = x.shape[-1]
    if n_valid is None:
        n_valid = n
    qmax = F32(2 ** bits - 1)
    xv = x[..., :n_valid]
    if n_valid == 0:
        shp = x.shape[:-1]
        return (np.zeros(x.shape, np.uint8), np.zeros(shp, F32), np.zeros(shp, F32))
    m = xv.min(axis=-1).astype(F32)
    mx = xv.max(axis=-1).astype(F32)
    m = (m + F32(0.0)).astype(F32)               # -0.0 -> +0.0
    D = (mx - m).astype(F32)
    s = ((D / qmax).astype(F32) + F32(0.0)).astype(F32)   # -0.0 -> +0.0
    if meta16:
        s = f16_rne(s)
        m = (f16_rne(m) + F32(0.0)).astype(F32)
    s_safe = np.where(s > 0, s, F32(1.0)).astype(F32)
    t = ((xv - m[..., None]).astype(F32) / s_safe[..., None]).astype(F32)
    code = np.clip(np.rint(t), 0, qmax)
    code = np.where((s > 0)[..., None], code, 0).astype(np.uint8)
    codes = np.zeros(x.shape, np.uint8)
    codes[..., :n_valid] = code
    return codes, s, m


def dequantize(codes, s, z, meta16=False):
    """x_hat = fmaf(code, s, z) in fp32 (single rounding); s, z broadcast against codes.

    meta16: s and z are fp16 values and x_hat = fp16_rne(code s + z), the value
    code s + z being exact in fp64 (code < 16 and two fp16 operands); returned as fp32.
    """
    codes = np.asarray(codes)
    s = np.broadcast_to(np.asarray(s, F32), codes.shape)
    z = np.broadcast_to(np.asarray(z, F32), codes.shape)
    if meta16:
        exact = codes.astype(F64) * s.astype(F64) + z.astype(F64)
        return f16_round(exact).astype(F32)
    return fma32(codes.astype(F32), s, z)


def round_to(x, dtype: str):
    """Round fp32/fp64 values to `dtype` with RNE and return them as fp64.

    dtype: 'f32', 'f16' or 'bf16' (torch's CPU conversions, which round to
    nearest even).
    """
    import torch
    t = torch.from_numpy(np.ascontiguousarray(np.asarray(x, dtype=F32)))
    if dtype == "f32":
        return t.double().numpy()
    if dtype == "f16":
        return t.to(torch.float16).double().numpy()
    if dtype == "bf16":
        return t.to(torch.bfloat16).double().numpy()
    raise ValueError(dtype)


def pack_codes(codes, bits):
    """Pack codes along the last axis into little-endian uint32 words.

    Element c of a row sits at bit ``bits * (c % (32 // bits))`` of word
    ``c // (32 // bits)``.  Returns uint32 [..., n * bits // 32].
    """
    codes = np.asarray(codes, dtype=np.uint32)
    per = 32 // bits
    n = codes.shape[-1]
    assert n % per == 0
    c = codes.reshape(codes.shape[:-1] + (n // per, per))
    shifts = (np.arange(per, dtype=np.uint32) * bits)
    return np.bitwise_or.reduce(c << shifts, axis=-1).astype(np.uint32)


def unpack_codes(words, bits, n):
    """Inverse of :func:`pack_codes`."""
    words = np.asarray(words, dtype=np.uint32)
    per = 32 // bits
    shifts = (np.arange(per, dtype=np.uint32) * bits)
    c = (words[..., None] >> shifts) & np.uint32(2 ** bits - 1)
    return c.reshape(words.shape[:-1] + (words.shape[-1] * per,))[..., :n].astype(np.uint8)
