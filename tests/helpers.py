"""Test helpers: drive the CUDA path through the C-ABI binding and the oracle on the same inputs."""

from __future__ import annotations

import numpy as np

from bit_kv_cache_28_b300 import bitkv as B

DT = {"f32": B.KV_F32, "f16": B.KV_F16, "bf16": B.KV_BF16}


def torch_dtype(name):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[name]


def to_dev(a, dtype, device="cuda"):
    """fp32 numpy holding dtype-exact values -> torch tensor of that dtype on the device (exact)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device).to(torch_dtype(dtype)).contiguous()


def n_blocks_for(chunks):
    return sum((n + 31) // 32 for n in chunks)


def gpu_uniform(case, bits, cap_extra=0, meta16=False):
    """Append every chunk of a chunk-case through kv_quantize_append (meta16: fp16 (s, z))."""
    dt = case["dtype"]
    cap = n_blocks_for(case["chunks"]) + cap_extra
    kind = B.KV_UNIFORM2 if bits == 2 else B.KV_UNIFORM4
    caps = (0, 0, cap) if bits == 2 else (0, cap, 0)
    tc = B.TorchCache(case["B"], case["Hkv"], case["d"], kind, caps, meta_dtype=B.KV_F16 if meta16 else B.KV_F32)
    t0 = 0
    for n in case["chunks"]:
        K = to_dev(case["K_cache"][:, :, t0:t0 + n], dt)
        V = to_dev(case["V_cache"][:, :, t0:t0 + n], dt)
        B.kv_quantize_append(K, V, DT[dt], n, tc.c)
        t0 += n
    return tc


def gpu_mixed(case, window_bits, caps, meta16=False):
    import torch
    dt = case["dtype"]
    tc = B.TorchCache(case["B"], case["Hkv"], case["d"], B.KV_MIXED, caps, raw_dtype=DT[dt],
                      meta_dtype=B.KV_F16 if meta16 else B.KV_F32)
    n = case["K_cache"].shape[2]
    wb = np.ascontiguousarray(window_bits, dtype=np.int8)
    wb_dev = torch.from_numpy(wb).cuda()
    opts = B.kv_append_opts(wb.ctypes.data, wb_dev.data_ptr())
    B.kv_quantize_append(to_dev(case["K_cache"], dt), to_dev(case["V_cache"], dt), DT[dt], n, tc.c, opts)
    torch.cuda.synchronize()
    return tc


def cache_bytes(tc):
    """(data [B,H,stream], blk_len [B,cap], blk_pos [B,cap]) of a TorchCache as numpy."""
    import torch
    torch.cuda.synchronize()
    L = tc.layout
    cap = sum(L.cap_blocks)
    data = tc.data.cpu().numpy().reshape(L.B, L.Hkv, -1)
    return data, tc.blk_len.cpu().numpy().reshape(L.B, cap), tc.blk_pos.cpu().numpy().reshape(L.B, cap)


def run_attention(tc, case, jensen=0, out_f32=False, path=B.KV_PATH_AUTO, splits=0, psac=0, Q=None, Kcur=None,
                  Vcur=None):
    import torch
    dt = case["dtype"]
    Q = case["Q"] if Q is None else Q
    Kcur = case["K_cur"] if Kcur is None else Kcur
    Vcur = case["V_cur"] if Vcur is None else Vcur
    Bn, Hq, nq, d = Q.shape
    n_cur = Kcur.shape[2]
    q = to_dev(Q, dt)
    kc = to_dev(Kcur, dt) if n_cur else None
    vc = to_dev(Vcur, dt) if n_cur else None
    opts = B.kv_attn_opts(0.0, jensen, psac, 1 if out_f32 else 0, splits, path)
    # out and lse sit between canary guard bands (16 KB of a fixed byte pattern on each
    # side), checked after the call: a kernel writing outside its outputs fails the test
    odt = torch.float32 if out_f32 else torch_dtype(dt)
    n_out, n_lse = Bn * Hq * nq * d, Bn * Hq * nq
    G = 16384
    ob = torch.full((2 * G + n_out * torch.empty((), dtype=odt).element_size(),), 0x5A, dtype=torch.uint8,
                    device="cuda")
    lb = torch.full((2 * G + 4 * n_lse,), 0x5A, dtype=torch.uint8, device="cuda")
    out = ob[G:G + n_out * torch.empty((), dtype=odt).element_size()].view(odt).view(Bn, Hq, nq, d)
    lse = lb[G:G + 4 * n_lse].view(torch.float32).view(Bn, Hq, nq)
    ws_bytes = B.kv_attention_workspace(tc.c, DT[dt], nq, n_cur, Hq, opts)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    B.kv_attention(q, kc, vc, DT[dt], nq, n_cur, Hq, tc.c, opts, out, lse, ws, ws_bytes)
    torch.cuda.synchronize()
    for buf, n in ((ob, ob.numel()), (lb, lb.numel())):
        assert bool((buf[:G] == 0x5A).all()) and bool((buf[n - G:] == 0x5A).all()), "write outside the output"
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def tol(io_dtype):
    """The required bound on outputs and lse against the oracle's definition: 2e-3 for fp32
    I/O; 1e-2 for 16-bit I/O (bf16 or fp16 inputs, whatever the output container)."""
    return 2e-3 if io_dtype == "f32" else 1e-2


TIGHT = 2e-3   # against the definition evaluated on a path's documented 16-bit operand storage


def assert_close(out, lse, ref_o, ref_lse, bound, rows=None, what=""):
    if rows is not None:
        out = out[:, :, rows]
        lse = lse[:, :, rows]
    err = np.abs(out - ref_o)
    worst = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= bound, f"{what}max err {err.max():.3e} at {worst} (bound {bound:.1e})"
    fin = np.isfinite(ref_lse)          # -inf: no key at all (empty cache, no current chunk)
    assert (np.isfinite(lse) == fin).all(), f"{what}lse finiteness differs"
    lerr = np.abs(lse[fin] - ref_lse[fin])
    assert lerr.max(initial=0.0) <= bound, f"{what}lse max err {lerr.max(initial=0.0):.3e} (bound {bound:.1e})"


def rne(x, dtype):
    """Round fp32 values to dtype (torch's CPU round-to-nearest-even) and back to fp64."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch_dtype(dtype)).double().numpy()


def assert_rounding_of(o16, o32, dtype):
    """A 16-bit output is the round-to-nearest-even of the same call's fp32 result, bit for bit."""
    exp = rne(o32, dtype)
    bad = np.flatnonzero(o16.ravel() != exp.ravel())
    assert bad.size == 0, f"{bad.size} 16-bit outputs are not the rounding of the fp32 result"


def attention_checked(tc, case, ref, io_dtype, tight=None, rows=None, **kw):
    """Runs kv_attention with an fp32 output and checks it (and the lse) against the oracle's
    definition `ref` = (o, lse) within tol(io_dtype), and against `tight` (the definition on the
    path's documented operand storage) within TIGHT if given; for 16-bit I/O runs it again with
    the 16-bit output and checks that output is the rounding of the first.  Returns (o, lse)."""
    o, l = run_attention(tc, case, out_f32=True, **kw)
    assert_close(o, l, ref[0], ref[1], tol(io_dtype), rows)
    if tight is not None:
        assert_close(o, l, tight[0], tight[1], TIGHT, rows, "operand storage: ")
    if io_dtype != "f32":
        o16, l16 = run_attention(tc, case, out_f32=False, **kw)
        assert_rounding_of(o16, o, io_dtype)
        assert np.array_equal(l16, l)
    return o, l
