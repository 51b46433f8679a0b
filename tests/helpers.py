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


def gpu_uniform(case, bits, cap_extra=0):
    """Append every chunk of a chunk-case through kv_quantize_append."""
    dt = case["dtype"]
    cap = n_blocks_for(case["chunks"]) + cap_extra
    kind = B.KV_UNIFORM2 if bits == 2 else B.KV_UNIFORM4
    caps = (0, 0, cap) if bits == 2 else (0, cap, 0)
    tc = B.TorchCache(case["B"], case["Hkv"], case["d"], kind, caps)
    t0 = 0
    for n in case["chunks"]:
        K = to_dev(case["K_cache"][:, :, t0:t0 + n], dt)
        V = to_dev(case["V_cache"][:, :, t0:t0 + n], dt)
        B.kv_quantize_append(K, V, DT[dt], n, tc.c)
        t0 += n
    return tc


def gpu_mixed(case, window_bits, caps):
    import torch
    dt = case["dtype"]
    tc = B.TorchCache(case["B"], case["Hkv"], case["d"], B.KV_MIXED, caps, raw_dtype=DT[dt])
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


def bf16_half_ulp(x):
    """Half the bf16 spacing at |x| (the rounding error of storing x in bf16)."""
    a = np.maximum(np.abs(x), 1e-30)
    e = np.floor(np.log2(a))
    return 2.0 ** (e - 8)


def out_tol(dtype, out_f32, ref):
    """Per-element bound: 2e-3 for fp32 outputs; 1e-2 plus the output's own rounding for 16-bit outputs."""
    if out_f32 or dtype == "f32":
        return np.full(ref.shape, 2e-3)
    if dtype == "bf16":
        return 1e-2 + bf16_half_ulp(ref)
    return 1e-2 + np.maximum(np.abs(ref), 1e-30) * 2.0 ** -11
