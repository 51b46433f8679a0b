"""Failure detection without a GPU fault.  Every device-side wait of the tensor-core and decode
kernels is bounded; BITKV_TEST_NEVER_ARRIVE makes one wait target a barrier that nothing
arrives on (with a short limit), so the kernel sets its status word and returns.  The call
reports KV_ERR_TIMEOUT at once under BITKV_DEBUG_SYNC, and otherwise through
kv_attention_status (kv_attention_noalloc_status for the no-workspace entry point); the next
call on the same context and workspace reports KV_OK and matches the oracle.  The range
flag of the tensor-core path's fp16 operands is reported the same way."""

import numpy as np
import pytest

from bit_kv_cache_28_b300 import bitkv as B
from bit_kv_cache_28_b300 import synth
from oracle import layout as OL
from oracle import attention as OA
from helpers import DT, gpu_uniform, run_attention, to_dev, assert_close, tol

pytestmark = pytest.mark.gpu


def _call(tc, case, path, jensen=1, Q=None):
    """One kv_attention call with its own workspace; returns (out, lse, workspace)."""
    import torch
    q = to_dev(case["Q"] if Q is None else Q, "bf16")
    Bn, Hq, nq, d = q.shape
    n_cur = case["K_cur"].shape[2]
    opts = B.kv_attn_opts(0.0, jensen, 0, 1, 0, path)
    wsb = B.kv_attention_workspace(tc.c, B.KV_BF16, nq, n_cur, Hq, opts)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    out = torch.empty((Bn, Hq, nq, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((Bn, Hq, nq), dtype=torch.float32, device="cuda")
    B.kv_attention(q, to_dev(case["K_cur"], "bf16"), to_dev(case["V_cur"], "bf16"), B.KV_BF16, nq, n_cur, Hq, tc.c,
                   opts, out, lse, ws, wsb)
    return out, lse, ws


def _oracle(case):
    oc = OL.build_uniform(case["K_cache"], case["V_cache"], 2, case["chunks"],
                          sum((n + 31) // 32 for n in case["chunks"]))
    return OA.attention_over_cache(oc, case["Q"], case["K_cur"], case["V_cur"], "bf16", jensen=1)


def _expect_timeout_then_recover(monkeypatch, tc, case, path):
    ref = _oracle(case)
    # (1) reported by the call itself under BITKV_DEBUG_SYNC
    monkeypatch.setenv("BITKV_DEBUG_SYNC", "1")
    monkeypatch.setenv("BITKV_TEST_NEVER_ARRIVE", "1")
    with pytest.raises(B.BitKVError) as e:
        run_attention(tc, case, jensen=1, out_f32=True, path=path)
    assert e.value.status == B.KV_ERR_TIMEOUT
    monkeypatch.delenv("BITKV_DEBUG_SYNC")
    # (2) without it: the call returns KV_OK, the status call reports the timeout
    _, _, ws = _call(tc, case, path)
    with pytest.raises(B.BitKVError) as e:
        B.kv_attention_status(ws)
    assert e.value.status == B.KV_ERR_TIMEOUT
    # (3) the next call on the same workspace clears the words and is correct
    monkeypatch.delenv("BITKV_TEST_NEVER_ARRIVE")
    import torch
    q = to_dev(case["Q"], "bf16")
    Bn, Hq, nq, d = q.shape
    opts = B.kv_attn_opts(0.0, 1, 0, 1, 0, path)
    out = torch.empty((Bn, Hq, nq, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((Bn, Hq, nq), dtype=torch.float32, device="cuda")
    B.kv_attention(q, to_dev(case["K_cur"], "bf16"), to_dev(case["V_cur"], "bf16"), B.KV_BF16, nq,
                   case["K_cur"].shape[2], Hq, tc.c, opts, out, lse, ws, ws.numel())
    B.kv_attention_status(ws)
    assert_close(out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ref[0], ref[1],
                 tol("bf16"))


def test_tc_bounded_wait_reports_timeout_and_context_survives(monkeypatch):
    case = synth.chunk_case(95, B=1, Hkv=2, d=128, chunks=[300], n_cur=130, n_q=130, dtype="bf16")
    _expect_timeout_then_recover(monkeypatch, gpu_uniform(case, 2), case, B.KV_PATH_TC)


def test_decode_bounded_wait_reports_timeout_and_context_survives(monkeypatch):
    case = synth.chunk_case(96, B=2, Hkv=2, Hq=4, d=128, chunks=[300, 77], n_cur=1, n_q=1, dtype="bf16")
    _expect_timeout_then_recover(monkeypatch, gpu_uniform(case, 2), case, B.KV_PATH_DECODE)


def test_noalloc_status_reports_timeout_then_ok(monkeypatch):
    import torch
    case = synth.chunk_case(97, B=1, Hkv=2, d=128, chunks=[300], n_cur=130, n_q=130, dtype="bf16")
    tc = gpu_uniform(case, 2)
    q = to_dev(case["Q"], "bf16")
    k, v = to_dev(case["K_cur"], "bf16"), to_dev(case["V_cur"], "bf16")
    out = torch.empty((1, 2, 130, 128), dtype=torch.float32, device="cuda")
    opts = B.kv_attn_opts(0.0, 1, 0, 1, 0, B.KV_PATH_TC)
    monkeypatch.setenv("BITKV_TEST_NEVER_ARRIVE", "1")
    B.kv_attention_noalloc(q, k, v, B.KV_BF16, 130, 130, 2, tc.c, opts, out, None)
    with pytest.raises(B.BitKVError) as e:
        B.kv_attention_noalloc_status()
    assert e.value.status == B.KV_ERR_TIMEOUT
    monkeypatch.delenv("BITKV_TEST_NEVER_ARRIVE")
    B.kv_attention_noalloc(q, k, v, B.KV_BF16, 130, 130, 2, tc.c, opts, out, None)
    B.kv_attention_noalloc_status()
    ref = _oracle(case)
    assert np.abs(out.cpu().numpy() - ref[0]).max() <= tol("bf16")


def test_tc_range_flag_for_queries_beyond_fp16():
    """A bf16 query entry of 70144 has no finite fp16 rounding: the tensor-core path (fp16
    operands) raises the range flag; the CUDA-core path (fp32 operands) is unaffected; a
    call with in-range queries on the same workspace reports KV_OK again."""
    case = synth.chunk_case(98, B=1, Hkv=1, d=128, chunks=[64], n_cur=32, n_q=32, dtype="bf16")
    tc = gpu_uniform(case, 2)
    Q = case["Q"].copy()
    Q[0, 0, 5, 17] = synth.to_bf16_values(np.array([70000.0], np.float32))[0]
    _, _, ws = _call(tc, case, B.KV_PATH_TC, jensen=0, Q=Q)
    with pytest.raises(B.BitKVError) as e:
        B.kv_attention_status(ws)
    assert e.value.status == B.KV_ERR_RANGE
    _, _, ws2 = _call(tc, case, B.KV_PATH_SIMT, jensen=0, Q=Q)
    B.kv_attention_status(ws2)
    _, _, ws3 = _call(tc, case, B.KV_PATH_TC, jensen=0)
    B.kv_attention_status(ws3)
