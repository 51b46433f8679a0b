"""Failure detection without a GPU fault: every device-side wait of the tensor-core and
decode kernels is bounded.  BITKV_TEST_NEVER_ARRIVE makes one wait target a barrier that
nothing arrives on (with a short limit); the kernel must then set its error word and
return, the call must report KV_ERR_TIMEOUT under BITKV_DEBUG_SYNC, and the next call on
the same context must work."""

import numpy as np
import pytest

from bit_kv_cache_28_b300 import bitkv as B
from bit_kv_cache_28_b300 import synth
from oracle import layout as OL
from oracle import attention as OA
from helpers import gpu_uniform, run_attention, out_tol

pytestmark = pytest.mark.gpu


def _expect_timeout_then_recover(monkeypatch, tc, case, path, operands):
    monkeypatch.setenv("BITKV_DEBUG_SYNC", "1")
    monkeypatch.setenv("BITKV_TEST_NEVER_ARRIVE", "1")
    with pytest.raises(B.BitKVError) as e:
        run_attention(tc, case, jensen=1, out_f32=True, path=path)
    assert e.value.status == B.KV_ERR_TIMEOUT
    monkeypatch.delenv("BITKV_TEST_NEVER_ARRIVE")
    oc = OL.build_uniform(case["K_cache"], case["V_cache"], 2, case["chunks"],
                          sum((n + 31) // 32 for n in case["chunks"]))
    ro, rl = OA.attention_over_cache(oc, case["Q"], case["K_cur"], case["V_cur"], "bf16", jensen=1,
                                     operands=operands)
    o, l = run_attention(tc, case, jensen=1, out_f32=True, path=path)
    assert (np.abs(o - ro) <= out_tol("bf16", True, ro)).all()
    assert np.abs(l - rl).max() < 2e-3


def test_tc_bounded_wait_reports_timeout_and_context_survives(monkeypatch):
    case = synth.chunk_case(95, B=1, Hkv=2, d=128, chunks=[300], n_cur=130, n_q=130, dtype="bf16")
    _expect_timeout_then_recover(monkeypatch, gpu_uniform(case, 2), case, B.KV_PATH_TC, "io")


def test_decode_bounded_wait_reports_timeout_and_context_survives(monkeypatch):
    case = synth.chunk_case(96, B=2, Hkv=2, Hq=4, d=128, chunks=[300, 77], n_cur=1, n_q=1, dtype="bf16")
    _expect_timeout_then_recover(monkeypatch, gpu_uniform(case, 2), case, B.KV_PATH_DECODE, "f32")
