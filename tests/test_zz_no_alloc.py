"""kv_attention_noalloc: the attention entry point for callers that cannot allocate.

Some callers of this library run where they may not call cudaMalloc (host
callbacks, allocator hooks, plug-ins that are handed only their input and
output buffers).  kv_attention_noalloc serves them by keeping its scratch in a
fixed device array inside the library.  These tests call it through the C ABI
and compare it with kv_attention, which takes a caller-allocated workspace, on
consecutive calls that reuse the shared array.  The file sorts last so that a
run stopping at its first failure has already run every other test.
"""

import numpy as np
import pytest

from bit_kv_cache_28_b300 import bitkv as B
from bit_kv_cache_28_b300 import synth
from helpers import DT, gpu_uniform, run_attention, to_dev, tol
from helpers import assert_close as close_within
from oracle import layout as OL, attention as OA

pytestmark = pytest.mark.gpu


def run_noalloc(tc, case, jensen=0, out_f32=False, path=B.KV_PATH_AUTO, splits=0):
    import torch
    dt = case["dtype"]
    Bn, Hq, nq, d = case["Q"].shape
    n_cur = case["K_cur"].shape[2]
    opts = B.kv_attn_opts(0.0, jensen, 0, 1 if out_f32 else 0, splits, path)
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dt]
    out = torch.full((Bn, Hq, nq, d), float("nan"), dtype=torch.float32 if out_f32 else tdt, device="cuda")
    lse = torch.full((Bn, Hq, nq), float("nan"), dtype=torch.float32, device="cuda")
    B.kv_attention_noalloc(to_dev(case["Q"], dt), to_dev(case["K_cur"], dt), to_dev(case["V_cur"], dt), DT[dt], nq,
                           n_cur, Hq, tc.c, opts, out, lse)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def assert_close(o, l, ro, rl, dtype):
    assert np.isfinite(o).all() and np.isfinite(l).all()
    close_within(o, l, ro, rl, tol(dtype))


def test_noalloc_matches_kv_attention_on_consecutive_calls():
    """Split partials go through the shared array; each call must see none of the previous one's."""
    tc_case = synth.chunk_case(71, B=2, Hkv=2, Hq=4, d=128, chunks=[300, 77], n_cur=150, n_q=150, dtype="bf16")
    tc = gpu_uniform(tc_case, 2)
    f32_case = synth.tiny()
    tf = gpu_uniform(f32_case, 2)
    calls = [(tc, tc_case, dict(jensen=1, out_f32=False, path=B.KV_PATH_TC, splits=3)),
             (tf, f32_case, dict(jensen=2, out_f32=True, path=B.KV_PATH_SIMT, splits=4)),
             (tc, tc_case, dict(jensen=0, out_f32=True, path=B.KV_PATH_TC, splits=2))]
    for cache, case, kw in calls:
        ro, rl = run_attention(cache, case, **kw)
        for _ in range(2):
            o, l = run_noalloc(cache, case, **kw)
            assert_close(o, l, ro, rl, case["dtype"])
            B.kv_attention_noalloc_status()


def test_noalloc_fits_automatic_splits_into_the_array():
    """The 24-head chunk workload's automatic split count needs more scratch than the
    array holds; the call takes fewer splits.  Consecutive calls agree bit for bit, and
    sampled rows match the oracle (the split count changes the rounding of the fp16
    attention weights, so the two entry points are compared through the oracle rather
    than with each other)."""
    case = synth.chunk()
    tc = gpu_uniform(case, 2)
    n = case["Q"].shape[2]
    auto = B.kv_attn_opts(0.0, 1, 0, 1, 0, 0)
    _, splits = B.kv_attention_plan(tc.c, B.KV_BF16, n, n, 24, auto)
    assert B.kv_attention_workspace(tc.c, B.KV_BF16, n, n, 24, auto) > (32 << 20)
    # the count the call takes: the largest below the automatic one whose scratch fits
    fit = [sp for sp in range(splits - 1, 0, -1)
           if B.kv_attention_workspace(tc.c, B.KV_BF16, n, n, 24, B.kv_attn_opts(0.0, 1, 0, 1, sp, 0)) <= (32 << 20)]
    assert fit and fit[0] < splits
    o1, l1 = run_noalloc(tc, case, jensen=1, out_f32=True)
    o2, l2 = run_noalloc(tc, case, jensen=1, out_f32=True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    oc = OL.build_uniform(case["K_cache"], case["V_cache"], 2, case["chunks"],
                          sum((m + 31) // 32 for m in case["chunks"]))
    rows = np.random.default_rng(3).choice(n, 24, replace=False)
    for h in [2, 17]:
        view = OL.Cache(1, 1, 128, oc.classes, oc.caps)
        view.blocks = [[oc.blocks[0][h]]]
        ro, rl = OA.attention_over_cache(view, case["Q"][:, h:h + 1], case["K_cur"][:, h:h + 1],
                                         case["V_cur"][:, h:h + 1], "bf16", jensen=1, rows=rows)
        assert_close(o1[:, h:h + 1, rows], l1[:, h:h + 1, rows], ro, rl, "bf16")


def test_noalloc_rejects_scratch_beyond_the_array():
    import torch
    case = synth.chunk_case(72, B=1, Hkv=4, d=128, chunks=[64], n_cur=32, n_q=4096, dtype="bf16")
    tc = gpu_uniform(case, 2)
    q = to_dev(case["Q"], "bf16")
    k, v = to_dev(case["K_cur"], "bf16"), to_dev(case["V_cur"], "bf16")
    out = torch.empty_like(q)
    opts = B.kv_attn_opts(0.0, 0, 0, 0, 8, B.KV_PATH_TC)
    need = B.kv_attention_workspace(tc.c, B.KV_BF16, 4096, 32, 4, opts)
    assert need > (32 << 20)
    with pytest.raises(B.BitKVError) as ei:
        B.kv_attention_noalloc(q, k, v, B.KV_BF16, 4096, 32, 4, tc.c, opts, out, None)
    assert ei.value.status == B.KV_ERR_WORKSPACE
    assert "fixed array" in str(ei.value)
