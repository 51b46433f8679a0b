"""CUDA graph capture of the library's calls.  A decode call, a tensor-core call (with and
without its split merge) and an append are captured once with torch.cuda.graph and replayed;
the replays give the eager calls' results bit for bit, since the kernels are deterministic and
take their arguments as captured.  The decode call's merge kernel is launched with
programmatic stream serialisation, which capture keeps as a programmatic graph edge."""

import numpy as np
import pytest

from bit_kv_cache_28_b300 import bitkv as B
from bit_kv_cache_28_b300 import synth
from oracle import window as OW
from helpers import DT, gpu_mixed, gpu_uniform, to_dev, cache_bytes

pytestmark = pytest.mark.gpu


def _attention_call(tc, case, path, splits=0, jensen=1):
    import torch
    dt = case["dtype"]
    q, kc, vc = to_dev(case["Q"], dt), to_dev(case["K_cur"], dt), to_dev(case["V_cur"], dt)
    Bn, Hq, nq, d = q.shape
    n_cur = kc.shape[2]
    opts = B.kv_attn_opts(0.0, jensen, 0, 1, splits, path)
    wsb = B.kv_attention_workspace(tc.c, DT[dt], nq, n_cur, Hq, opts)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device="cuda")
    out = torch.empty((Bn, Hq, nq, d), dtype=torch.float32, device="cuda")
    lse = torch.empty((Bn, Hq, nq), dtype=torch.float32, device="cuda")

    def call(stream):
        B.kv_attention(q, kc, vc, DT[dt], nq, n_cur, Hq, tc.c, opts, out, lse, ws, wsb, stream)

    return call, out, lse, ws


def _check_replay(call, out, lse, ws):
    """Eager call on a side stream, then capture on it and replay three times."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call(side.cuda_stream)
    torch.cuda.synchronize()
    B.kv_attention_status(ws)
    ref_o, ref_l = out.clone(), lse.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        call(side.cuda_stream)
    for _ in range(3):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
        B.kv_attention_status(ws)


def _mixed(case):
    bits = np.stack([OW.window_plan(case["sim"][b], 0.2, 0.3)[0] for b in range(case["B"])])
    caps = [int((bits[0] == k).sum()) for k in (16, 4, 2)]
    return gpu_mixed(case, bits, caps)


@pytest.mark.parametrize("full", [False, True])
def test_decode_call_replays_bit_exact(full):
    """Small mixed case (uniform split counts) and the full decode workload (one wave of
    resident CTAs, streams with different split counts)."""
    case = synth.decode_case() if full else synth.decode_case(seed=81, B=3, Hq=6, Hkv=2, d=64, n_cache=1000)
    tc = _mixed(case)
    _check_replay(*_attention_call(tc, case, B.KV_PATH_DECODE))


@pytest.mark.parametrize("splits", [1, 3])
def test_tensor_core_call_replays_bit_exact(splits):
    case = synth.chunk_case(95, B=1, Hkv=2, d=128, chunks=[300, 260], n_cur=130, n_q=130, dtype="bf16")
    tc = gpu_uniform(case, 2)
    _check_replay(*_attention_call(tc, case, B.KV_PATH_TC, splits=splits))


def test_append_replays_bit_exact():
    """An append captured into a graph writes, on replay, the bytes the eager append writes."""
    import torch
    case = synth.chunk_case(17, B=2, Hkv=3, d=128, chunks=[200, 77], n_cur=8, n_q=8, dtype="bf16")
    cap_extra = 0
    eager = gpu_uniform(case, 2, cap_extra)
    first = dict(case, chunks=[200])
    graphed = gpu_uniform(first, 2, cap_extra=(77 + 31) // 32)
    K = to_dev(case["K_cache"][:, :, 200:277], "bf16")
    V = to_dev(case["V_cache"][:, :, 200:277], "bf16")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        B.kv_quantize_append(K, V, B.KV_BF16, 77, graphed.c, None, side.cuda_stream)
    g.replay()
    torch.cuda.synchronize()
    assert list(graphed.c.n_blocks) == list(eager.c.n_blocks) and graphed.c.n_tokens == eager.c.n_tokens
    for a, b in zip(cache_bytes(eager), cache_bytes(graphed)):
        assert np.array_equal(a, b)
