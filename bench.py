"""Benchmark of the quantised-KV attention hot path (one JSON line on rank 0).

Workloads (seeded synthetic inputs; no dataset exists for this path, shapes
follow the chunk-wise video-diffusion and video-VLM settings of the pages):

* ``rollout`` (default; the largest single-GPU workload): 40 heads, d 128, bf16;
  the 1560 queries of the current chunk attend to a cache of 21 INT2 chunks
  (32760 tokens) plus the chunk itself with the Jensen correction on, then the
  finished chunk is quantised and appended.  One step = attention + append; the
  cache is rewound on the host after each step so every step sees the same cache.
* ``chunk``: the same with 24 heads and 3 cached chunks (4680 tokens).
* ``decode``: batch 8, 28 query heads over 4 kv heads, d 64, fp16; one query per
  sequence attends to 19600 cached tokens in 613 windows of FP16 / INT4 / INT2
  (planned by kv_window_plan from a seeded similarity) plus its own token.
  One step = one split-K decode attention.
* ``codebook``: 24 heads, d 128, bf16; 1560 queries over 8192 cached tokens with
  codebook keys (4 centroids per channel from a device k-means of the cached keys,
  weighted by 256 historical queries) and INT2 values, plus the chunk itself, with the
  rank-8 PSAC logit term; then the chunk is appended.  Calibration runs once, outside
  the step, and is reported as ``calibration_ms``.
* ``rollout_decode``: the rollout cache (40 heads, d 128, 21 INT2 chunks = 32760 tokens)
  read by one decode query per head plus its own token, Jensen on: the streaming path
  over a video-diffusion cache.  One step = one split-K decode attention.
* ``tiny``: 1 head, d 64, fp32, 1024 cached + 64 current tokens.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload rollout|chunk|decode|codebook|rollout_decode|tiny]
                    [--jensen 0|1|2|3] [--meta16]

``--meta16`` stores the INT blocks' step and zero point as fp16 pairs (not for codebook):
an INT2 block at d 128 is 3072 bytes instead of 4096.
    python bench.py --impl reference ...   # the CPU oracle, timed on the host cores

N > 1 runs independent replicas (weak scaling): every rank owns its own
workload; no data moves between ranks, the process group only carries the
barrier and the max-over-ranks of the timings.
"""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized-KV attention cache GB/s and query-tokens/s, % of HBM/TC roofline"
L2_FLUSH_BYTES = 512 << 20
L2_BYTES = 126 << 20        # B300 L2


# ------------------------------------------------------------ workloads ----

def workload_spec(name):
    """Shapes and algorithmic bytes / FLOPs of one step."""
    if name in ("chunk", "rollout"):
        H = 24 if name == "chunk" else 40
        n_chunks = 3 if name == "chunk" else 21
        n, d = 1560, 128
        n_cache = n * n_chunks
        groups = n_chunks * ((n + 31) // 32)
        cache_bytes = H * n_cache * d * 2 * 2 / 8 + H * groups * d * 8 + H * n_cache * (d // 32) * 8
        flops = 4.0 * n * (n_cache + n) * d * H
        append_read = 2 * H * n * d * 2
        append_write = H * ((n + 31) // 32) * 4096
        return dict(name=name, kind="chunk", B=1, Hkv=H, Hq=H, d=d, n_q=n, n_cur=n, chunks=[n] * n_chunks,
                    dtype="bf16", cache_bytes=cache_bytes, attn_flops=flops, append_bytes=append_read + append_write,
                    jensen=1, seed=2 if name == "chunk" else 3,
                    label=f"{name}: B1 H{H} d{d} chunk {n} cache {n_cache} INT2, Jensen taylor2")
    if name == "tiny":
        d, n_cache, n = 64, 1024, 64
        cache_bytes = n_cache * d * 2 * 2 / 8 + (n_cache // 32) * d * 8 + n_cache * (d // 32) * 8
        return dict(name=name, kind="chunk", B=1, Hkv=1, Hq=1, d=d, n_q=n, n_cur=n, chunks=[1024], dtype="f32",
                    cache_bytes=cache_bytes, attn_flops=4.0 * n * (n_cache + n) * d,
                    append_bytes=2 * n * d * 4 + 2 * 2048, jensen=1, seed=1,
                    label="tiny: B1 H1 d64 chunk 64 cache 1024 INT2 fp32, Jensen taylor2")
    if name == "codebook":
        H, d, n_cache, n, r = 24, 128, 8192, 1560, 8
        rp = (r + 7) // 8 * 8
        blk = 24 * d + 32 * rp * 2                      # key indices | value codes | value (s, z) | coefficients
        cache_bytes = H * (n_cache // 32) * blk
        flops = 4.0 * n * (n_cache + n) * d * H + 2.0 * n * n_cache * r * H
        return dict(name=name, kind="chunk", B=1, Hkv=H, Hq=H, d=d, n_q=n, n_cur=n, chunks=[n_cache], r=r,
                    n_hist=256, dtype="bf16", cache_bytes=cache_bytes, attn_flops=flops,
                    append_bytes=2 * H * n * d * 2 + H * ((n + 31) // 32) * blk, jensen=0, psac=1, seed=5,
                    label=f"codebook: B1 H{H} d{d} chunk {n} cache {n_cache} codebook INT2 keys (4 centroids per "
                          f"channel, device k-means) + INT2 values, PSAC rank {r}")
    if name == "rollout_decode":
        H, n, d, n_chunks = 40, 1560, 128, 21
        n_cache = n * n_chunks
        groups = n_chunks * ((n + 31) // 32)
        cache_bytes = H * n_cache * d * 2 * 2 / 8 + H * groups * d * 8 + H * n_cache * (d // 32) * 8
        return dict(name=name, kind="chunkdecode", B=1, Hkv=H, Hq=H, d=d, n_q=1, n_cur=1, chunks=[n] * n_chunks,
                    dtype="bf16", cache_bytes=cache_bytes, attn_flops=4.0 * H * (n_cache + 1) * d,
                    append_bytes=0, jensen=1, seed=3,
                    label=f"rollout_decode: B1 H{H} d{d}, one query per head over {n_cache} INT2 cached tokens "
                          "(21 chunks) + its own token, Jensen taylor2, split-K")
    if name == "decode":
        B, Hq, Hkv, d, n_cache = 8, 28, 4, 64, 19600
        return dict(name=name, kind="decode", B=B, Hkv=Hkv, Hq=Hq, d=d, n_q=1, n_cur=1, n_cache=n_cache,
                    dtype="f16", jensen=0, seed=4, attn_flops=4.0 * B * Hq * (n_cache + 1) * d,
                    label=f"decode: B{B} Hq{Hq} Hkv{Hkv} d{d} 1 query, cache {n_cache} tokens in 32-token "
                          "windows FP16/INT4/INT2 20/30/50%, split-K")
    raise ValueError(f"unknown workload {name}")


def make_inputs(spec):
    from bit_kv_cache_28_b300 import synth
    if spec["name"] == "tiny":
        return synth.tiny(spec["seed"])
    if spec["kind"] == "decode":
        return synth.decode_case(spec["seed"])
    if spec["name"] == "codebook":
        return synth.codebook_case(spec["seed"])
    if spec["kind"] == "chunkdecode":
        return synth.chunk_case(spec["seed"], Hkv=spec["Hkv"], chunks=spec["chunks"], n_cur=1, n_q=1)
    return synth.chunk_case(spec["seed"], Hkv=spec["Hkv"], chunks=spec["chunks"], n_cur=spec["n_cur"])


# --------------------------------------------------------------- clocks ----

class _Nvml:
    """Read-only NVML queries through the driver's libnvidia-ml (ctypes): SM clock, maximum
    SM clock and the active clock-event reasons."""

    NVML_CLOCK_SM = 1

    def __init__(self):
        import ctypes as C
        self.C = C
        self.lib = C.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")

    def handle(self, dev_index):
        C = self.C
        h = C.c_void_p()
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(dev_index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            if self.lib.nvmlDeviceGetHandleByUUID(C.c_char_p(uuid.encode()), C.byref(h)) == 0:
                return h
        except Exception:
            pass
        if self.lib.nvmlDeviceGetHandleByIndex_v2(C.c_uint(dev_index), C.byref(h)) != 0:
            raise RuntimeError("no NVML handle")
        return h

    def clock(self, h, maximum=False):
        v = self.C.c_uint()
        f = self.lib.nvmlDeviceGetMaxClockInfo if maximum else self.lib.nvmlDeviceGetClockInfo
        if f(h, self.C.c_int(self.NVML_CLOCK_SM), self.C.byref(v)) != 0:
            raise RuntimeError("clock query failed")
        return float(v.value)

    def reasons(self, h):
        v = self.C.c_ulonglong()
        f = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        if f(h, self.C.byref(v)) != 0:
            raise RuntimeError("reason query failed")
        return int(v.value)


class ClockSampler:
    """SM clock and throttle reasons of this process's GPU, sampled through NVML every 2 ms on
    a background thread from before the warm-up to the end of the timed steps (nvidia-smi
    every 200 ms if NVML cannot be loaded)."""

    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}

    def __init__(self, dev_index):
        self.dev_index = dev_index
        self.rows = []
        self.nvml = None
        self.stop = threading.Event()
        self.thread = None
        self.proc = None
        self.error = None

    def _loop(self, h):
        try:
            mx = self.nvml.clock(h, maximum=True)
        except Exception as e:  # pragma: no cover - depends on the driver
            mx, self.error = float("nan"), repr(e)
        while not self.stop.is_set():
            try:
                sm = self.nvml.clock(h)
                try:
                    rs = self.nvml.reasons(h)
                except Exception as e:
                    rs, self.error = 0, repr(e)
                self.rows.append((sm, mx, rs))
            except Exception as e:
                self.error = repr(e)
            self.stop.wait(0.002)

    def __enter__(self):
        try:
            self.nvml = _Nvml()
            h = self.nvml.handle(self.dev_index)
            self.thread = threading.Thread(target=self._loop, args=(h,), daemon=True)
            self.thread.start()
        except Exception as e:
            self.error = repr(e)
            self.nvml = None
            self.path = os.path.join("/tmp", f"bitkv_clocks_{os.getpid()}.csv")
            try:
                self.fh = open(self.path, "w")
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.dev_index), "--query-gpu=clocks.sm,clocks.max.sm,"
                     "clocks_event_reasons.active", "--format=csv,noheader,nounits", "-lms", "200"],
                    stdout=self.fh, stderr=subprocess.DEVNULL)
            except (OSError, FileNotFoundError):
                self.proc = None
        return self

    def __exit__(self, *a):
        if self.thread is not None:
            self.stop.set()
            self.thread.join(timeout=2)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()
            for line in open(self.path):
                p = [x.strip() for x in line.split(",")]
                try:
                    self.rows.append((float(p[0]), float(p[1]), int(p[2], 16)))
                except (ValueError, IndexError):
                    continue

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0,
                    "error": self.error}
        sm = [r[0] for r in self.rows]
        reasons = sorted({name for r in self.rows for bit, name in self.REASONS.items() if r[2] & bit})
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(r[1] for r in self.rows), "reasons": reasons,
                "samples": len(self.rows), "source": "nvml" if self.nvml is not None else "nvidia-smi"}


# ----------------------------------------------------------- own arm -------

class L2Flush:
    """Evicts L2 between timed steps: writes a buffer four times the L2's size, then reads
    another as large.  The read makes L2 write back the written lines before the timed
    region; after a write alone, L2 is left full of dirty lines, and their write-back lands
    inside the next timed kernel (about 80 MB of extra DRAM writes for an 80 MB read)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)

    def __call__(self, k):
        self.w.fill_(k & 0xFF)
        self.r.sum()


def pack_inputs(tensors):
    """The step's input tensors as views of one contiguous device buffer (each view 16-byte
    aligned), so that a step's inputs arrive in one host-to-device copy; returns (flat, views)."""
    import torch
    align = 16 // tensors[0].element_size()
    offs, o = [], 0
    for t in tensors:
        offs.append(o)
        o += (t.numel() + align - 1) // align * align
    flat = torch.zeros(o, dtype=tensors[0].dtype, device=tensors[0].device)
    views = views_of(flat, offs, [t.shape for t in tensors])
    for v, t in zip(views, tensors):
        v.copy_(t)
    return flat, views


def views_of(flat, offs, shapes):
    import math
    return [flat[a:a + math.prod(sh)].view(sh) for a, sh in zip(offs, shapes)]


def input_layout(r):
    """(offsets, shapes) of a runner's input views inside its flat buffer."""
    base = r.in_flat.data_ptr()
    es = r.in_flat.element_size()
    return [(t.data_ptr() - base) // es for t in r.inputs], [t.shape for t in r.inputs]


class ChunkRunner:
    """Device state of one replica of a chunk workload: the cache after the
    workload's cached chunks, and the step inputs."""

    def __init__(self, spec, inputs, dev):
        import torch
        from bit_kv_cache_28_b300 import bitkv as B
        self.B, self.spec, self.dev = B, spec, dev
        tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[spec["dtype"]]
        self.dt = {"bf16": B.KV_BF16, "f16": B.KV_F16, "f32": B.KV_F32}[spec["dtype"]]
        to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev).to(tdt)
        nb_cache = sum((n + 31) // 32 for n in spec["chunks"])
        nb_cur = (spec["n_cur"] + 31) // 32
        r = spec.get("r", 0)
        kind = B.KV_CODEBOOK2 if spec["name"] == "codebook" else B.KV_UNIFORM2
        self.tc = B.TorchCache(spec["B"], spec["Hkv"], spec["d"], kind, (0, 0, nb_cache + nb_cur),
                               raw_dtype=B.KV_BF16, psac_rank=r, device=dev,
                               meta_dtype=B.KV_F16 if spec.get("meta16") else B.KV_F32)
        self.calib_ms = None
        if kind == B.KV_CODEBOOK2:
            # calibration of the prefill on the device: per-channel centroids of the cached keys,
            # the PSAC basis of the historical queries
            K = to(inputs["K_cache"])
            Qh = to(inputs["Q_hist"][None])
            ws_b = B.kv_psac_workspace(self.tc.layout)
            ws = torch.empty(max(ws_b, 16), dtype=torch.uint8, device=dev)
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            wts = torch.zeros((1, spec["Hkv"], spec["d"]), dtype=torch.float32, device=dev)
            B.kv_codebook_fit(K, self.dt, K.shape[2], self.tc.c, 20, Qh, spec["n_hist"], wts)
            B.kv_psac_basis(Qh, self.dt, spec["n_hist"], self.tc.c, None, ws, ws_b)
            e1.record()
            torch.cuda.synchronize(dev)
            self.calib_ms = e0.elapsed_time(e1)
        t0 = 0
        for n in spec["chunks"]:
            B.kv_quantize_append(to(inputs["K_cache"][:, :, t0:t0 + n]), to(inputs["V_cache"][:, :, t0:t0 + n]),
                                 self.dt, n, self.tc.c)
            t0 += n
        self.saved = (list(self.tc.c.n_blocks), self.tc.c.n_tokens)
        self.in_flat, self.inputs = pack_inputs([to(inputs["Q"]), to(inputs["K_cur"]), to(inputs["V_cur"])])
        self.Q, self.Kc, self.Vc = self.inputs
        self.opts = B.kv_attn_opts(0.0, spec["jensen"], spec.get("psac", 0), 0, 0, B.KV_PATH_AUTO)
        self.out = torch.empty_like(self.Q)
        self.lse = torch.empty(self.Q.shape[:3], dtype=torch.float32, device=dev)
        self.ws_bytes = B.kv_attention_workspace(self.tc.c, self.dt, spec["n_q"], spec["n_cur"], spec["Hq"],
                                                 self.opts)
        self.ws = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=dev)
        self.path, self.splits = B.kv_attention_plan(self.tc.c, self.dt, spec["n_q"], spec["n_cur"], spec["Hq"],
                                                     self.opts)
        # attention kernel (+ one merge launch when the key range is split) + one append launch
        self.launches_per_step = 2 + (1 if self.splits > 1 else 0)
        self.cache_bytes = spec["cache_bytes"]

    def rewind(self):
        n_blocks, n_tok = self.saved
        for i in range(3):
            self.tc.c.n_blocks[i] = n_blocks[i]
        self.tc.c.n_tokens = n_tok

    def attention(self, stream):
        s = self.spec
        self.B.kv_attention(self.Q, self.Kc, self.Vc, self.dt, s["n_q"], s["n_cur"], s["Hq"], self.tc.c, self.opts,
                            self.out, self.lse, self.ws, self.ws_bytes, stream)

    def append(self, stream):
        s = self.spec
        self.B.kv_quantize_append(self.Kc, self.Vc, self.dt, s["n_cur"], self.tc.c, None, stream)
        self.rewind()


class DecodeRunner:
    """Device state of one replica of the decode workload: the mixed cache of one prefill
    (window bit-widths from kv_window_plan) and the step's query and current token."""

    def __init__(self, spec, inputs, dev):
        import torch
        from bit_kv_cache_28_b300 import bitkv as B
        self.B, self.spec, self.dev = B, spec, dev
        self.dt = B.KV_F16
        to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev).to(torch.float16)
        Bn, n, d, Hkv = spec["B"], spec["n_cache"], spec["d"], spec["Hkv"]
        W = (n + 31) // 32
        bits = np.zeros((Bn, W), np.int8)
        th = B.kv_thresholds(0.2, 0.3, 1)
        for b in range(Bn):
            B.kv_window_plan(np.ascontiguousarray(inputs["sim"][b], np.float32), W, th, bits[b])
        caps = [int((bits[0] == k).sum()) for k in (16, 4, 2)]
        m16 = bool(spec.get("meta16"))
        self.tc = B.TorchCache(Bn, Hkv, d, B.KV_MIXED, caps, raw_dtype=B.KV_F16, device=dev,
                               meta_dtype=B.KV_F16 if m16 else B.KV_F32)
        bits_dev = torch.from_numpy(bits).to(dev)
        self.K_cache = to(inputs["K_cache"])
        B.kv_quantize_append(self.K_cache, to(inputs["V_cache"]), self.dt, n, self.tc.c,
                             B.kv_append_opts(bits.ctypes.data, bits_dev.data_ptr()))
        torch.cuda.synchronize(dev)
        # algorithmic cache bytes: codes of valid tokens + all metadata (key and value pairs,
        # 2 d of each per block); 16-bit windows' valid rows
        bl = self.tc.blk_len.cpu().numpy().reshape(Bn, -1)
        nb = list(self.tc.c.n_blocks)
        lens = [bl[:, :nb[0]], bl[:, nb[0]:nb[0] + nb[1]], bl[:, nb[0] + nb[1]:nb[0] + nb[1] + nb[2]]]
        meta = (8 if m16 else 16) * d
        per_b = (lens[0].sum(1) * 2 * d * 2 + lens[1].sum(1) * 2 * d * 4 / 8 + nb[1] * meta
                 + lens[2].sum(1) * 2 * d * 2 / 8 + nb[2] * meta)
        self.cache_bytes = float(per_b.sum() * Hkv)
        self.in_flat, self.inputs = pack_inputs([to(inputs["Q"]), to(inputs["K_cur"]), to(inputs["V_cur"])])
        self.Q, self.Kc, self.Vc = self.inputs
        self.opts = B.kv_attn_opts(0.0, spec["jensen"], 0, 0, 0, B.KV_PATH_AUTO)
        self.out = torch.empty_like(self.Q)
        self.lse = torch.empty(self.Q.shape[:3], dtype=torch.float32, device=dev)
        self.ws_bytes = B.kv_attention_workspace(self.tc.c, self.dt, 1, 1, spec["Hq"], self.opts)
        self.ws = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=dev)
        self.path, self.splits = B.kv_attention_plan(self.tc.c, self.dt, 1, 1, spec["Hq"], self.opts)
        self.launches_per_step = 2   # the decode kernel and its split merge

    def attention(self, stream):
        s = self.spec
        self.B.kv_attention(self.Q, self.Kc, self.Vc, self.dt, 1, 1, s["Hq"], self.tc.c, self.opts, self.out,
                            self.lse, self.ws, self.ws_bytes, stream)

    def append(self, stream):
        pass

    def time_window_similarity(self, flush, steps, stream):
        """The window-similarity kernel over this workload's cache keys, the current token
        standing in for the question: mean seconds per call (L2 flushed before each) and
        the keys' bytes it reads."""
        import torch
        s = self.spec
        Bn, Hkv, n, d = s["B"], s["Hkv"], s["n_cache"], s["d"]
        sim = torch.empty((Bn, (n + 31) // 32), dtype=torch.float32, device=self.dev)
        run = lambda: self.B.kv_window_similarity(self.K_cache, self.Kc, self.dt, Bn, Hkv, n, 1, d, sim, stream)
        for _ in range(3):
            run()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for k in range(steps):
            flush(k)
            ev[k][0].record(torch.cuda.current_stream(self.dev))
            run()
            ev[k][1].record(torch.cuda.current_stream(self.dev))
        torch.cuda.synchronize(self.dev)
        t = sum(a.elapsed_time(b) for a, b in ev) / steps * 1e-3
        return t, float(self.K_cache.numel() * self.K_cache.element_size())


def with_jensen(spec, jensen):
    """The workload with its Jensen mode overridden (None keeps the workload's own)."""
    if jensen is None or jensen == spec["jensen"]:
        return spec
    names = {0: "off", 1: "taylor2", 2: "exact", 3: "isotropic"}
    spec = dict(spec, jensen=jensen)
    spec["label"] = spec["label"].replace("Jensen taylor2", f"Jensen {names[jensen]}")
    if "Jensen" not in spec["label"]:
        spec["label"] += f", Jensen {names[jensen]}"
    return spec


def with_meta16(spec, on):
    """The workload on a cache with fp16 (s, z) metadata: the algorithmic cache and append
    bytes count 4-byte pairs instead of 8-byte ones."""
    if not on:
        return spec
    if spec["name"] == "codebook":
        raise SystemExit("--meta16: codebook caches keep fp32 metadata")
    spec = dict(spec, meta16=True)
    if spec["kind"] in ("chunk", "chunkdecode"):
        H, d, chunks = spec["Hkv"], spec["d"], spec["chunks"]
        n_cache = sum(chunks)
        groups = sum((n + 31) // 32 for n in chunks)
        spec["cache_bytes"] = H * n_cache * d * 2 * 2 / 8 + H * groups * d * 4 + H * n_cache * (d // 32) * 4
        if spec["kind"] == "chunk":
            n = spec["n_cur"]
            spec["append_bytes"] = (2 * H * n * d * (4 if spec["dtype"] == "f32" else 2)
                                    + H * ((n + 31) // 32) * (32 * d * 2 * 2 // 8 + 8 * d))
    spec["label"] += ", fp16 (s, z) metadata"
    return spec


def max_over_ranks(times, dist, device):
    """Each timing (seconds) as the slowest rank measured it: the job's step ends when its
    last replica does."""
    import torch
    tt = torch.tensor(times, dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return tt.tolist()


def capture_step(r, spec, dev, stream):
    """CUDA graphs of the step's attention call and of its append (when the workload appends),
    captured once on a side stream; returns functions that replay them on `stream`.  The
    graphs hold the calls' kernels with their arguments as captured: the same buffers and the
    same cache length (the append re-appends the same blocks each replay, as the rewind does)."""
    import torch
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        r.attention(side.cuda_stream)
        r.append(side.cuda_stream)
    stream.wait_stream(side)
    torch.cuda.synchronize(dev)
    ga = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ga, stream=side):
        r.attention(side.cuda_stream)
    gp = None
    if spec["kind"] == "chunk":
        gp = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gp, stream=side):
            r.append(side.cuda_stream)
    torch.cuda.synchronize(dev)

    def replay(g):
        with torch.cuda.stream(stream):
            g.replay()

    return (lambda: replay(ga)), ((lambda: replay(gp)) if gp is not None else (lambda: None))


def e2e_pipelined(r, hin, hO, steps, stream, dev):
    """Seconds per step of the end-to-end loop with the copies overlapped: step k+1's inputs go
    host -> device on one copy stream and step k's output device -> host on another while step
    k computes; device inputs and outputs are double-buffered, and every step still copies its
    own inputs in and its own output out.  Timed with one event pair around all steps."""
    import torch
    flats = [r.in_flat, torch.empty_like(r.in_flat)]
    offs, shapes = input_layout(r)
    sets = [list(r.inputs), views_of(flats[1], offs, shapes)]
    outs = [r.out, torch.empty_like(r.out)]
    hOs = [hO, torch.empty_like(hO).pin_memory()]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    done = [torch.cuda.Event(), torch.cuda.Event()]      # the step that used buffer b has computed
    fetched = [torch.cuda.Event(), torch.cuda.Event()]   # its output has reached the host
    loaded = [torch.cuda.Event(), torch.cuda.Event()]    # inputs of the next user of buffer b are in
    for e in done + fetched:
        e.record(stream)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    up.wait_event(t0)
    down.wait_event(t0)

    def load(k):
        b = k % 2
        up.wait_event(done[b])
        with torch.cuda.stream(up):
            flats[b].copy_(hin, non_blocking=True)
        loaded[b].record(up)

    sh = stream.cuda_stream
    load(0)
    for k in range(steps):
        b = k % 2
        if k + 1 < steps:
            load(k + 1)
        stream.wait_event(loaded[b])
        stream.wait_event(fetched[b])
        r.Q, r.Kc, r.Vc = sets[b]
        r.out = outs[b]
        r.attention(sh)
        r.append(sh)
        done[b].record(stream)
        down.wait_event(done[b])
        with torch.cuda.stream(down):
            hOs[b].copy_(outs[b], non_blocking=True)
        fetched[b].record(down)
    stream.wait_stream(down)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    r.Q, r.Kc, r.Vc = sets[0]
    r.out = outs[0]
    return t0.elapsed_time(t1) / steps * 1e-3


def job_value(units_per_rank, world, seconds):
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    return world * units_per_rank / seconds


def run_own(args, rank, world, dist):
    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    spec = with_meta16(with_jensen(workload_spec(args.workload), args.jensen), args.meta16)
    inputs = make_inputs(spec)
    r = (DecodeRunner if spec["kind"] == "decode" else ChunkRunner)(spec, inputs, dev)
    if spec["kind"] == "chunkdecode":
        r.launches_per_step = 1     # the decode kernel only (no append in the step)
        r.append = lambda stream: None
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    flush = L2Flush(dev)

    sampler = ClockSampler(local)
    with sampler:
        for _ in range(args.warmup):
            r.attention(sh)
            r.append(sh)
        torch.cuda.synchronize(dev)
        # the step's calls as written (eager), or replayed from CUDA graphs captured once
        attn_fn, app_fn = (lambda: r.attention(sh)), (lambda: r.append(sh))
        if args.graph:
            attn_fn, app_fn = capture_step(r, spec, dev, stream)

        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)
        for k in range(args.steps):
            flush(k)                                   # evicts L2 (outside the timed events)
            ev[k][0].record(stream)
            attn_fn()
            ev[k][1].record(stream)
            app_fn()
            ev[k][2].record(stream)
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
    t_step = sum(e[0].elapsed_time(e[2]) for e in ev) / args.steps * 1e-3
    t_attn = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps * 1e-3
    t_app = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps * 1e-3

    # end to end through the C ABI with host buffers: H2D of the step's inputs (one pinned buffer
    # holding Q, K_cur and V_cur, one copy), D2H of the output
    hin = r.in_flat.cpu().pin_memory()
    hO = torch.empty_like(r.out, device="cpu").pin_memory()
    h2d = hin.numel() * hin.element_size()
    d2h = hO.numel() * hO.element_size()
    working = r.cache_bytes + h2d + d2h
    pipelined = working > L2_BYTES
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    if pipelined:
        t_e2e = e2e_pipelined(r, hin, hO, args.steps, stream, dev)
    else:
        e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)]
        for k in range(args.steps):
            flush(k)
            e_ev[k][0].record(stream)
            r.in_flat.copy_(hin, non_blocking=True)
            attn_fn()
            app_fn()
            hO.copy_(r.out, non_blocking=True)
            e_ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        t_e2e = sum(a.elapsed_time(b) for a, b in e_ev) / args.steps * 1e-3
    if dist:
        dist.barrier()

    if dist:
        t_step, t_attn, t_app, t_e2e = max_over_ranks([t_step, t_attn, t_app, t_e2e], dist, dev)

    if rank != 0:
        return
    rows = spec["B"] * spec["Hq"] * spec["n_q"]
    peaks = load_peaks()
    kernel = {1: "attn_simt_kernel", 2: "attn_tc_kernel", 3: "attn_decode_kernel"}.get(r.path)
    cache_gbs = r.cache_bytes / t_attn / 1e9
    if spec["kind"] in ("decode", "chunkdecode"):
        roof = {"bound": "hbm", "achieved": cache_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": cache_gbs / peaks["hbm_gbs"]}
    else:
        achieved = spec["attn_flops"] / t_attn / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"]}
        if peaks.get("bf16_tflops_sustained"):
            # the kernel is timed alone (burst peak above); the power-capped figure for context
            roof["frac_of_sustained"] = achieved / peaks["bf16_tflops_sustained"]
    tkey = spec["name"] + ("+meta16" if spec.get("meta16") else "")
    roof.update({"traffic": traffic_for(kernel, tkey), "kernel": kernel, "splits": r.splits,
                 "peak_source": peaks["source"],
                 "algorithmic": ("cache bytes (codes of valid tokens + all metadata) per launch"
                                 if spec["kind"] in ("decode", "chunkdecode")
                                 else "4 n_q (n_cache + n_cur) d FLOPs per head"),
                 "roofline_time_frac_of_step": max(r.cache_bytes / (peaks["hbm_gbs"] * 1e9),
                                                   spec["attn_flops"] / (peaks["bf16_tflops"] * 1e12)) / t_step})
    line = {
        "metric": METRIC, "value": job_value(rows, world, t_step), "unit": "query-tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": spec["dtype"], "data": "synthetic (seeded, PCG64)",
        "config": {"workload": spec["label"], "query_tokens": "B*Hq*n_q per step (one row per query head)",
                   "l2": "flushed between steps (512 MiB written, then another 512 MiB read)",
                   "execution": "CUDA graph replay (graphs captured once)" if args.graph else "eager calls",
                   "parallelism": f"replicas x{world}"},
        "cache_gbs": world * cache_gbs,
        "attn_ms": t_attn * 1e3, "append_ms": t_app * 1e3,
        "roofline": roof,
        "e2e": {"value": job_value(rows, world, t_e2e), "unit": "query-tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "schedule": ("pipelined: step k+1's H2D and step k's D2H on two copy streams while step k "
                             "computes (double-buffered device inputs and outputs), one event pair over all "
                             f"steps; L2 not flushed, the step's {working / 1e6:.0f} MB exceed the 126 MB L2"
                             if pipelined else
                             "serial: H2D, attention, append, D2H on one stream per step, L2 flushed between "
                             "steps")},
        "gpu_launches": r.launches_per_step * args.steps,
        "clocks": sampler.summary(),
    }
    if spec["kind"] == "chunk":
        line["append_gbs"] = spec["append_bytes"] / t_app / 1e9
    if spec["kind"] == "chunkdecode":
        line.pop("append_ms", None)
    if getattr(r, "calib_ms", None) is not None:
        line["calibration_ms"] = r.calib_ms   # once per prefill, outside the step
    if spec["kind"] == "decode":
        # the similarity that feeds the window plan, once per prefill and outside the step
        t_ws, b_ws = r.time_window_similarity(flush, args.steps, sh)
        line["window_similarity"] = {"us": t_ws * 1e6, "bytes": b_ws, "gbs": b_ws / t_ws / 1e9,
                                     "frac_hbm": b_ws / t_ws / 1e9 / peaks["hbm_gbs"]}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(spec, inputs)
    print(json.dumps(line), flush=True)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured (MEASURED_PEAKS.json)"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def traffic_for(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p) or kernel is None:
        return None
    d = json.load(open(p)).get(f"{kernel}:{workload}")
    if not d:
        return None
    import hashlib
    src = os.path.join(ROOT, "bit_kv_cache_28_b300", "csrc", d["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != d["sha"]:
        return None
    return d["bytes_per_launch"]


# ------------------------------------------------------- oracle arms -------

def oracle_sample_step(spec, inputs, heads):
    """One bounded sample of the step on the CPU oracle; returns the query rows it covered.

    chunk workloads: `heads` heads of cache build + attention + append.
    decode: `heads` kv heads of sequence 0 (cache build + attention of their query heads).
    """
    from oracle import layout as OL, attention as OA, window as OW
    m16 = bool(spec.get("meta16"))
    if spec["kind"] == "decode":
        sl = slice(0, heads)
        b = slice(0, 1)
        bits, _ = OW.window_plan(inputs["sim"][0], 0.2, 0.3)
        caps = [int((bits == k).sum()) for k in (16, 4, 2)]
        oc = OL.build_mixed(inputs["K_cache"][b, sl], inputs["V_cache"][b, sl], bits[None], caps, "f16", m16)
        g = spec["Hq"] // spec["Hkv"]
        OA.attention_over_cache(oc, inputs["Q"][b, :heads * g], inputs["K_cur"][b, sl], inputs["V_cur"][b, sl],
                                "f16")
        return heads * g
    sl = slice(0, heads)
    if spec["kind"] == "chunkdecode":
        oc = OL.build_uniform(inputs["K_cache"][:, sl], inputs["V_cache"][:, sl], 2, spec["chunks"],
                              sum((n + 31) // 32 for n in spec["chunks"]), m16)
        OA.attention_over_cache(oc, inputs["Q"][:, sl], inputs["K_cur"][:, sl], inputs["V_cur"][:, sl],
                                spec["dtype"], jensen=spec["jensen"])
        return spec["B"] * heads
    if spec["name"] == "codebook":
        from oracle import codebook as OC, psac as OP
        cent = np.stack([OC.fit_centroids(inputs["K_cache"][0, h]) for h in range(heads)])[None].astype(np.float32)
        U = np.stack([OP.psac_basis(inputs["Q_hist"][h], spec["r"])[0] for h in range(heads)])[None].astype(
            np.float32)
        nb = inputs["K_cache"].shape[2] // 32
        oc = OC.build_codebook(inputs["K_cache"][:, sl], inputs["V_cache"][:, sl], cent, U, nb)
        OA.attention_over_cache(oc, inputs["Q"][:, sl], inputs["K_cur"][:, sl], inputs["V_cur"][:, sl],
                                spec["dtype"], psac_U=U)
        OC.build_codebook(inputs["K_cur"][:, sl], inputs["V_cur"][:, sl], cent, U, (spec["n_cur"] + 31) // 32)
        return spec["B"] * heads * spec["n_q"]
    oc = OL.build_uniform(inputs["K_cache"][:, sl], inputs["V_cache"][:, sl], 2, spec["chunks"],
                          sum((n + 31) // 32 for n in spec["chunks"]), m16)
    OA.attention_over_cache(oc, inputs["Q"][:, sl], inputs["K_cur"][:, sl], inputs["V_cur"][:, sl],
                            spec["dtype"], jensen=spec["jensen"])
    OL.build_uniform(inputs["K_cur"][:, sl], inputs["V_cur"][:, sl], 2, [spec["n_cur"]],
                     (spec["n_cur"] + 31) // 32, m16)
    return spec["B"] * heads * spec["n_q"]


def oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:
        return os.cpu_count() or 1


def sample_text(spec, heads):
    if spec["kind"] == "decode":
        return (f"{heads} kv head of sequence 0 ({heads * spec['Hq'] // spec['Hkv']} query heads): mixed cache "
                f"build of {spec['n_cache']} tokens + decode attention, fp64 numpy")
    if spec["kind"] == "chunkdecode":
        return (f"{heads} head of {spec['Hq']}: cache build of {sum(spec['chunks'])} tokens + decode attention, "
                f"fp64 numpy")
    if spec["name"] == "codebook":
        return (f"{heads} head of {spec['Hq']}: k-means + PSAC basis + cache build + attention of "
                f"{spec['n_q']} queries + append, fp64 numpy")
    return (f"{heads} head of {spec['Hq']}: cache build + attention of {spec['n_q']} queries + append, "
            f"fp64 numpy")


def cpu_baseline(spec, inputs):
    heads = 1
    t = time.perf_counter()
    rows = 0
    n = 0
    while True:
        rows += oracle_sample_step(spec, inputs, heads)
        n += 1
        if time.perf_counter() - t > 10.0 or n >= 3:
            break
    dt = time.perf_counter() - t
    return {"value": rows / dt, "unit": "query-tokens/s", "cores": oracle_threads(), "kind": "oracle",
            "sample": f"{n} x ({sample_text(spec, heads)})"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    spec = with_meta16(with_jensen(workload_spec(args.workload), args.jensen), args.meta16)
    inputs = make_inputs(spec)
    heads = 1
    for _ in range(args.warmup):
        oracle_sample_step(spec, inputs, heads)
    t = time.perf_counter()
    rows = 0
    for _ in range(args.steps):
        rows += oracle_sample_step(spec, inputs, heads)
    dt = time.perf_counter() - t
    value = rows / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "query-tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, PCG64)",
            "config": {"workload": spec["label"], "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": "query-tokens/s", "cores": oracle_threads(), "kind": "oracle",
                             "sample": f"per step: {sample_text(spec, heads)}"},
            "e2e": {"value": value, "unit": "query-tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="own", choices=["own", "reference"])
    ap.add_argument("--workload", default="rollout")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--jensen", type=int, default=None, choices=[0, 1, 2, 3],
                    help="override the workload's Jensen mode (0 off, 1 TAYLOR2, 2 EXACT, 3 ISOTROPIC)")
    ap.add_argument("--meta16", action="store_true",
                    help="fp16 step / zero-point metadata in the INT blocks (not for codebook)")
    ap.add_argument("--graph", action="store_true",
                    help="replay each step's calls from CUDA graphs captured once (default: eager calls)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3) if args.impl == "own" else args.warmup
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    try:
        run_own(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
