"""Benchmark of the quantised-KV attention hot path (one JSON line on rank 0).

A step is one pass of the hot path over one chunk of the workload: attention
of the current chunk's queries over the packed cache plus the chunk itself
(Jensen correction on), then quantise-and-append of the finished chunk.  The
cache is rewound on the host after each step so every step sees the same
cache.  Inputs are seeded synthetic tensors (no dataset exists for this
workload; shapes follow the chunk-wise video-diffusion setting).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload chunk|rollout|decode|tiny|codebook]
    python bench.py --impl reference ...   # the CPU oracle timed on the host cores

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
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized-KV attention cache GB/s and query-tokens/s, % of HBM/TC roofline"
L2_FLUSH_BYTES = 512 << 20


# ------------------------------------------------------------ workloads ----

def workload_spec(name):
    """Shapes, algorithmic bytes/FLOPs of one step."""
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
        return dict(name=name, B=1, Hkv=H, Hq=H, d=d, n_q=n, n_cur=n, chunks=[n] * n_chunks, dtype="bf16",
                    cache_bytes=cache_bytes, attn_flops=flops, append_bytes=append_read + append_write,
                    jensen=1, seed=2 if name == "chunk" else 3)
    if name == "tiny":
        d, n_cache, n = 64, 1024, 64
        cache_bytes = n_cache * d * 2 * 2 / 8 + (n_cache // 32) * d * 8 + n_cache * (d // 32) * 8
        return dict(name=name, B=1, Hkv=1, Hq=1, d=d, n_q=n, n_cur=n, chunks=[1024], dtype="f32",
                    cache_bytes=cache_bytes, attn_flops=4.0 * n * (n_cache + n) * d,
                    append_bytes=2 * n * d * 4 + 2 * 2048, jensen=1, seed=1)
    raise ValueError(f"unknown workload {name}")


def make_inputs(spec):
    from bit_kv_cache_28_b300 import synth
    if spec["name"] == "tiny":
        return synth.tiny(spec["seed"])
    return synth.chunk_case(spec["seed"], Hkv=spec["Hkv"], chunks=spec["chunks"], n_cur=spec["n_cur"])


# --------------------------------------------------------------- clocks ----

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"bitkv_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                rows.append((float(p[1]), float(p[2]), p[5], p[6], p[7], p[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [r[0] for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[2 + i].lower().startswith("active")})
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------- own arm -------

class Runner:
    """Device state of one replica: the cache after the workload's cached chunks, the step inputs."""

    def __init__(self, spec, inputs, dev):
        import torch
        from bit_kv_cache_28_b300 import bitkv as B
        self.B, self.spec, self.dev = B, spec, dev
        tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[spec["dtype"]]
        self.dt = {"bf16": B.KV_BF16, "f16": B.KV_F16, "f32": B.KV_F32}[spec["dtype"]]
        self.tdt = tdt
        to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev).to(tdt)
        nb_cache = sum((n + 31) // 32 for n in spec["chunks"])
        nb_cur = (spec["n_cur"] + 31) // 32
        self.tc = B.TorchCache(spec["B"], spec["Hkv"], spec["d"], B.KV_UNIFORM2, (0, 0, nb_cache + nb_cur),
                               device=dev)
        t0 = 0
        for n in spec["chunks"]:
            B.kv_quantize_append(to(inputs["K_cache"][:, :, t0:t0 + n]), to(inputs["V_cache"][:, :, t0:t0 + n]),
                                 self.dt, n, self.tc.c)
            t0 += n
        self.saved = (list(self.tc.c.n_blocks), self.tc.c.n_tokens)
        self.Q, self.Kc, self.Vc = to(inputs["Q"]), to(inputs["K_cur"]), to(inputs["V_cur"])
        self.opts = B.kv_attn_opts(0.0, spec["jensen"], 0, 0, 0, B.KV_PATH_AUTO)
        self.out = torch.empty_like(self.Q)
        self.lse = torch.empty(self.Q.shape[:3], dtype=torch.float32, device=dev)
        self.ws_bytes = B.kv_attention_workspace(self.tc.c, self.dt, spec["n_q"], spec["n_cur"], spec["Hq"],
                                                 self.opts)
        self.ws = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=dev)
        self.path, self.splits = B.kv_attention_plan(self.tc.c, self.dt, spec["n_q"], spec["n_cur"], spec["Hq"],
                                                     self.opts)
        # attention kernel (+ one merge launch when the key range is split) + one append launch
        self.launches_per_step = 2 + (1 if self.splits > 1 else 0)

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


def run_own(args, rank, world, dist):
    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    spec = workload_spec(args.workload)
    inputs = make_inputs(spec)
    r = Runner(spec, inputs, dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    for _ in range(args.warmup):
        r.attention(sh)
        r.append(sh)
    torch.cuda.synchronize(dev)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    with sampler:
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)
        for k in range(args.steps):
            flush.fill_(k & 0xFF)                      # evicts L2 (outside the timed events)
            ev[k][0].record(stream)
            r.attention(sh)
            ev[k][1].record(stream)
            r.append(sh)
            ev[k][2].record(stream)
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
    t_step = sum(e[0].elapsed_time(e[2]) for e in ev) / args.steps * 1e-3
    t_attn = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps * 1e-3
    t_app = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps * 1e-3

    # end to end through the C ABI with host buffers: H2D of the step's inputs, D2H of the output
    pin = lambda t: t.cpu().pin_memory()
    hQ, hK, hV = pin(r.Q), pin(r.Kc), pin(r.Vc)
    hO = torch.empty_like(r.out, device="cpu").pin_memory()
    h2d = (hQ.numel() + hK.numel() + hV.numel()) * hQ.element_size()
    d2h = hO.numel() * hO.element_size()
    e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        e_ev[k][0].record(stream)
        r.Q.copy_(hQ, non_blocking=True)
        r.Kc.copy_(hK, non_blocking=True)
        r.Vc.copy_(hV, non_blocking=True)
        r.attention(sh)
        r.append(sh)
        hO.copy_(r.out, non_blocking=True)
        e_ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    t_e2e = sum(a.elapsed_time(b) for a, b in e_ev) / args.steps * 1e-3

    if dist:
        tt = torch.tensor([t_step, t_attn, t_app, t_e2e], dtype=torch.float64, device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        t_step, t_attn, t_app, t_e2e = tt.tolist()

    if rank != 0:
        return
    rows = spec["B"] * spec["Hq"] * spec["n_q"]
    value = world * rows / t_step
    peaks = load_peaks()
    flops = spec["attn_flops"]
    tc_peak, peak_src = peaks["bf16_tflops"], peaks["source"]
    achieved = flops / t_attn / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "query-tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": spec["dtype"], "data": "synthetic (seeded, PCG64)",
        "config": {"workload": f"{spec['name']}: B{spec['B']} H{spec['Hq']} d{spec['d']} chunk {spec['n_cur']} "
                               f"cache {sum(spec['chunks'])} INT2, Jensen taylor2",
                   "query_tokens": "B*Hq*n_q per step (one row per head)", "l2": "flushed between steps (512 MiB write)",
                   "parallelism": f"replicas x{world}"},
        "cache_gbs": world * spec["cache_bytes"] / t_attn / 1e9,
        "attn_ms": t_attn * 1e3, "append_ms": t_app * 1e3,
        "append_gbs": spec["append_bytes"] / t_app / 1e9,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                     "frac": achieved / tc_peak, "traffic": traffic_for("attn", spec["name"]),
                     "kernel": {1: "attn_simt_kernel", 2: "attn_tc_kernel", 3: "attn_decode_kernel"}.get(r.path),
                     "splits": r.splits, "peak_source": peak_src,
                     "roofline_frac_of_step": (max(spec["cache_bytes"] / (peaks["hbm_gbs"] * 1e9),
                                                   flops / (tc_peak * 1e12)) / t_step)},
        "e2e": {"value": world * rows / t_e2e, "unit": "query-tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": r.launches_per_step * args.steps,
        "clocks": sampler.summary(),
    }
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
    """DRAM bytes per launch from a committed ncu summary, if one matches the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
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
    """One bounded sample of the step on the CPU oracle: `heads` heads of append + attention."""
    from oracle import layout as OL, attention as OA
    sl = slice(0, heads)
    oc = OL.build_uniform(inputs["K_cache"][:, sl], inputs["V_cache"][:, sl], 2, spec["chunks"],
                          sum((n + 31) // 32 for n in spec["chunks"]))
    OA.attention_over_cache(oc, inputs["Q"][:, sl], inputs["K_cur"][:, sl], inputs["V_cur"][:, sl],
                            spec["dtype"], jensen=spec["jensen"])
    OL.build_uniform(inputs["K_cur"][:, sl], inputs["V_cur"][:, sl], 2, [spec["n_cur"]],
                     (spec["n_cur"] + 31) // 32)
    return spec["B"] * heads * spec["n_q"]


def oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(spec, inputs):
    heads = 1 if spec["Hq"] <= 24 else 1
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
            "sample": f"{n} x ({heads} head of {spec['Hq']}: cache build + attention of {spec['n_q']} queries + "
                      f"append), fp64 numpy"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    spec = workload_spec(args.workload)
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
    sample = f"per step: {heads} head of {spec['Hq']} (cache build + attention of {spec['n_q']} queries + append)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "query-tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, PCG64)",
            "config": {"workload": f"{spec['name']}: B{spec['B']} H{spec['Hq']} d{spec['d']} chunk {spec['n_cur']} "
                                   f"cache {sum(spec['chunks'])} INT2, Jensen taylor2", "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": "query-tokens/s", "cores": oracle_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "query-tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="own", choices=["own", "reference"])
    ap.add_argument("--workload", default="chunk")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
