"""Benchmark of the quantized MLA decode step on GB300.

Workload (the 4-bit rotated-int4 tier): a decode step of a 32-layer MLA stack, each
layer with its own cache of T = 32768 rows (512-wide latent as TQ4 codes + radius,
64-wide rope key as fp8 + scale, 328 B/row; 343 MB in all, larger than L2), H = 64
heads, one query.  Per layer and step: quantize-on-append of the new token's row
(kvq_encode_mla: its TQ4 latent and fp8 rope key into row T-1, one launch), then
kvq_mla_decode over the T rows (query image, split-T partials, log-sum-exp combine +
unrotation).

metric  KV rows/s = layers x T / step time (higher is better); effective GB/s in the
        roofline object.
e2e     the same step through host buffers: new rows and queries copied host->device
        from pinned memory, outputs copied back, every step.
--impl reference  times the CPU oracle (test infrastructure) on a bounded sample.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized-KV MLA decode attention: KV rows/s (TQ4 tier)"
UNIT = "rows/s"
ROW_BYTES_TQ4 = 256 + 4 + 64 + 4


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=32)
    ap.add_argument("--T", type=int, default=32768)
    ap.add_argument("--H", type=int, default=64)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--preload-s", type=float, default=1.5,
                    help="decode suite: seconds of untimed load before the timed steps, so that "
                         "the clock sampler sees loaded clocks (0 for profiling runs)")
    ap.add_argument("--no-configs", action="store_true",
                    help="decode suite: skip the per-configuration records (hbm_points, configs)")
    ap.add_argument("--suite", default="decode", choices=["decode", "codecs", "decode-configs"],
                    help="decode: the decode step (one JSON line); codecs: one line per codec "
                         "kernel; decode-configs: one line per decode configuration")
    ap.add_argument("--only", default="",
                    help="decode-configs: run only the configurations whose name contains this text")
    ap.add_argument("--decode-impl", type=int, default=0,
                    help="decode kernel: 0 library's choice, 1 CUDA cores, 2 tcgen05 (32 heads), "
                         "3 warp-level MMA, 4 tcgen05 (16 heads), 5 tcgen05 on e4m3 codes (fp8 tier)")
    return ap.parse_args()


# ------------------------------------------------------------------------- helpers -----

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms around the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def peaks():
    """(hbm GB/s, sustained bf16 TFLOP/s, kind): the measured figures when present."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops_sustained"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1700.0, "fallback"


def profile_traffic(kernel_file: str, summary: str = "mla_decode_tq4_T32768_H64.txt"):
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken on
    the kernel source as it is now (its sha256 matches); else None."""
    path = os.path.join(ROOT, "profiles", summary)
    src = os.path.join(ROOT, "quantized_kv_cache_fp8_gb300", "csrc", kernel_file)
    try:
        text = open(path).read()
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    fields = dict(l.split("=", 1) for l in text.splitlines() if "=" in l and not l.startswith("#"))
    if fields.get("source_sha256", "").strip() != digest:
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return world, rank, local


# --------------------------------------------------------------------------- oracle ----

def cpu_model() -> str:
    """The host CPU's model name (lscpu), or the machine type when lscpu has none."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for l in out.splitlines():
            if l.split(":")[0].strip() == "Model name":
                return l.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine()


def _oracle_worker(job):
    """One process of the oracle baseline: the fp64 decode of heads [h0, h1) of the
    sample (plus, in the first process, the encode of the step's new row), repeated
    until `seconds` have passed.  Returns (iterations, heads, elapsed seconds)."""
    T_sample, H, h0, h1, seconds = job
    import oracle
    import workloads as W
    oracle.build()
    rows = W.unit_rows(T_sample, seed=0)
    signs = W.sign_bits(0)
    lat, rad = oracle.encode_tq4(rows.c, signs)
    rope, rs = oracle.encode_fp8(rows.k_rope)
    cache = dict(lat=lat, lat_scale=rad, rope=rope, rope_scale=rs)
    q = W.queries(1, 1, H, seed=0)
    new = W.unit_rows(1, seed=1)
    n, t0 = 0, time.perf_counter()
    while True:
        if h0 == 0:
            oracle.encode_tq4(new.c, signs)
            oracle.encode_fp8(new.k_rope)
        oracle.mla_decode(seq_len=[T_sample], seq_fmt=[2], q_lat=q.q_lat, q_rope=q.q_rope,
                          sm_scale=W.SM_SCALE, tq4=cache, signs=signs, heads=(h0, h1))
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return n, h1 - h0, el


def oracle_sample(T_sample: int, H: int, seconds_target: float = 12.0):
    """The oracle, as it stands, on a bounded sample of the workload (the new-row encode
    plus an fp64 decode over T_sample rows for all H heads), timed on one host core and
    on every host core (one process per core, each decoding a share of the heads, started
    with `spawn`).  Returns the all-core figure and the single-core one, each as rows/s of
    the full step's unit."""
    import multiprocessing as mp
    import oracle
    oracle.build()
    n1, _, el1 = _oracle_worker((T_sample, H, 0, H, seconds_target / 2))
    single = n1 * T_sample / el1
    cores = max(1, min(os.cpu_count() or 1, H))
    bounds = [(H * k // cores, H * (k + 1) // cores) for k in range(cores)]
    with mp.get_context("spawn").Pool(cores) as pool:
        res = pool.map(_oracle_worker, [(T_sample, H, a, b, seconds_target / 2) for a, b in bounds])
    # full-step iterations per second: each process covers its share of the heads
    allcore = sum(n * h / el for n, h, el in res) / H * T_sample
    model = cpu_model()
    desc = (f"oracle (plain C, fp64) on {model}: encode 1 new row + decode over T={T_sample} "
            f"rows, H={H}; {cores} processes of {H // cores}-{-(-H // cores)} heads each, "
            f"{seconds_target / 2:.0f} s; one core alone: {single:.4g} rows/s")
    return {"value": allcore, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc,
            "cpu_model": model, "single_core": {"value": single, "unit": UNIT, "cores": 1}}


def run_reference(args, world, rank):
    if rank != 0:
        return
    base = oracle_sample(4096, args.H, seconds_target=max(8.0, min(40.0, 2.0 * args.steps)))
    rate = base["value"]
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"tq4 MLA decode step, T={args.T}, H={args.H}, nq=1 (oracle "
                               f"sampled at T=4096)"},
        "cpu_baseline": base,
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- ours ----

def run_ours(args, world, rank, local):
    import torch
    import __graft_entry__
    import quantized_kv_cache_fp8_gb300 as kvq
    from quantized_kv_cache_fp8_gb300.sharding import max_over_ranks
    import workloads as W

    __graft_entry__.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    Lyr, T, H = args.layers, args.T, args.H
    stream = torch.cuda.current_stream()

    # ---- a cache of T rows encoded on the GPU, replicated into Lyr distinct layers
    rows = W.unit_rows(T, seed=0)
    signs = torch.from_numpy(W.sign_bits(0)).to(dev)
    c = torch.from_numpy(rows.c).to(dev)
    kr = torch.from_numpy(rows.k_rope).to(dev)
    lat = torch.empty(Lyr, T, 256, dtype=torch.uint8, device=dev)
    rad = torch.empty(Lyr, T, dtype=torch.float32, device=dev)
    rope = torch.empty(Lyr, T, 64, dtype=torch.uint8, device=dev)
    rsc = torch.empty(Lyr, T, dtype=torch.float32, device=dev)
    kvq.kvq_encode_tq4(c, signs, lat[0], rad[0])
    kvq.kvq_encode_fp8(kr, rope[0], rsc[0])
    for l in range(1, Lyr):
        lat[l].copy_(lat[0]); rad[l].copy_(rad[0]); rope[l].copy_(rope[0]); rsc[l].copy_(rsc[0])
    del c, kr
    q = W.queries(Lyr, 1, H, seed=0)
    q_lat = torch.from_numpy(q.q_lat).to(dev)          # [L][1][H][512]
    q_rope = torch.from_numpy(q.q_rope).to(dev)
    new = W.unit_rows(Lyr, seed=1)
    new_c = torch.from_numpy(new.c).to(dev)            # [L][512]
    new_r = torch.from_numpy(new.k_rope).to(dev)       # [L][64]
    out = torch.empty(Lyr, 1, 1, H, 512, dtype=torch.float32, device=dev)
    lse = torch.empty(Lyr, 1, 1, H, dtype=torch.float32, device=dev)
    seq_len = torch.tensor([T], dtype=torch.int32, device=dev)
    probs = []
    for l in range(Lyr):
        planes = dict(lat=lat[l], lat_scale=rad[l], rope=rope[l], rope_scale=rsc[l])
        probs.append(kvq.make_problem(seq_len=seq_len, q_lat=q_lat[l:l + 1], q_rope=q_rope[l:l + 1],
                                      sm_scale=W.SM_SCALE, max_seq_len=T, fmt=kvq.FMT_TQ4,
                                      tq4=planes, signs=signs,
                                      impl=0 if args.decode_impl == 5 else args.decode_impl))
    ws = torch.empty(kvq.kvq_mla_decode_workspace(probs[0]), dtype=torch.uint8, device=dev)

    def encode_step():
        for l in range(Lyr):
            kvq.kvq_encode_mla(new_c[l:l + 1], new_r[l:l + 1], kvq.FMT_TQ4, signs, lat[l, T - 1:T],
                               rad[l, T - 1:T], rope[l, T - 1:T], rsc[l, T - 1:T])

    def decode_step():
        for l in range(Lyr):
            kvq.kvq_mla_decode(probs[l], out[l, 0], lse[l, 0], ws)

    # ---- capture the two halves of the step as CUDA graphs
    encode_step(); decode_step(); torch.cuda.synchronize()
    g_enc, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_enc):
        encode_step()
    with torch.cuda.graph(g_dec):
        decode_step()
    launches_per_step = Lyr * 1 + Lyr * 3          # append + (query image, decode, combine)

    for _ in range(max(3, args.warmup)):
        g_enc.replay(); g_dec.replay()
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    with ClockSampler(local) as clk:
        # keep the GPU under the same load while the sampler starts, so that its
        # samples fall on loaded clocks; then time exactly K steps
        t_end = time.perf_counter() + args.preload_s
        while time.perf_counter() < t_end:
            g_enc.replay(); g_dec.replay()
            torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        for k in range(K):
            ev[k][0].record()
            g_enc.replay()
            ev[k][1].record()
            g_dec.replay()
            ev[k][2].record()
        torch.cuda.synchronize()
    step_ms = [ev[k][0].elapsed_time(ev[k][2]) for k in range(K)]
    dec_ms = [ev[k][1].elapsed_time(ev[k][2]) for k in range(K)]
    total_ms = ev[0][0].elapsed_time(ev[K - 1][2])
    total_ms = max_over_ranks(total_ms, device=dev)
    ms_per_step = total_ms / K
    rows_per_step = Lyr * T
    value = rows_per_step * world / (ms_per_step / 1e3)

    # ---- roofline of the dominant kernel (the decode call, per launch = one layer).
    # At H = 64 the decode is a dense contraction of 2 H (512 + 64 + 512) flops per row,
    # which the tensor cores run as split fp16 (hi + lo halves of q and w: twice the
    # algorithmic flops); that roofline binds before HBM (328 B per row).
    dec_launch_s = statistics.mean(dec_ms) / Lyr / 1e3
    alg_bytes = T * ROW_BYTES_TQ4 + H * (512 + 64) * 4 + H * 512 * 4 + H * 4
    alg_flops = 2 * H * (512 + 64 + 512) * T
    hbm_peak, tc_peak, peak_kind = peaks()
    achieved_tf = alg_flops / dec_launch_s / 1e12
    achieved_gbs = alg_bytes / dec_launch_s / 1e9
    kname, ksrc, ksum = {2: ("tcgen05", "kvq_decode_tc.cu", "mla_decode_tq4_T32768_H64.txt"),
                         4: ("tcgen05x16", "kvq_decode_tc16.cu", "mla_decode_tc16_tq4_T32768_H64.txt"),
                         3: ("warp-mma", "kvq_decode_mma.cu", "none"),
                         1: ("cuda-cores", "kvq_decode.cu", "none")}[kvq.kvq_mla_decode_kernel(probs[0])]
    roofline = {"bound": "tensor", "achieved": round(achieved_tf, 2), "peak": tc_peak, "unit": "TFLOP/s",
                "frac": round(achieved_tf / tc_peak, 4), "traffic": profile_traffic(ksrc, ksum),
                "peak_kind": f"{peak_kind} bf16 sustained (fp16 runs at the same rate)",
                "kernel": f"kvq_mla_decode (TQ4, T={T}, H={H}) on the {kname} kernel: query image, "
                          f"decode, combine",
                "decode_us_per_layer": round(dec_launch_s * 1e6, 2),
                "flops_per_launch": alg_flops, "tensor_flops_executed_per_launch": 2 * alg_flops,
                "tensor_pipe_frac": round(2 * achieved_tf / tc_peak, 4),
                "bytes_per_launch": alg_bytes, "hbm_achieved_gbs": round(achieved_gbs, 1),
                "hbm_peak_gbs": hbm_peak, "hbm_frac": round(achieved_gbs / hbm_peak, 4)}

    # ---- e2e: host buffers in and out every step
    e2e = None
    if not args.no_e2e:
        h_new_c = new_c.cpu().pin_memory()
        h_new_r = new_r.cpu().pin_memory()
        h_ql = q_lat.cpu().pin_memory()
        h_qr = q_rope.cpu().pin_memory()
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (h_new_c, h_new_r, h_ql, h_qr))
        d2h = h_out.numel() * 4 + h_lse.numel() * 4

        def e2e_step():
            new_c.copy_(h_new_c, non_blocking=True)
            new_r.copy_(h_new_r, non_blocking=True)
            q_lat.copy_(h_ql, non_blocking=True)
            q_rope.copy_(h_qr, non_blocking=True)
            g_enc.replay()
            g_dec.replay()
            h_out.copy_(out, non_blocking=True)
            h_lse.copy_(lse, non_blocking=True)
            stream.synchronize()

        for _ in range(3):
            e2e_step()
        t0 = time.perf_counter()
        for _ in range(K):
            e2e_step()
        e2e_s = (time.perf_counter() - t0) / K
        assert np.isfinite(h_out.numpy()).all()
        e2e = {"value": rows_per_step * world / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_s * 1e3, 3)}

    # every other decode configuration (the HBM-bound 16-head points among them), each a
    # CUDA graph over a stack of distinct caches, against both rooflines
    records = decode_records(args, dev) if not args.no_configs else []
    hbm_points = [r for r in records if r["config"].startswith("HBM point")]
    configs = [r for r in records if not r["config"].startswith("HBM point")]

    if rank != 0:
        return
    cpu = oracle_sample(4096, H, seconds_target=12.0)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"tq4 MLA decode step: {Lyr} layers x T={T} rows (TQ4 latent + "
                               f"fp8 rope, 328 B/row), H={H}, nq=1, append 1 row/layer + decode",
                   "layers": Lyr, "T": T, "H": H, "n_q": 1, "split": "library default",
                   "decode_impl": args.decode_impl,
                   "l2": f"inputs larger than L2 ({Lyr * T * ROW_BYTES_TQ4 / 1e6:.0f} MB of caches)",
                   "graph": "CUDA graphs (encode half, decode half)"},
        "effective_gbs": round(Lyr * T * ROW_BYTES_TQ4 / (ms_per_step / 1e3) / 1e9, 1),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "clocks": clk.summary(),
        "hbm_points": hbm_points,
        "configs": configs,
    }
    print(json.dumps(line), flush=True)


def run_codecs(args, local):
    """One JSON line per codec / gather kernel on its workload's sizes: median of K
    launches, each timed with CUDA events after writing a buffer larger than L2 (so the
    inputs come from HBM), against the algorithmic bytes the kernel must move."""
    import torch
    import __graft_entry__
    import quantized_kv_cache_fp8_gb300 as kvq
    import workloads as W

    __graft_entry__.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hbm_peak, _, peak_kind = peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    K = max(5, args.steps)

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        ts = []
        for _ in range(K):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / 1e3)
        return statistics.median(ts)

    def report(kernel, workload, alg_bytes, seconds, units, unit_name, extra=None):
        gbs = alg_bytes / seconds / 1e9
        line = {"suite": "codecs", "kernel": kernel, "workload": workload,
                "us": round(seconds * 1e6, 2), f"{unit_name}_per_s": units / seconds,
                "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak,
                             "unit": "GB/s", "frac": round(gbs / hbm_peak, 4),
                             "bytes_per_launch": alg_bytes, "peak_kind": peak_kind},
                "l2": "flushed before each timed launch", "steps": K}
        line.update(extra or {})
        print(json.dumps(line), flush=True)

    # a1: fp8 encode of the latent and rope planes, T = 131072 rows (the long-context cache)
    T = 131072
    x = torch.randn(T, 512, generator=gen, device=dev)
    xr = torch.randn(T, 64, generator=gen, device=dev)
    codes = torch.empty(T, 512, dtype=torch.uint8, device=dev)
    rcodes = torch.empty(T, 64, dtype=torch.uint8, device=dev)
    sc = torch.empty(T, device=dev)
    rsc = torch.empty(T, device=dev)
    s = timed(lambda: (kvq.kvq_encode_fp8(x, codes, sc), kvq.kvq_encode_fp8(xr, rcodes, rsc)))
    report("kvq_encode_fp8", f"T={T} rows of 512 + 64 (two launches)", T * (576 * 4 + 576 + 8), s, T, "rows")
    # the same rows as an MLA append: latent and rope key in one launch (kvq_encode_mla)
    s = timed(lambda: kvq.kvq_encode_mla(x, xr, kvq.FMT_FP8, None, codes, sc, rcodes, rsc))
    report("kvq_encode_mla (fp8 + fp8 rope)", f"T={T} rows of 512 + 64 (one launch)",
           T * (576 * 4 + 576 + 8), s, T, "rows")
    del x, xr, codes, rcodes, sc, rsc

    # a2: TQ4 encode of the latent, T = 32768 rows (the 4-bit tier's cache)
    T = 32768
    x = torch.randn(T, 512, generator=gen, device=dev)
    signs = torch.from_numpy(W.sign_bits(0)).to(dev)
    packed = torch.empty(T, 256, dtype=torch.uint8, device=dev)
    rad = torch.empty(T, device=dev)
    s = timed(lambda: kvq.kvq_encode_tq4(x, signs, packed, rad))
    report("kvq_encode_tq4", f"T={T} rows of 512", T * (512 * 4 + 256 + 4) + 64, s, T, "rows")
    # the rotated tier at 6 and 3 bits on the same rows
    for bits in (6, 3):
        pk = torch.empty(T, 512 * bits // 8, dtype=torch.uint8, device=dev)
        s = timed(lambda: kvq.kvq_encode_tq(x, signs, bits, pk, rad))
        report(f"kvq_encode_tq ({bits} bits)", f"T={T} rows of 512",
               T * (512 * 4 + 512 * bits // 8 + 4) + 64, s, T, "rows")
        del pk
    # append-time form: a row's TQ4 latent and fp8 rope key in one launch, in bulk and
    # for a single row (the per-token append of one layer)
    xr = torch.randn(T, 64, generator=gen, device=dev)
    rc = torch.empty(T, 64, dtype=torch.uint8, device=dev)
    rs = torch.empty(T, device=dev)
    s = timed(lambda: kvq.kvq_encode_mla(x, xr, kvq.FMT_TQ4, signs, packed, rad, rc, rs))
    report("kvq_encode_mla (TQ4 + fp8 rope)", f"T={T} rows of 512 + 64 (one launch)",
           T * (576 * 4 + 256 + 4 + 64 + 4) + 64, s, T, "rows")
    s = timed(lambda: kvq.kvq_encode_mla(x[:1], xr[:1], kvq.FMT_TQ4, signs, packed[:1], rad[:1], rc[:1], rs[:1]))
    report("kvq_encode_mla (TQ4 + fp8 rope)", "1 row (a per-token append)", 576 * 4 + 256 + 4 + 64 + 4, s, 1, "rows")
    del x, xr, packed, rad, rc, rs

    # a3 / a4: q4_0 paged append and gather, 16 sequences x 8192 tokens x 8 heads x 256
    n_seq, n_tok, n_heads, ps = 16, 8192, 8, 64
    pos0, table, n_cells = W.paged_table(n_seq, n_tok, ps, ps - 8, seed=0)
    amp = torch.tensor([1e-3, 1.0, 40.0], device=dev)

    def rows_kv(n=n_seq):
        r = torch.randn(n, n_tok, n_heads, 256, generator=gen, device=dev)
        return r * amp[torch.randint(0, 3, (n, n_tok, n_heads, 1), generator=gen, device=dev)]

    k, v = rows_kv(), rows_kv()
    pos0_d = torch.from_numpy(pos0).to(dev)
    table_d = torch.from_numpy(table).to(dev)
    k_pool = torch.zeros(n_cells, n_heads, 144, dtype=torch.uint8, device=dev)
    v_pool = torch.zeros(n_cells, n_heads, 144, dtype=torch.uint8, device=dev)
    toks = n_seq * n_tok
    s = timed(lambda: kvq.kvq_append_q4(k, v, pos0_d, table_d, ps, n_cells, k_pool, v_pool))
    report("kvq_append_q4", f"{n_seq} seqs x {n_tok} tokens x K,V x {n_heads} heads x 256, pages of {ps}",
           toks * (2 * n_heads * 256 * 4 + 2 * n_heads * 144) + table.size * 4, s, toks, "tokens")
    del k, v
    out = torch.empty(n_seq, n_tok, n_heads, 256, dtype=torch.float16, device=dev)
    s = timed(lambda: kvq.kvq_gather_q4(k_pool, pos0_d, n_tok, table_d, ps, n_cells, out))
    report("kvq_gather (q4_0)", f"one pool: {n_seq} seqs x {n_tok} tokens x {n_heads} heads -> fp16",
           toks * n_heads * (144 + 256 * 2) + table.size * 4, s, toks, "tokens")
    del out

    # the producer with its K/V projection fused (one new token per sequence, as in a
    # decode step): hidden rows of 4096, bfloat16 weights [4096][8 heads x 256] for K and V
    d_model = 4096
    hp = torch.randn(n_seq, 1, d_model, generator=gen, device=dev)
    wk = (torch.randn(d_model, n_heads * 256, generator=gen, device=dev) / 64).to(torch.bfloat16)
    wv = (torch.randn(d_model, n_heads * 256, generator=gen, device=dev) / 64).to(torch.bfloat16)
    pos0p = torch.full((n_seq,), n_tok - 1, dtype=torch.int32, device=dev)
    for n_new in (n_seq, 1):                         # a 16-sequence step, then one token
        s = timed(lambda: kvq.kvq_project_append_q4(hp[:n_new], wk, wv, pos0p[:n_new], table_d, ps,
                                                    n_cells, k_pool, v_pool))
        # the fixed-order fp32 sum runs on the CUDA cores: n_new * d_model * 2 * n_heads * 256
        # fmas against 152 SMs x 128 fp32 lanes x 2.07 GHz (the fp32 fma peak)
        fmas = n_new * d_model * 2 * n_heads * 256
        alu_peak = 152 * 128 * 2.07e9
        report("kvq_project_append_q4", f"{n_new} seqs x 1 token, d_model {d_model}, K,V x {n_heads} "
               f"heads x 256, bf16 weights",
               2 * d_model * n_heads * 256 * 2 + n_new * d_model * 4 + 2 * n_new * n_heads * 144, s,
               n_new, "tokens",
               {"alu": {"fmas_per_launch": fmas, "achieved_tfma_s": round(fmas / s / 1e12, 2),
                        "peak_tfma_s": round(alu_peak / 1e12, 2), "frac": round(fmas / s / alu_peak, 4),
                        "peak_kind": "derived: 152 SMs x 128 fp32 lanes x 2.07 GHz"}})
    del hp, wk, wv

    # q4_0 decode attention over the same pools' layout: 16 sequences x 8192 positions
    # (appended from position 0), 8 KV heads, 16 query heads (two per KV head), gated
    pos0z, table_z, _ = W.paged_table(n_seq, n_tok, ps, 0, seed=1)
    pos0z_d, table_zd = torch.from_numpy(pos0z).to(dev), torch.from_numpy(table_z).to(dev)
    for s0 in range(0, n_seq, 4):                   # 4 sequences of K, V rows at a time
        kk, vv = rows_kv(4), rows_kv(4)
        kvq.kvq_append_q4(kk, vv, pos0z_d[s0:s0 + 4], table_zd[s0:s0 + 4], ps, n_cells, k_pool, v_pool)
        del kk, vv
    n_qh = 16
    qd = torch.randn(n_seq, n_qh, 256, generator=gen, device=dev)
    gate = torch.randn(n_seq, n_qh, 256, generator=gen, device=dev)
    seq_len = torch.full((n_seq,), n_tok, dtype=torch.int32, device=dev)
    prob = kvq.make_q4_problem(seq_len=seq_len, page_table=table_zd, page_size=ps, k_pool=k_pool,
                               v_pool=v_pool, q=qd, gate=gate, sm_scale=1.0 / 16, max_seq_len=n_tok)
    ws = torch.empty(kvq.kvq_q4_decode_workspace(prob), dtype=torch.uint8, device=dev)
    out = torch.empty(n_seq, n_qh, 256, device=dev)
    lse = torch.empty(n_seq, n_qh, device=dev)
    s = timed(lambda: kvq.kvq_q4_decode(prob, out, lse, ws))
    assert torch.isfinite(out).all()
    report("kvq_q4_decode", f"{n_seq} seqs x {n_tok} positions, {n_heads} KV heads x 2 query heads, "
           f"head_dim 256, pages of {ps}, gated",
           toks * n_heads * 288 + 3 * n_seq * n_qh * 1024 + n_seq * n_qh * 4 + table_z.size * 4,
           s, toks, "tokens")
    del out, k_pool, v_pool, ws

    # cache files: save and load of the 4-bit tier's cache (T=32768 rows), and the
    # quantize-on-load of an fp32 file into the fp8 tier; host I/O through the page cache,
    # so file bytes per second, not an HBM fraction
    import tempfile
    T = 32768
    c = torch.randn(T, 512, generator=gen, device=dev)
    r = torch.randn(T, 64, generator=gen, device=dev)
    planes = dict(lat=torch.empty(T, 256, dtype=torch.uint8, device=dev), lat_scale=torch.empty(T, device=dev),
                  rope=torch.empty(T, 64, dtype=torch.uint8, device=dev), rope_scale=torch.empty(T, device=dev))
    kvq.kvq_encode_tq4(c, signs, planes["lat"], planes["lat_scale"])
    kvq.kvq_encode_fp8(r, planes["rope"], planes["rope_scale"])
    p8 = dict(lat=torch.empty(T, 512, dtype=torch.uint8, device=dev), lat_scale=torch.empty(T, device=dev),
              rope=torch.empty(T, 64, dtype=torch.uint8, device=dev), rope_scale=torch.empty(T, device=dev))
    ws_up = torch.empty(kvq.kvq_cache_load_workspace(), dtype=torch.uint8, device=dev)
    with tempfile.TemporaryDirectory() as td:
        f4, f32 = os.path.join(td, "tq4.kvq"), os.path.join(td, "f32.kvq")
        kvq.kvq_cache_save_f32(f32, c, r)
        for name, fn, path in (("kvq_cache_save (TQ4)", lambda: kvq.kvq_cache_save(f4, kvq.FMT_TQ4, planes, T, signs=signs), f4),
                               ("kvq_cache_load (TQ4)", lambda: kvq.kvq_cache_load(f4, kvq.FMT_TQ4, planes, signs=signs), f4),
                               ("kvq_cache_load (fp32 file -> fp8 tier)",
                                lambda: kvq.kvq_cache_load(f32, kvq.FMT_FP8, p8, workspace=ws_up), f32)):
            fn()
            ts = []
            for _ in range(max(3, min(K, 10))):
                t0 = time.perf_counter()
                fn()
                torch.cuda.synchronize()
                ts.append(time.perf_counter() - t0)
            sec = statistics.median(ts)
            nb = os.path.getsize(path)
            print(json.dumps({"suite": "codecs", "kernel": name, "workload": f"T={T} rows, file {nb} B",
                              "us": round(sec * 1e6, 1), "rows_per_s": T / sec,
                              "file_gbs": round(nb / sec / 1e9, 3),
                              "note": "host file I/O through the page cache (wall clock)",
                              "steps": len(ts)}), flush=True)
    del c, r, planes, p8, ws_up

    # a7: sparse row gather of the fp8 MLA cache, top-k = 2048 of T = 131072
    T, k_sel = 131072, 2048
    src = dict(lat=torch.zeros(T, 512, dtype=torch.uint8, device=dev), lat_scale=torch.ones(T, device=dev),
               rope=torch.zeros(T, 64, dtype=torch.uint8, device=dev), rope_scale=torch.ones(T, device=dev))
    idx = torch.from_numpy(W.sparse_indices(T, k_sel, 1, seed=0)[0]).to(dev)
    dst = dict(lat=torch.empty(k_sel, 512, dtype=torch.uint8, device=dev), lat_scale=torch.empty(k_sel, device=dev),
               rope=torch.empty(k_sel, 64, dtype=torch.uint8, device=dev), rope_scale=torch.empty(k_sel, device=dev))
    s = timed(lambda: kvq.kvq_gather_rows(kvq.FMT_FP8, src, T, idx, dst))
    report("kvq_gather (fp8 rows by index)", f"top-k {k_sel} of T={T} rows", k_sel * (584 * 2 + 4), s, k_sel, "rows")


def decode_records(args, dev, wanted=lambda name: True):
    """Every decode configuration, each timed as a CUDA graph of back-to-back calls over a
    stack of distinct caches of about 512 MB (more than L2), so that rows come from HBM
    as in a multi-layer decode.  Returns one record per configuration: the kernel that
    ran, microseconds per call (query image + decode + combine), KV rows/s, and the call
    against both rooflines with the binding one named by the arithmetic intensity."""
    import torch
    import quantized_kv_cache_fp8_gb300 as kvq
    import workloads as W

    hbm_peak, tc_peak, peak_kind = peaks()
    ridge = tc_peak * 1e12 / (hbm_peak * 1e9)      # executed FLOP per byte at the ridge
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    signs = torch.from_numpy(W.sign_bits(0)).to(dev)
    names = {1: "cuda-cores", 2: "tcgen05", 3: "warp-mma", 4: "tcgen05x16", 5: "tcgen05-e4m3",
             6: "tcgen05-e4m3 (fp8 seqs) + tcgen05 (TQ4 seqs)"}
    target = 512 << 20
    records = []

    def encode_pool(n_rows, fmt, mag=None):
        c = torch.randn(n_rows, 512, generator=gen, device=dev)
        r = torch.randn(n_rows, 64, generator=gen, device=dev)
        if mag is not None:
            m = torch.exp(torch.empty(n_rows, 1, device=dev).uniform_(
                float(np.log(mag[0])), float(np.log(mag[1])), generator=gen))
            c *= m
            r *= m
        bits = {kvq.FMT_TQ3: 3, kvq.FMT_TQ4: 4, kvq.FMT_TQ6: 6}.get(fmt, 8)
        lat = torch.empty(n_rows, 512 * bits // 8, dtype=torch.uint8, device=dev)
        ls = torch.empty(n_rows, device=dev)
        rope = torch.empty(n_rows, 64, dtype=torch.uint8, device=dev)
        rs = torch.empty(n_rows, device=dev)
        if fmt == kvq.FMT_FP8:
            kvq.kvq_encode_fp8(c, lat, ls)
        else:
            kvq.kvq_encode_tq(c, signs, bits, lat, ls)
        kvq.kvq_encode_fp8(r, rope, rs)
        return dict(lat=lat, lat_scale=ls, rope=rope, rope_scale=rs)

    def clone(pool):
        return {k: v.clone() for k, v in pool.items()}

    def measure(name, probs, out_shape, rows_read, row_bytes, flops, extra=None):
        n = len(probs)
        ws = torch.empty(max(1, max(kvq.kvq_mla_decode_workspace(p) for p in probs)),
                         dtype=torch.uint8, device=dev)
        out = torch.empty((n,) + out_shape, device=dev)
        lse = torch.empty((n,) + out_shape[:-1], device=dev)

        def calls():
            for i, p in enumerate(probs):
                kvq.kvq_mla_decode(p, out[i], lse[i], ws)
        calls()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            calls()
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        reps = max(3, min(20, args.steps))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        sec = e0.elapsed_time(e1) / 1e3 / (reps * n)
        assert torch.isfinite(out).all()
        gbs = rows_read * row_bytes / sec / 1e9
        tf = flops / sec / 1e12
        intensity = 2 * flops / (rows_read * row_bytes)   # executed (split fp16) per byte
        rec = {"config": name, "kernel": names[kvq.kvq_mla_decode_kernel(probs[0])],
               "us": round(sec * 1e6, 2), "kv_rows_per_s": rows_read / sec,
               "bound": "hbm" if intensity < ridge else "tensor",
               "hbm": {"achieved_gbs": round(gbs, 1), "peak": hbm_peak, "frac": round(gbs / hbm_peak, 4),
                       "bytes": int(rows_read * row_bytes)},
               "tensor": {"achieved_tflops": round(tf, 2), "peak": tc_peak, "frac": round(tf / tc_peak, 4),
                          "executed_frac": round(2 * tf / tc_peak, 4), "flops": int(flops)},
               "stack": f"{n} distinct caches in one CUDA graph, {reps} replays"}
        if extra:
            rec.update(extra)
        records.append(rec)
        return rec

    def one_seq(name, fmt, T, H, idx_k=0, mag=None, overlap=0):
        if not wanted(name):
            return
        rb = {kvq.FMT_FP8: 584, kvq.FMT_TQ4: 328, kvq.FMT_TQ6: 456, kvq.FMT_TQ3: 264}[fmt]
        layers = max(2, min(256, -(-target // (T * rb))))
        base = encode_pool(T, fmt, mag)
        q = W.queries(1, 1, H, seed=0)
        q_lat = torch.from_numpy(q.q_lat).to(dev)
        q_rope = torch.from_numpy(q.q_rope).to(dev)
        seq_len = torch.tensor([T], dtype=torch.int32, device=dev)
        impl = args.decode_impl
        if fmt in (kvq.FMT_TQ3, kvq.FMT_TQ6) and impl in (2, 3):
            impl = 4
        if fmt != kvq.FMT_FP8 and impl == 5:
            impl = 0
        probs, keep = [], []
        for l in range(layers):
            cache = base if l == 0 else clone(base)
            idx = None
            if idx_k:
                idx = torch.from_numpy(W.sparse_indices(T, idx_k, 1, seed=l)).to(dev).reshape(1, 1, idx_k)
            keep.append((cache, idx))
            kw = dict(fp8=cache) if fmt == kvq.FMT_FP8 else dict(tq4=cache, signs=signs)
            probs.append(kvq.make_problem(seq_len=seq_len, q_lat=q_lat, q_rope=q_rope,
                                          sm_scale=W.SM_SCALE, max_seq_len=T, fmt=fmt, idx=idx,
                                          impl=impl, overlap_prior=overlap, **kw))
        n = idx_k or T
        measure(name, probs, (1, 1, H, 512), n, rb, 2 * H * 1088 * n)
        del probs, keep, base
        torch.cuda.empty_cache()

    def batch_seq(name, fmt, n_seq, T, H, overlap=0):
        """n_seq sequences of T rows (contiguous, one query each) in one call: the per-call
        fixed cost (start-up, last tile, combine) spread over n_seq x T rows."""
        if not wanted(name):
            return
        rb = {kvq.FMT_FP8: 584, kvq.FMT_TQ4: 328}[fmt]
        layers = max(2, min(64, -(-target // (n_seq * T * rb))))
        base = encode_pool(n_seq * T, fmt)
        q = W.queries(n_seq, 1, H, seed=0)
        q_lat = torch.from_numpy(q.q_lat).to(dev)
        q_rope = torch.from_numpy(q.q_rope).to(dev)
        seq_len = torch.full((n_seq,), T, dtype=torch.int32, device=dev)
        impl = args.decode_impl
        if fmt != kvq.FMT_FP8 and impl == 5:
            impl = 0
        probs, keep = [], []
        for l in range(layers):
            cache = base if l == 0 else clone(base)
            keep.append(cache)
            kw = dict(fp8=cache) if fmt == kvq.FMT_FP8 else dict(tq4=cache, signs=signs)
            probs.append(kvq.make_problem(seq_len=seq_len, q_lat=q_lat, q_rope=q_rope,
                                          sm_scale=W.SM_SCALE, max_seq_len=T, fmt=fmt,
                                          seq_stride_rows=T, impl=impl, overlap_prior=overlap, **kw))
        measure(name, probs, (n_seq, 1, H, 512), n_seq * T, rb, 2 * H * 1088 * n_seq * T)
        del probs, keep, base
        torch.cuda.empty_cache()

    F8, T4 = kvq.FMT_FP8, kvq.FMT_TQ4
    one_seq("fp8 tiny: T=1024, H=16, magnitudes log-uniform [1e-3, 40]", F8, 1024, 16, mag=(1e-3, 40.0))
    one_seq("TQ4: T=32768, H=64", T4, 32768, 64)
    one_seq("fp8 long context dense: T=131072, H=128", F8, 131072, 128)
    one_seq("fp8 long context sparse: top-k 2048 of T=131072, H=128", F8, 131072, 128, idx_k=2048)
    for fmt, tag in ((F8, "fp8"), (T4, "TQ4")):
        for T in (32768, 131072):
            one_seq(f"HBM point: {tag}, T={T}, H=16", fmt, T, 16)
        batch_seq(f"HBM point, batch: {tag}, 8 seqs x T=32768, H=16", fmt, 8, 32768, 16)
    # the same fp8 calls with overlap_prior: each decode of the graph's back-to-back calls
    # (distinct caches, nothing written between them) may start during the combine before it
    for T in (32768, 131072):
        one_seq(f"HBM point, calls overlapped: fp8, T={T}, H=16", F8, T, 16, overlap=1)
    batch_seq("HBM point, batch, calls overlapped: fp8, 8 seqs x T=32768, H=16", F8, 8, 32768, 16, overlap=1)
    for fmt, tag in ((kvq.FMT_TQ6, "TQ6"), (kvq.FMT_TQ3, "TQ3")):
        one_seq(f"{tag}: T=32768, H=16", fmt, 32768, 16)

    # ragged mixed-tier batch: 32 sequences, L ~ U[1024, 65536], 4 causal queries, H=64
    name = "ragged: 32 seqs, L ~ U[1024, 65536], 4 causal queries, H=64, fp8 + TQ4, pages of 64"
    if wanted(name):
        n_seq, n_q, H, ps = 32, 4, 64, 64
        L, fmt, table, pool_pages = W.ragged_layout(n_seq, 1024, 65536, ps, seed=0)
        pools = {f: encode_pool(pool_pages[f] * ps, f, mag=(1e-2, 10.0)) for f in (F8, T4)}
        q = W.queries(n_seq, n_q, H, seed=0)
        p = kvq.make_problem(seq_len=torch.from_numpy(L).to(dev), q_lat=torch.from_numpy(q.q_lat).to(dev),
                             q_rope=torch.from_numpy(q.q_rope).to(dev), sm_scale=W.SM_SCALE,
                             max_seq_len=int(L.max()), seq_fmt=torch.from_numpy(fmt).to(dev),
                             block_table=torch.from_numpy(table).to(dev), page_size=ps, causal=True,
                             fp8=pools[F8], tq4=pools[T4], signs=signs,
                             impl=0 if args.decode_impl == 5 else args.decode_impl)
        rows_fp8 = int(L[fmt == 1].sum())
        rows_tq4 = int(L[fmt == 2].sum())
        rows = rows_fp8 + rows_tq4
        measure(name, [p], (n_seq, n_q, H, 512), rows, (rows_fp8 * 584 + rows_tq4 * 328) / rows,
                2 * H * n_q * 1088 * rows, extra={"rows": rows})
        del pools
        torch.cuda.empty_cache()
    return records


def run_decode_configs(args, local):
    """One JSON line per decode configuration (see decode_records)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    for rec in decode_records(args, dev, wanted=lambda name: args.only in name):
        rec.update({"suite": "decode-configs", "decode_impl": args.decode_impl})
        print(json.dumps(rec), flush=True)


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.suite == "codecs":
        if rank == 0:
            run_codecs(args, local)
    elif args.suite == "decode-configs":
        if rank == 0:
            run_decode_configs(args, local)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
