"""Benchmark of the paged KV-cache hot path on GB300.

One step is one decode layer-step of the whole hot path: pa_store_decode (the step's new K/V
rows into the pool and the split-K paged GQA decode in one launch, + the merge), over the
``qwen3_06b_decode`` workload (256 sequences, contexts U[100, 4096], 16/8 heads, D 128,
256-token blocks, bf16). Two layers' pools are used in turn so that consecutive steps read
different data; each pool (2.7 GB) is far larger than the 129 MB L2.

Headline: KV bytes the step must read (every cached row of K and V once per kv head) divided
by the device time of the step, in GB/s, and as a fraction of the measured HBM peak; decode
steps per second per layer. The same line carries:

* ``roofline``: the step's call (split kernel + merge): its mean duration over the timed region
  (the events around the K steps; each step is exactly this call, and no event between steps
  holds a launch back from overlapping the one before), against the measured copy bandwidth;
* ``e2e``: the same metric through the C-ABI's host-buffer call (pa_store_decode_host): every
  step copies its inputs from pinned host memory and reads the output back, synchronising each
  step (the pool stays resident, as in an engine);
* ``cpu_baseline``: the fp64 CPU oracle on a bounded sample of the same workload, on the
  host's cores;
* ``rows``: the other rows of the path measured the same way: the same step as two calls
  (pa_store_kv, then pa_decode), the store alone, the varlen prefill with a 512-token cached
  prefix (``prefill_prefix``) with its store, the same prefill at the Qwen2.5-0.5B head shape
  (``qwen25_prefill``: 14/2 heads, head dim 64), and the two small decode workloads as CUDA graphs.

``--impl reference`` times the CPU oracle as the reference arm, on the same metric.
Multi-GPU (torchrun): every rank runs an independent replica (the path shards by sequence
with no exchange), value = all ranks' bytes / the slowest rank's time.
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
import tempfile
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

import workloads as W  # noqa: E402

METRIC = "paged-decode KV-read GB/s (% of GB300 HBM peak); decode steps/sec per layer"
DEFAULT_WORKLOAD = "qwen3_06b_decode"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic (read + write bytes) of one launch, from the ncu captures of these kernels (layer 0
# of the default workload; prefill_prefix; qwen25_prefill). Each is valid only for the kernel sources it was taken
# on, identified by their hash; after any change the bench reports null.
DECODE_TRAFFIC = {"sources": ("decode.cu", "pa_common.cuh"), "bytes": 2_289_404_160,
                  "sha256": "32d9050a51c21d042a5c2a0305b231dea999efc7c6625484aaf31d9639da8bb0"}
STORE_TRAFFIC = {"sources": ("store_kv.cu", "pa_common.cuh"), "bytes": 218_096_128,
                 "sha256": "9940671f5a00740d1ba3ee485ac0d8bdb7dee7db79bbd1fe95feb25da0dc412c"}
PREFILL_TRAFFIC = {"sources": ("prefill_tc.cu", "pa_common.cuh"), "bytes": 418_674_432,
                   "sha256": "d665bf6dcb2d3691c3698422946b45614298a0afd57c138209ca60fe9fdeb949"}
PREFILL_QWEN25_TRAFFIC = {"sources": ("prefill_tc.cu", "pa_common.cuh"), "bytes": 111_464_960,
                          "sha256": "d665bf6dcb2d3691c3698422946b45614298a0afd57c138209ca60fe9fdeb949"}


def peaks() -> tuple[dict, str]:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        return json.loads(p.read_text()), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kv_bytes(context_lens, Hkv, D, elem=2) -> int:
    return int(np.asarray(context_lens, np.int64).sum()) * Hkv * D * 2 * elem


def prefill_flops(q_lens, k_lens, Hq, D) -> int:
    tot = 0
    for ql, kl in zip(np.asarray(q_lens, np.int64), np.asarray(k_lens, np.int64)):
        P = int(kl - ql)
        tot += 4 * Hq * D * (int(ql) * P + int(ql) * (int(ql) + 1) // 2)
    return tot


def src_hash(*names: str) -> str:
    m = hashlib.sha256()
    for name in names:
        m.update((ROOT / "paged_kv_cache_83_gb300" / "csrc" / name).read_bytes())
    return m.hexdigest()


def traffic_of(rec: dict):
    return rec["bytes"] if src_hash(*rec["sources"]) == rec["sha256"] else None


def step_config(workload: str, n_layers: int, world: int) -> dict:
    """The ``config`` object of the JSON line: the workload one step runs (rank 0's layers),
    computed from its lengths alone, so that both arms print the same keys and values."""
    w = W.CONFIGS[workload]
    p = w.params
    nbytes = [kv_bytes(W.lengths(workload, rank_seed(w.seed, 0, l)), p["Hkv"], p["D"])
              for l in range(n_layers)]
    mean = statistics.mean(nbytes)
    return {"workload": workload, "seqs": int(len(W.lengths(workload, w.seed))), "Hq": p["Hq"],
            "Hkv": p["Hkv"], "D": p["D"], "block_size": p["block_size"],
            "kv_bytes_per_step": int(mean), "layers_rotated": n_layers,
            "l2": f"inputs larger than L2: each step reads a {mean / 1e9:.1f} GB KV set of its own "
                  f"layer ({n_layers} layers alternate)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


# ---------------------------------------------------------------------------------------------
# distributed plumbing
# ---------------------------------------------------------------------------------------------

def rank_seed(base: int, rank: int, layer: int) -> int:
    """Seed of one rank's layer: every rank runs its own replica on its own data."""
    return base + 1000 * rank + layer


def slowest(torch, value: float, dist, device) -> float:
    """The largest value over the ranks (the slowest rank's time); the value itself alone."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_gbs(world: int, bytes_per_rank: float, elapsed_ms: float) -> float:
    """Whole-job GB/s of `world` replicas that each moved bytes_per_rank in the slowest rank's
    elapsed_ms."""
    return world * bytes_per_rank / (elapsed_ms * 1e-3) / 1e9


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons while the GPU is busy."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in Path(self.path).read_text().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]), "power": float(parts[3]),
                             "hw": parts[5], "hw_thermal": parts[6], "sw_thermal": parts[7],
                             "sw_power": parts[8]})
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        busy = [r for r in rows if r["power"] > 200.0] or rows
        reasons = []
        for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                          ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
            if any(r[key].lower() == "active" for r in busy):
                reasons.append(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(busy),
                "power_w_median": statistics.median(r["power"] for r in busy)}


# ---------------------------------------------------------------------------------------------
# CPU oracle timing (the baseline and the reference arm)
# ---------------------------------------------------------------------------------------------

def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (model name, else implementer/part ids), with the
    core count."""
    name = ""
    try:
        info = open("/proc/cpuinfo").read().splitlines()
        for key in ("model name", "Model name", "CPU part"):
            hits = [l.split(":", 1)[1].strip() for l in info if l.startswith(key)]
            if hits:
                name = f"{key}: {hits[0]}"
                break
    except OSError:
        pass
    import platform
    return f"{platform.machine()}, {os.cpu_count()} cores" + (f", {name}" if name else "")


def oracle_decode_rate(case, budget_s: float = 12.0, threads: int = 0) -> dict:
    """Time the oracle's decode on a bounded sample of the case's sequences (after applying the
    step's store, as the GPU step does), growing the sample until ~budget_s of work."""
    import oracle
    orc = oracle.get()
    threads = threads or (os.cpu_count() or 1)
    kc, vc = orc.store_kv(case.k_new, case.v_new, case.k_cache, case.v_cache, case.slot_mapping)
    order = np.random.default_rng(123).permutation(case.B)
    n = min(case.B, 2)
    while True:
        rows = np.sort(order[:n])
        t = time.perf_counter()
        orc.decode(case.q[rows], kc, vc, case.block_tables[rows], case.context_lens[rows],
                   scale=case.scale, dtype=case.dtype, threads=threads)
        dt = time.perf_counter() - t
        if dt >= budget_s / 4 or n == case.B:
            break
        n = min(case.B, max(n + 1, int(n * min(8.0, (budget_s / 4) / max(dt, 1e-3)))))
    reps = 1
    if dt < budget_s / 4:  # the whole case is quick: repeat it to time a meaningful span
        reps = int(min(1000, max(1, (budget_s / 4) / max(dt, 1e-4))))
        t = time.perf_counter()
        for _ in range(reps):
            orc.decode(case.q[rows], kc, vc, case.block_tables[rows], case.context_lens[rows],
                       scale=case.scale, dtype=case.dtype, threads=threads)
        dt = (time.perf_counter() - t) / reps
    nbytes = kv_bytes(case.context_lens[rows], case.Hkv, case.D)
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": min(threads, orc.max_threads()), "kind": "oracle",
            "sample": f"{n} of {case.B} sequences of {case.name} (store applied, fp64 decode), "
                      f"{nbytes / 1e6:.1f} MB of KV in {dt:.4f} s" + (f", mean of {reps} runs" if reps > 1 else ""),
            "seconds": dt, "seqs": int(n), "rows": rows}


def run_reference(args, ws_, rank):
    if rank != 0:
        return
    case = W.make(args.workload)
    probe = oracle_decode_rate(case, budget_s=4.0)
    rows = probe["rows"]
    import oracle
    orc = oracle.get()
    kc, vc = orc.store_kv(case.k_new, case.v_new, case.k_cache, case.v_cache, case.slot_mapping)
    times = []
    for i in range(args.warmup + args.steps):
        t = time.perf_counter()
        orc.decode(case.q[rows], kc, vc, case.block_tables[rows], case.context_lens[rows],
                   scale=case.scale, dtype=case.dtype, threads=os.cpu_count() or 1)
        if i >= args.warmup:
            times.append(time.perf_counter() - t)
    nbytes = kv_bytes(case.context_lens[rows], case.Hkv, case.D)
    tot = sum(times)
    value = nbytes * len(times) / tot / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws_,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": step_config(args.workload, args.layers, ws_),
            "cpu_baseline": {"value": value, "unit": "GB/s", "kind": "oracle",
                             "cores": orc.max_threads(),
                             "sample": f"{len(rows)} of {case.B} sequences of {case.name} (layer 0) "
                                       f"per step, fp64"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------------------------

def to_dev(torch, bits, dt, dev):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev)
    return t.view(torch.float16 if dt == "f16" else torch.bfloat16)


class DecodeLayer:
    def __init__(self, torch, pa, case, dev):
        self.c = case
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
        self.kc = to_dev(torch, case.k_cache, case.dtype, dev)
        self.vc = to_dev(torch, case.v_cache, case.dtype, dev)
        self.q = to_dev(torch, case.q, case.dtype, dev)
        self.k_new = to_dev(torch, case.k_new, case.dtype, dev)
        self.v_new = to_dev(torch, case.v_new, case.dtype, dev)
        self.bt, self.cl, self.sm = i32(case.block_tables), i32(case.context_lens), i32(case.slot_mapping)
        n = pa.pa_decode_workspace_size(case.B, case.Hq, case.Hkv, case.D, case.max_blocks_per_seq,
                                        case.block_size)
        self.ws = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
        self.out = torch.empty_like(self.q)


def run_gpu(args, ws_, rank, local):
    import torch
    import paged_kv_cache_83_gb300 as pa

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if ws_ > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    pa.load()
    stream = torch.cuda.current_stream()
    pk, pk_kind = peaks()
    hbm = float(pk["hbm_gbs"])
    # the prefill kernel is timed alone (L2 flushed around it): its fraction is of the burst peak
    bf16_peak = float(pk["bf16_tflops"])
    bf16_sustained = float(pk.get("bf16_tflops_sustained", bf16_peak))

    if args.only is not None:
        # one group of rows alone: the prefill rows (store + varlen prefill on the two prefill
        # workloads) or the small decode workloads as CUDA graphs; a short command for profiling
        # their kernels without the headline's decode pools on the device
        if args.only == "prefill":
            rows = bench_prefill(torch, pa, dev, stream, bf16_peak, bf16_sustained, hbm, args, pk_kind)
        else:
            rows = {"decode_small_graphs": bench_small_decode(torch, pa, dev, hbm)}
        if rank == 0:
            print(json.dumps({"rows": rows}), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return

    # ---- inputs: two layers of the decode workload (seeds differ per layer and rank) ----
    base = W.CONFIGS[args.workload].seed
    layers = [DecodeLayer(torch, pa, W.make(args.workload, seed=rank_seed(base, rank, l)), dev)
              for l in range(args.layers)]
    c0 = layers[0].c
    nbytes = [kv_bytes(L.c.context_lens, L.c.Hkv, L.c.D) for L in layers]
    nl = len(layers)
    plan_splits = pa.pa_decode_workspace_size(c0.B, c0.Hq, c0.Hkv, c0.D, c0.max_blocks_per_seq,
                                              c0.block_size) > 0
    # one layer step = pa_store_decode: the store of the new token and the decode in one launch
    # (+ the merge kernel when contexts are split across CTAs)
    launches_per_step = 1 + (1 if plan_splits else 0)

    ev = lambda: torch.cuda.Event(enable_timing=True)

    def step(i):
        L = layers[i % nl]
        pa.pa_store_decode(L.out, L.q, L.k_new, L.v_new, L.kc, L.vc, L.bt, L.cl, L.c.scale,
                           workspace=L.ws)

    def barrier():
        if dist is not None:
            dist.barrier()

    for i in range(args.warmup):
        step(i)
    clocks = Clocks(local)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    t0, t1 = ev(), ev()
    t0.record(stream)
    for i in range(args.steps):
        step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    # keep the GPU busy ~1 s more with the same step so the clock sampler sees it under load
    t_end = time.perf_counter() + (0.0 if args.no_clock_tail else 1.0)
    j = 0
    while time.perf_counter() < t_end:
        step(j)
        j += 1
        if j % 64 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    clk = clocks.stop()

    elapsed = t0.elapsed_time(t1)  # ms
    # this rank's mean call: the steps run back to back, one pa_store_decode each
    dec_mean = elapsed / args.steps
    # the same step as two calls (pa_store_kv, then pa_decode), for comparison
    n2 = max(3, min(args.steps, 200))
    st_ev = [(ev(), ev(), ev()) for _ in range(n2)]
    for i in range(n2):
        L = layers[i % nl]
        st_ev[i][0].record(stream)
        pa.pa_store_kv(L.k_new, L.v_new, L.kc, L.vc, L.sm)
        st_ev[i][1].record(stream)
        pa.pa_decode(L.out, L.q, L.kc, L.vc, L.bt, L.cl, L.c.scale, workspace=L.ws)
        st_ev[i][2].record(stream)
    torch.cuda.synchronize()
    st_ms = [a.elapsed_time(b) for a, b, _ in st_ev]
    two_ms = [a.elapsed_time(c) for a, _, c in st_ev]
    if dist is not None:
        elapsed = slowest(torch, elapsed, dist, dev)
    ms_step = elapsed / args.steps
    step_bytes = sum(nbytes[i % nl] for i in range(args.steps))
    value = weak_gbs(ws_, step_bytes, elapsed)
    dec_bytes_mean = statistics.mean(nbytes[i % nl] for i in range(args.steps))
    achieved = dec_bytes_mean / (dec_mean * 1e-3) / 1e9
    # traffic was captured on layer 0; report it for the launches on that layer
    traffic = traffic_of(DECODE_TRAFFIC)

    # ---- e2e: inputs from pinned host memory each step, output read back each step ----
    # through the C-ABI's host-buffer entry (pa_store_decode_host): the library queues the
    # transfer of the packed inputs into its workspace, the fused store + decode, and the
    # transfer of the output back
    L = layers[0]
    c = L.c
    # the step's inputs sit in one pinned buffer at the library's packed offsets, as an engine's
    # scheduler would write them, so the call moves them in one copy
    h_offs, h_total = pa.pa_store_decode_host_layout(c.B, c.Hq, c.Hkv, c.D, c.max_blocks_per_seq)
    h_pack = torch.zeros(h_total, dtype=torch.uint8).pin_memory()
    h_in = []
    for x, o in zip((L.q, L.k_new, L.v_new, L.bt, L.cl), h_offs):
        nb_ = x.numel() * x.element_size()
        v = h_pack[o:o + nb_].view(x.dtype).view(x.shape)
        v.copy_(x.cpu())
        h_in.append(v)
    h_out = torch.empty(L.out.shape, dtype=L.out.dtype).pin_memory()
    ws_host = torch.empty(max(256, pa.pa_store_decode_host_workspace_size(
        c.B, c.Hq, c.Hkv, c.D, c.max_blocks_per_seq, c.block_size)), dtype=torch.uint8, device=dev)
    h2d = h_total  # the packed span, alignment gaps included
    d2h = h_out.numel() * h_out.element_size()
    e_steps = 0 if args.no_e2e else max(1, min(args.steps, 200))

    host_s = [0.0]

    def e2e_step():
        q, kn, vn, bt, cl = h_in
        t = time.perf_counter()
        pa.pa_store_decode_host(h_out, q, kn, vn, L.kc, L.vc, bt, cl, c.scale, workspace=ws_host)
        host_s[0] += time.perf_counter() - t
        stream.synchronize()

    # the same step with torch staging the same packed buffer (one copy) around the device
    # call, for comparison
    d_buf = torch.empty(h_total, dtype=torch.uint8, device=dev)
    d_in = [d_buf[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape)
            for x, o in zip(h_in, h_offs)]

    def torch_staged_step():
        d_buf.copy_(h_pack, non_blocking=True)
        q, kn, vn, bt, cl = d_in
        pa.pa_store_decode(L.out, q, kn, vn, L.kc, L.vc, bt, cl, c.scale, workspace=L.ws)
        h_out.copy_(L.out, non_blocking=True)
        stream.synchronize()

    def timed_loop(fn):
        for _ in range(3 if e_steps else 0):
            fn()
        barrier()
        torch.cuda.synchronize()
        e0, e1 = ev(), ev()
        e0.record(stream)
        for _ in range(e_steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        if dist is not None:
            ms = slowest(torch, ms, dist, dev)
        return ms

    e_ms = timed_loop(e2e_step)
    host_us = host_s[0] / (e_steps + 3) * 1e6 if e_steps else None  # the call itself, on the host
    e2e_value = weak_gbs(ws_, nbytes[0] * e_steps, e_ms) if e_steps else None
    ts_ms = timed_loop(torch_staged_step) if e_steps else 0.0
    e2e_torch_staged = weak_gbs(ws_, nbytes[0] * e_steps, ts_ms) if e_steps else None

    # ---- other rows: prefill with a cached prefix (store + varlen prefill) ----
    rows = {}
    if not args.skip_prefill:
        rows.update(bench_prefill(torch, pa, dev, stream, bf16_peak, bf16_sustained, hbm, args,
                                  pk_kind))
    if not args.skip_small:
        rows["decode_small_graphs"] = bench_small_decode(torch, pa, dev, hbm)
    if not args.skip_groups:
        rows["decode_group_sweep"] = bench_group_sweep(torch, pa, dev, hbm)
    if not args.skip_longtail:
        rows["decode_longtail"] = bench_longtail(torch, pa, dev, hbm)
    if rank == 0 and not args.skip_cpu:
        rows["block_manager"] = bench_block_manager(pa)
    st_mean = statistics.mean(st_ms)
    st_bytes = 4 * c0.B * c0.Hkv * c0.D * 2
    rows["store_kv_decode"] = {"kernel": "store_kv_kernel", "ms": st_mean,
                               "GB_per_s": st_bytes / (st_mean * 1e-3) / 1e9,
                               "bytes": st_bytes, "note": "256 new rows: launch-latency bound"}
    rows["decode"] = {"kernel": "pa_store_decode: decode_kernel (+ the new token's store) + "
                                "decode_merge_kernel", "ms": dec_mean,
                      "GB_per_s": achieved, "frac_of_hbm": achieved / hbm}
    rows["two_call_step"] = {"calls": "pa_store_kv + pa_decode", "ms": statistics.mean(two_ms),
                             "GB_per_s": kv_bytes(c0.context_lens, c0.Hkv, c0.D) /
                             (statistics.mean(two_ms) * 1e-3) / 1e9,
                             "note": "layer 0's KV bytes; the fused call is the step"}

    cpu = None
    if rank == 0 and not args.skip_cpu:
        r = oracle_decode_rate(layers[0].c)
        r.pop("rows")
        r.pop("seqs")
        cpu = r
        cpu["cpu_model"] = cpu_model()
        # beside it: the oracle on one thread, and on the two small decode configurations
        one = oracle_decode_rate(layers[0].c, budget_s=4.0, threads=1)
        cpu["one_thread"] = {"value": one["value"], "unit": "GB/s", "sample": one["sample"]}
        small = {}
        for name in ("tiny", "qwen25_05b_decode"):
            sc = W.make(name)
            a = oracle_decode_rate(sc, budget_s=2.0)
            b = oracle_decode_rate(sc, budget_s=2.0, threads=1)
            small[name] = {"all_cores_GB_per_s": a["value"], "one_thread_GB_per_s": b["value"],
                           "sample_all_cores": a["sample"], "sample_one_thread": b["sample"]}
        cpu["small_configs"] = small

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws_, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": c0.dtype, "data": "synthetic",
        "config": step_config(args.workload, nl, ws_),
        "pct_of_hbm_peak": 100.0 * value / hbm / ws_,
        "decode_steps_per_sec_per_layer": 1e3 / ms_step,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic,
                     "kernel": "pa_store_decode: decode_kernel + decode_merge_kernel",
                     "peak_source": f"{pk_kind} hbm_gbs"},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e_steps,
                "call": "pa_store_decode_host (C-ABI, host buffers)",
                "note": "pool resident; per step one call that queues the H2D copy of q, new K/V, "
                        "tables and lengths (one pinned buffer in the library's packed layout), "
                        "the fused store + decode, and the D2H copy of the output; then a "
                        "stream sync",
                "torch_staged_value": e2e_torch_staged, "host_us_per_call": host_us,
                "device_ms_per_step": ms_step, "e2e_ms_per_step": e_ms / e_steps if e_steps else None},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "rows": rows,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def bench_small_decode(torch, pa, dev, hbm) -> dict:
    """The two small decode workloads, whose whole KV set fits in L2: one layer-step is a few
    microseconds, so they are timed as a CUDA graph of L independent layers (own pools and inputs),
    L chosen so that the graph's pools exceed 4x L2 (at most 32), and reported per layer."""
    ev = lambda: torch.cuda.Event(enable_timing=True)
    l2 = int(torch.cuda.get_device_properties(dev).L2_cache_size)
    res = {}
    for name in ("tiny", "qwen25_05b_decode"):
        base = W.CONFIGS[name].seed
        first = W.make(name, seed=base)
        pool_bytes = 2 * int(first.k_cache.nbytes)
        n_layers = max(1, min(32, -(-4 * l2 // pool_bytes)))
        layers = [DecodeLayer(torch, pa, first if l == 0 else W.make(name, seed=base + 100 + l), dev)
                  for l in range(n_layers)]
        kv = statistics.mean(kv_bytes(L.c.context_lens, L.c.Hkv, L.c.D) for L in layers)

        def body(mode):
            for L in layers:
                if mode == "fused":
                    pa.pa_store_decode(L.out, L.q, L.k_new, L.v_new, L.kc, L.vc, L.bt, L.cl,
                                       L.c.scale, workspace=L.ws)
                    continue
                if mode == "two":
                    pa.pa_store_kv(L.k_new, L.v_new, L.kc, L.vc, L.sm)
                pa.pa_decode(L.out, L.q, L.kc, L.vc, L.bt, L.cl, L.c.scale, workspace=L.ws)

        us = {}
        for mode in ("fused", "two", "decode"):
            body(mode)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                body(mode)
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            ts = []
            for _ in range(20):
                a, b = ev(), ev()
                a.record()
                g.replay()
                b.record()
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b))
            us[mode] = statistics.median(ts) * 1e3 / n_layers
            del g
        c = layers[0].c
        res[name] = {"seqs": c.B, "Hq": c.Hq, "Hkv": c.Hkv, "D": c.D, "block_size": c.block_size,
                     "dtype": c.dtype, "kv_bytes_per_layer": int(kv), "layers_in_graph": n_layers,
                     "us_store_decode_per_layer": us["fused"],
                     "us_store_then_decode_per_layer": us["two"], "us_decode_per_layer": us["decode"],
                     "decode_GB_per_s": kv / (us["decode"] * 1e-6) / 1e9,
                     "frac_of_hbm": kv / (us["decode"] * 1e-6) / 1e9 / hbm,
                     "l2": f"{n_layers} layers x {pool_bytes / 1e6:.1f} MB of pools per graph replay"}
        del layers
        torch.cuda.empty_cache()
    return res


# GQA group sizes of common model shapes beyond the two named decode workloads: 256 sequences,
# contexts U[100, 4096] (seeded), each KV set larger than L2
GROUP_SWEEP = ((4, 4, 128, 256, "bf16"), (7, 2, 64, 16, "f16"), (8, 2, 128, 256, "bf16"))


def bench_group_sweep(torch, pa, dev, hbm) -> dict:
    """pa_decode across GQA group sizes G = Hq / Hkv (G >= 4 runs the tensor-core consumers).
    Like the main step: calls back to back on two layers whose pools alternate (each KV set is
    larger than L2), one pair of CUDA events around the n calls, the mean call reported. (An event
    between two calls would hold the next decode launch until the previous merge has finished,
    which no step loop does: 2-3 µs a call.)"""
    res = {}
    for G, Hkv, D, bs, dt in GROUP_SWEEP:
        lens = np.random.default_rng(0).integers(100, 4096, size=256, endpoint=True)
        layers = [DecodeLayer(torch, pa, W.decode_case(B=256, Hq=G * Hkv, Hkv=Hkv, D=D, block_size=bs,
                                                       dtype=dt, context_lens=lens, seed=1 + l), dev)
                  for l in range(2)]
        c = layers[0].c

        def run(L):
            pa.pa_decode(L.out, L.q, L.kc, L.vc, L.bt, L.cl, L.c.scale, workspace=L.ws)

        for i in range(4):
            run(layers[i % 2])
        n = 20
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for i in range(n):
            run(layers[i % 2])
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
        kv = kv_bytes(c.context_lens, c.Hkv, c.D)
        res[f"G{G}_Hkv{Hkv}_D{D}_bs{bs}_{dt}"] = {
            "us": ms * 1e3, "kv_bytes": kv, "GB_per_s": kv / (ms * 1e-3) / 1e9,
            "frac_of_hbm": kv / (ms * 1e-3) / 1e9 / hbm,
            "consumers": "tensor-core fragments" if G >= 4 else "fp32"}
        del layers
        torch.cuda.empty_cache()
    return res


def bench_longtail(torch, pa, dev, hbm) -> dict:
    """The max-batch long-tail decode workload (512 sequences, lognormal contexts up to 16384, a
    near-full pool): the same step as the headline (pa_store_decode), calls back to back on one
    layer whose 6.8 GB KV set is far larger than L2, one pair of CUDA events around the n calls;
    the mean call reported."""
    c = W.make("longtail_decode")
    L = DecodeLayer(torch, pa, c, dev)

    def run():
        pa.pa_store_decode(L.out, L.q, L.k_new, L.v_new, L.kc, L.vc, L.bt, L.cl, c.scale, workspace=L.ws)

    for _ in range(3):
        run()
    n = 10
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(n):
        run()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    kv = kv_bytes(c.context_lens, c.Hkv, c.D)
    res = {"workload": "longtail_decode", "seqs": c.B, "kv_bytes": kv, "ms": ms,
           "GB_per_s": kv / (ms * 1e-3) / 1e9, "frac_of_hbm": kv / (ms * 1e-3) / 1e9 / hbm,
           "call": "pa_store_decode"}
    del L
    torch.cuda.empty_cache()
    return res


def bench_block_manager(pa) -> dict:
    """The host block manager on a serving-shaped trace: 256 sequences that share a 512-token
    system prompt, 256-token blocks; admit all, 256 decode appends each, release all. Timed
    through the Python binding (one ctypes call per operation, which dominates the per-call
    times) and, beside it, the reference model in oracle/block_manager.py on the same trace."""
    from oracle.block_manager import BlockManagerModel
    rng = np.random.default_rng(7)
    bs, n_seq, steps = 256, 256, 256
    system = list(rng.integers(0, 150000, size=512))
    prompts = [system + list(rng.integers(0, 150000, size=int(rng.integers(100, 1000))))
               for _ in range(n_seq)]
    need = sum(-(-(len(t) + steps) // bs) for t in prompts)
    N = int(need * 1.25)
    out = {"trace": f"{n_seq} seqs, 512-token shared prefix + U[100,1000), {steps} appends each, "
                    f"bs {bs}, {N} blocks"}
    arrays = [np.asarray(p, dtype=np.int32) for p in prompts]  # the library takes int32 arrays
    for name, make, ps in (("library", lambda: pa.BlockManager(N, bs), arrays),
                           ("reference_model", lambda: BlockManagerModel(N, bs), prompts)):
        bm = make()
        t0 = time.perf_counter()
        cached = sum(bm.allocate(i, p) for i, p in enumerate(ps))
        t1 = time.perf_counter()
        for step in range(steps):
            for i in range(n_seq):
                bm.append(i, step)
        t2 = time.perf_counter()
        for i in range(n_seq):
            bm.release(i)
        t3 = time.perf_counter()
        out[name] = {"us_per_allocate": (t1 - t0) / n_seq * 1e6,
                     "us_per_append": (t2 - t1) / (n_seq * steps) * 1e6,
                     "us_per_release": (t3 - t2) / n_seq * 1e6, "tokens_cached": int(cached)}
    return out


def time_prefill(torch, pa, dev, stream, name, steps):
    """Store + varlen prefill of one prefill workload, L2 flushed before each iteration: the median
    CUDA-event times (ms) of the store and of the prefill, and the case."""
    c = W.make(name)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
    kc, vc = to_dev(torch, c.k_cache, c.dtype, dev), to_dev(torch, c.v_cache, c.dtype, dev)
    k, v, q = (to_dev(torch, x, c.dtype, dev) for x in (c.k, c.v, c.q))
    sm, cq, ck, bt = i32(c.slot_mapping), i32(c.cu_seqlens_q), i32(c.cu_seqlens_k), i32(c.block_tables)
    out = torch.empty_like(q)
    # 256 MB > L2, swept by a read (a reduction) between iterations: L2 is left holding clean lines
    # of the sweep, so the timed calls neither hit their own data nor pay for dirty write-backs
    flush = torch.zeros(256 << 20, dtype=torch.uint8, device=dev).view(torch.int32)

    def run(timed_evs=None):
        if timed_evs:
            timed_evs[0].record(stream)
        pa.pa_store_kv(k, v, kc, vc, sm)
        if timed_evs:
            timed_evs[1].record(stream)
        pa.pa_prefill_varlen(out, q, None, None, kc, vc, cq, ck, c.max_seqlen_q, c.max_seqlen_k, bt,
                             Hkv=c.Hkv, scale=c.scale)
        if timed_evs:
            timed_evs[2].record(stream)

    for _ in range(3):
        run()
    n = max(3, min(steps, 50))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    torch.cuda.synchronize()
    # a bounded on-device wait (outside the events) while the host queues the timed calls, so
    # that a host stall cannot put launch latency between the first event and the store (a private
    # torch helper: without it the calls are timed as they come)
    gpu_sleep = getattr(torch.cuda, "_sleep", None)
    for e in evs:
        torch.amax(flush)  # L2 flush between iterations (outside the events)
        if gpu_sleep is not None:
            gpu_sleep(200_000)
        run(e)
    torch.cuda.synchronize()
    st = statistics.median(e[0].elapsed_time(e[1]) for e in evs)
    pf = statistics.median(e[1].elapsed_time(e[2]) for e in evs)
    return st, pf, c


def bench_prefill(torch, pa, dev, stream, bf16_peak, bf16_sustained, hbm, args, pk_kind) -> dict:
    rows = {}
    for name, row, traffic in (("prefill_prefix", "prefill", PREFILL_TRAFFIC),
                               ("qwen25_prefill", "prefill_qwen25", PREFILL_QWEN25_TRAFFIC)):
        st, pf, c = time_prefill(torch, pa, dev, stream, name, args.steps)
        flops = prefill_flops(c.q_lens, c.k_lens, c.Hq, c.D)
        rows[row] = {"workload": name, "kernel": "prefill_tc_kernel",
                     "Hq": c.Hq, "Hkv": c.Hkv, "D": c.D, "block_size": c.block_size, "dtype": c.dtype,
                     "ms": pf, "TFLOP_per_s": flops / (pf * 1e-3) / 1e12,
                     "frac_of_bf16_peak": flops / (pf * 1e-3) / 1e12 / bf16_peak,
                     "peak": bf16_peak, "peak_source": f"{pk_kind} bf16_tflops (burst: the "
                                                       f"kernel is timed alone)",
                     "frac_of_bf16_sustained": flops / (pf * 1e-3) / 1e12 / bf16_sustained,
                     "flops": flops, "l2": "flushed between iterations (a 256 MB read sweep)",
                     "traffic": traffic_of(traffic)}
        if name == "prefill_prefix":
            st_bytes = 4 * int(c.q.shape[0]) * c.Hkv * c.D * 2
            rows["store_kv_prefill"] = {"kernel": "store_kv_kernel", "ms": st, "bytes": st_bytes,
                                        "GB_per_s": st_bytes / (st * 1e-3) / 1e9,
                                        "frac_of_hbm": st_bytes / (st * 1e-3) / 1e9 / hbm,
                                        "traffic": traffic_of(STORE_TRAFFIC),
                                        "traffic_note": "ncu DRAM read + write of one launch; part of "
                                                        "the writes are still in L2 when it ends"}
    return rows


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=[k for k, w in W.CONFIGS.items() if w.kind == "decode"])
    ap.add_argument("--skip-prefill", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-small", action="store_true",
                    help="skip the CUDA-graph timing of the two small decode workloads")
    ap.add_argument("--skip-groups", action="store_true",
                    help="skip the decode timing across GQA group sizes")
    ap.add_argument("--skip-longtail", action="store_true",
                    help="skip the long-tail 512-sequence decode row")
    ap.add_argument("--layers", type=int, default=2, help="layers whose pools alternate")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clock-tail", action="store_true")
    ap.add_argument("--only", choices=["prefill", "small"], default=None,
                    help="run one row alone (no headline line): for profiling its kernels")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    ws_, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, ws_, rank)
        return
    run_gpu(args, ws_, rank, local)


if __name__ == "__main__":
    main()
