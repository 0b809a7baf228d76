#!/usr/bin/env python3
"""Benchmark of the C128 compressor (compress -> RMSNorm -> FP8/UE8M0 + RoPE -> paged store).

Workload: the all-boundary sweep at token_num = 16374 — each token its own request at a window
end, 16 distinct state blocks per token (8.58 GB of fp32 state read per call), kv block size 2.
A step is one call of the whole path (plan kernel + compress kernel) on inputs already resident
in HBM. The state is larger than L2, so no flush is needed between steps.

Prints one JSON line: compressed windows/s (whole job), ms per step, the dominant kernel's
roofline (algorithmic bytes / CUDA-event kernel time vs the measured HBM copy bandwidth),
an end-to-end figure through the public API with the per-step metadata uploaded from pinned host
memory and the k_cache read back, SM clocks sampled during the timed region, the CPU oracle
timed on a bounded sample of the same workload, and µs/call over the token_num sweep.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-sweep]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from deepseek_v4_sparse_c128_gb300 import inputs  # noqa: E402

METRIC = "compressed windows/s and achieved HBM GB/s vs GB300 peak; µs per call vs token_num"
UNIT = "windows/s"
HEADLINE_T = 16374
STATE_BYTES_PER_WINDOW = 128 * 1024 * 4                       # 524,288
ALGO_BYTES_PER_WINDOW = STATE_BYTES_PER_WINDOW + 64 + 256 + 584  # + block ids, cos/sin row, k_cache write
PAGES_US_16374 = 1425.900  # vLLM PR #44230, Performance table (B300), token_num 16374
OTHER_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "other_configurations_traffic.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "compress_kernel_sweep4096_traffic.json")


def workload_config(T: int, n_gpus: int) -> dict:
    return {"workload": f"sweep{T}: all-boundary, token_num {T}, each token its own request at a window end, "
                        f"16 distinct fp32 state blocks per token ({T * STATE_BYTES_PER_WINDOW / 1e9:.2f} GB of "
                        f"state per call), kv block size 2",
            "token_num": T, "active_windows": T, "kv_block_size": 2, "state_block_size": 8, "head": 512,
            "l2": "inputs larger than L2 (state read per call >> 129 MB)", "parallelism": f"replicas x{n_gpus}"}


# ------------------------------------------------------------------------------- distributed
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max_sum(ws, local_ms: float, local_units: float):
    """(max over ranks of the timed-region length, sum over ranks of the units processed)."""
    if ws == 1:
        return local_ms, local_units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ------------------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str):
        self.uuid = uuid
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                                          "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            time.sleep(0.3)
        except FileNotFoundError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9 or (self.uuid and self.uuid not in parts[0]):
                continue
            try:
                sm.append(float(parts[1].split()[0]))
                mx.append(float(parts[2].split()[0]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------- CPU oracle
def oracle_sample_problem(p, sample, state_blocks):
    """A compact problem holding only the sampled windows (their 16 blocks each)."""
    S = sample.size
    first = (p.positions[sample] - 127) // 8
    bt = np.zeros((S, p.block_table.shape[1]), np.int32)
    for i in range(S):
        bt[i, first[i]:first[i] + 16] = np.arange(16 * i, 16 * i + 16)
    return inputs.Problem("sample", np.arange(S, dtype=np.int32), p.positions[sample].copy(),
                          p.slot_mapping[sample].copy(), bt, state_blocks, p.rms_w, p.eps, p.cos_sin,
                          p.k_cache.copy(), p.kv_slot_mapping[sample].copy(), p.kv_block_size)


def time_oracle(sub, threads: int, min_cpu_s: float = 10.0, max_wall_s: float = 60.0):
    import oracle
    oracle.build()
    S = sub.num_tokens
    windows, wall, passes = 0, 0.0, 0
    cpu0 = time.process_time()
    t0 = time.perf_counter()
    while True:
        kc = sub.k_cache.copy()
        oracle.forward(sub, k_cache=kc, threads=threads)
        windows += S
        passes += 1
        wall = time.perf_counter() - t0
        if time.process_time() - cpu0 >= min_cpu_s or wall >= max_wall_s:
            break
    return windows / wall, passes, time.process_time() - cpu0


def gather_blocks_to_host(p, state_dev, sample):
    import torch
    first = (p.positions[sample] - 127) // 8
    blk = np.stack([p.block_table[int(t), first[i]:first[i] + 16] for i, t in enumerate(sample)]).reshape(-1)
    idx = torch.from_numpy(blk.astype(np.int64)).to(state_dev.device)
    return state_dev.index_select(0, idx).cpu().numpy()


# --------------------------------------------------------------------------------- our arm
def run_ours(args, ws, rank, local):
    import torch
    from deepseek_v4_sparse_c128_gb300 import binding, build

    torch.cuda.set_device(local)
    build.build()
    binding.load()
    dev = torch.device("cuda", local)
    T = args.tokens
    p = inputs.make_problem("sweep", seed=inputs.CONFIG_SEEDS["sweep"] + 7919 * rank, tokens=T, state_device=str(dev))
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    d = {k: to(getattr(p, k)) for k in ("token_to_req", "positions", "slot_mapping", "block_table", "rms_w",
                                        "cos_sin", "k_cache", "kv_slot_mapping")}
    d["state"] = p.state
    stream = torch.cuda.current_stream()

    step = binding.PreparedCall(d["token_to_req"], d["positions"], d["slot_mapping"], d["block_table"], d["state"],
                                d["rms_w"], p.eps, d["cos_sin"], d["k_cache"], d["kv_slot_mapping"], p.kv_block_size,
                                stream=stream)
    binding.reserve_workspace(T)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert binding.device_errors(clear=True) == 0, "device error during warm-up"
    uuid = str(getattr(torch.cuda.get_device_properties(dev), "uuid", "") or "")
    uuid = uuid if uuid.startswith("GPU-") or not uuid else "GPU-" + uuid
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(uuid) as clocks:
        barrier(ws)
        torch.cuda.synchronize()
        # ten equal chunks of the timed steps, each between two events on the stream, for min/median
        chunk = args.steps // 10 if args.steps >= 10 else args.steps
        marks = []
        # the calls exactly as a caller makes them: no kernel timer, so the planning kernel and the
        # compress kernel overlap through programmatic dependent launch
        e0.record(stream)
        for i in range(args.steps):
            if i % chunk == 0 and len(marks) < args.steps // chunk:
                marks.append((i, torch.cuda.Event(enable_timing=True)))
                marks[-1][1].record(stream)
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
    local_ms = e0.elapsed_time(e1)
    ends = marks[1:] + [(args.steps, e1)]
    chunk_ms = [a.elapsed_time(b) / (j - i) for (i, a), (j, b) in zip(marks, ends)]
    assert binding.device_errors(clear=True) == 0, "device error in the timed region"
    max_ms, total_windows = reduce_max_sum(ws, local_ms, float(T * args.steps))
    value = total_windows / (max_ms / 1e3)
    ms_per_step = max_ms / args.steps
    # the compress kernel alone, in a separate pass after the timed region: the library's kernel
    # timer records events around it (which turns programmatic dependent launch off for these calls)
    timer_calls = max(3, min(args.steps, 200))
    with binding.KernelTimer() as ktimer:
        for _ in range(timer_calls):
            step()
        torch.cuda.synchronize()
    assert binding.device_errors(clear=True) == 0, "device error in the kernel-timer pass"
    kernel_ms = ktimer.total_ms / max(1, ktimer.launches)

    # ---- end to end through the public API: every step uploads its token metadata and block table
    # from pinned host memory and reads the k_cache back; copies run on a side stream, double
    # buffered, so step k+1's upload and step k's read-back overlap step k's kernels.
    e2e = None
    if not args.no_e2e:
        keys = ("token_to_req", "positions", "slot_mapping", "block_table", "kv_slot_mapping")
        host = {k: torch.from_numpy(np.ascontiguousarray(getattr(p, k))).pin_memory() for k in keys}
        bufs = [dict(d), {k: torch.empty_like(v) for k, v in d.items() if k != "state"}]
        bufs[1]["state"] = d["state"]
        for k in ("rms_w", "cos_sin"):
            bufs[1][k].copy_(d[k])
        bufs[1]["k_cache"].copy_(d["k_cache"])
        kc_host = [torch.empty(d["k_cache"].shape, dtype=torch.uint8).pin_memory() for _ in range(2)]
        up_stream, down_stream = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        calls = [binding.PreparedCall(b["token_to_req"], b["positions"], b["slot_mapping"], b["block_table"],
                                      b["state"], b["rms_w"], p.eps, b["cos_sin"], b["k_cache"], b["kv_slot_mapping"],
                                      p.kv_block_size, stream=stream) for b in bufs]
        h2d = sum(int(v.numel() * v.element_size()) for v in host.values())
        d2h = int(kc_host[0].numel())
        uploaded = [torch.cuda.Event() for _ in range(2)]
        computed = [torch.cuda.Event() for _ in range(2)]
        read_back = [torch.cuda.Event() for _ in range(2)]

        def upload(i):
            j = i & 1
            with torch.cuda.stream(up_stream):
                if i >= 2:
                    up_stream.wait_event(computed[j])           # metadata buffer j free again
                for k in keys:
                    bufs[j][k].copy_(host[k], non_blocking=True)
                uploaded[j].record(up_stream)

        def run_e2e(n):
            upload(0)
            for i in range(n):
                j = i & 1
                if i + 1 < n:
                    upload(i + 1)                               # next step's inputs stream in meanwhile
                stream.wait_event(uploaded[j])
                if i >= 2:
                    stream.wait_event(read_back[j])             # k_cache j read back before reuse
                calls[j]()
                computed[j].record(stream)
                with torch.cuda.stream(down_stream):
                    down_stream.wait_event(computed[j])
                    kc_host[j].copy_(bufs[j]["k_cache"], non_blocking=True)
                    read_back[j].record(down_stream)
            torch.cuda.synchronize()

        e2e_steps = max(3, min(args.steps, 200))
        binding.reserve_workspace(T, stream)
        run_e2e(3)
        barrier(ws)
        t0 = time.perf_counter()
        run_e2e(e2e_steps)
        e2e_s = time.perf_counter() - t0
        barrier(ws)
        e2e_max_ms, e2e_windows = reduce_max_sum(ws, e2e_s * 1e3, float(T * e2e_steps))
        e2e = {"value": e2e_windows / (e2e_max_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "note": "public API (binding.PreparedCall -> C-ABI) with host buffers: each step uploads token "
                       "metadata + block table from pinned memory and reads the whole k_cache back; copies on a "
                       "upload and read-back streams, double-buffered so both overlap the kernels; state cache resident (it is a cache)"}

    out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": value / (HEADLINE_T / (PAGES_US_16374 * 1e-6)) if T == HEADLINE_T else None,
           "dtype": "f32", "data": "synthetic (seeded: kv~N(0,1), score~N(0,2), rms_w=1+0.1N(0,1))",
           "config": workload_config(T, ws),
           "us_per_call": ms_per_step * 1e3,
           "us_per_call_chunks": {"chunks": len(chunk_ms), "min": min(chunk_ms) * 1e3,
                                  "median": statistics.median(chunk_ms) * 1e3, "max": max(chunk_ms) * 1e3},
           "hbm_gbs_per_gpu": T * ALGO_BYTES_PER_WINDOW / (ms_per_step * 1e-3) / 1e9,
           "gpu_launches": launches_per_call(T, torch.cuda.get_device_properties(dev).multi_processor_count) * args.steps}
    out["e2e"] = e2e
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    peak, peak_src = (float(peaks["hbm_gbs"]), "measured") if "hbm_gbs" in peaks else (6800.0, "fallback")
    achieved = T * ALGO_BYTES_PER_WINDOW / (kernel_ms * 1e-3) / 1e9
    out["roofline"] = {"bound": "hbm", "kernel": "compress_kernel", "achieved": achieved, "peak": peak,
                       "peak_source": peak_src, "unit": "GB/s", "frac": achieved / peak,
                       "traffic": traffic_per_launch(T), "kernel_us": kernel_ms * 1e3,
                       "kernel_us_from": f"library kernel timer (CUDA events on the stream around the compress "
                                         f"kernel), {ktimer.launches} calls after the timed region",
                       "algorithmic_bytes_per_launch": T * ALGO_BYTES_PER_WINDOW}
    out["clocks"] = clocks.summary()
    if not args.no_read_probe:
        probe = read_probe_rate(d["state"], stream)
        out["hbm_read_probe"] = probe
        out["roofline"]["read_probe_gbs"] = probe["gbs"]
        out["roofline"]["frac_of_read_probe"] = achieved / probe["gbs"]

    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        rng = np.random.default_rng(11)
        sample = np.sort(rng.choice(T, size=min(T, 1024), replace=False))
        sub = oracle_sample_problem(p, sample, gather_blocks_to_host(p, p.state, sample))
        threads = os.cpu_count() or 1
        wps, passes, cpu_s = time_oracle(sub, threads)
        # the same oracle on one thread, over the first 128 sampled windows (a few seconds)
        sub1 = oracle_sample_problem(p, sample[:128], sub.state[:16 * 128])
        wps1, passes1, _ = time_oracle(sub1, 1, min_cpu_s=3.0, max_wall_s=20.0)
        out["cpu_baseline"] = {"value": wps, "unit": UNIT, "cores": threads, "kind": "oracle",
                               "sample": f"{sample.size} random windows of sweep{T} x {passes} passes "
                                         f"({cpu_s:.1f} s CPU), oracle over host threads",
                               "single_thread": {"value": wps1, "unit": UNIT, "cores": 1,
                                                 "sample": f"128 of those windows x {passes1} passes"}}
    if not args.no_workloads and ws == 1:
        out["workloads"] = bench_workloads(args, dev, peak, out.get("hbm_read_probe", {}).get("gbs"))
    if not args.no_next and ws == 1:
        out["other_configurations"] = bench_next(args, dev)
    if not args.no_sweep and ws == 1:
        del d, p
        torch.cuda.empty_cache()
        out["sweep_us_per_call"] = sweep(args, dev)
    if rank == 0:
        print(json.dumps(out), flush=True)


READ_PROBE_SHAPES = ((1024, 1, 8), (512, 2, 8), (512, 2, 4), (256, 4, 8), (1024, 2, 4), (512, 4, 4))


def read_probe_rate(buf, stream, launches: int = 10) -> dict:
    """DRAM read rate of a plain streaming read (c128_read_probe) over the whole buffer ``buf``
    (larger than L2), best over a few launch shapes; CUDA events on ``stream``."""
    import torch
    from deepseek_v4_sparse_c128_gb300 import binding
    word = torch.zeros(1, dtype=torch.int32, device=buf.device)
    nbytes = buf.numel() * buf.element_size()
    rates = {}
    for threads, ctas, loads in READ_PROBE_SHAPES:
        for _ in range(2):
            binding.read_probe(buf, word, threads, ctas, loads, stream=stream)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(launches):
            binding.read_probe(buf, word, threads, ctas, loads, stream=stream)
        b.record(stream)
        b.synchronize()
        rates[f"{threads}x{ctas}x{loads}"] = nbytes * launches / (a.elapsed_time(b) * 1e-3) / 1e9
    best = max(rates, key=rates.get)
    t, c, l = (int(x) for x in best.split("x"))
    return {"gbs": rates[best], "unit": "GB/s", "bytes": nbytes,
            "shape": {"threads_per_cta": t, "ctas_per_sm": c, "loads_in_flight": l},
            "all_shapes_gbs": {k: round(v, 1) for k, v in rates.items()},
            "how": f"c128_read_probe: one pass of 16-byte streaming loads over the {nbytes / 1e9:.2f} GB state "
                   f"buffer (> L2) per launch, {launches} launches per shape (threads per CTA x CTAs per SM x "
                   f"loads in flight per thread) after 2 warm-ups, CUDA events, best shape; right after the "
                   f"timed region"}


def launches_per_call(T: int, sm_count: int) -> int:
    """Kernels one C128 call launches: the cluster-split kernel for T x S <= #SM (S >= 1), the
    one-CTA-per-token kernel up to 8 tokens per SM, else the planning kernel and the compress kernel."""
    return 1 if T <= 8 * sm_count else 2


def sources_sha256(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def current_traffic_record(rec):
    """The record if the kernel sources it lists are unchanged since its ncu capture, else None."""
    try:
        return rec if rec.get("kernel_source_sha256") == sources_sha256(rec["kernel_sources"]) else None
    except (OSError, KeyError, TypeError):
        return None


def traffic_per_launch(T: int):
    """DRAM bytes per launch from the committed ncu capture, scaled by windows, or None when the
    kernel's sources changed since the capture."""
    try:
        rec = current_traffic_record(json.load(open(TRAFFIC_FILE)))
    except (OSError, ValueError):
        return None
    return None if rec is None else rec["dram_bytes_per_window"] * T


def sweep(args, dev):
    """µs per call vs token_num. Before every timed call a 512 MB buffer is written (L2 flush); the
    flush, the events and the call are enqueued back to back and synchronised once per size, so
    host launch time hides behind the flush. Columns: eager calls, CUDA-graph replays of the same
    call, the pages' method (four input sets in rotation, back to back, no flush), a cold
    rotation (enough state sets that four times L2 separates two uses of one set, no flush), and
    L2-hot (one input set, back to back, no flush: what fits in L2 is read from it)."""
    import torch
    from deepseek_v4_sparse_c128_gb300 import binding
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 129 * 1024 * 1024))
    eager, graph, rot4, cold, hot = {}, {}, {}, {}, {}
    for T in inputs.SWEEP_TOKENS:
        p = inputs.make_problem("sweep", tokens=T, state_device=str(dev))
        to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        d = {k: to(getattr(p, k)) for k in ("token_to_req", "positions", "slot_mapping", "block_table", "rms_w",
                                            "cos_sin", "k_cache", "kv_slot_mapping")}
        s = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(s):
            binding.reserve_workspace(T)
            call = binding.PreparedCall(d["token_to_req"], d["positions"], d["slot_mapping"], d["block_table"],
                                        p.state, d["rms_w"], p.eps, d["cos_sin"], d["k_cache"], d["kv_slot_mapping"],
                                        p.kv_block_size, stream=s)
            for _ in range(args.sweep_warmup):
                call()
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                call()
            n = args.sweep_calls
            # L2-hot: the same call back to back, no flush
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            for _ in range(n):
                call()
            b.record(s)
            s.synchronize()
            hot[str(T)] = round(a.elapsed_time(b) * 1e3 / n, 3)
            # the pages' method (PR #44230, Performance: bench_inputs=4): four input sets used in
            # rotation, no flush in between, so small sizes partly hit L2
            sets = [call]
            for k in range(1, 4):
                dk = dict(d)
                dk["k_cache"] = d["k_cache"].clone()
                st_k = inputs.draw_state(1000 + k, p.state.shape[0], str(dev))
                sets.append(binding.PreparedCall(dk["token_to_req"], dk["positions"], dk["slot_mapping"],
                                                 dk["block_table"], st_k, dk["rms_w"], p.eps, dk["cos_sin"],
                                                 dk["k_cache"], dk["kv_slot_mapping"], p.kv_block_size, stream=s))
            for i in range(max(4, args.sweep_warmup)):
                sets[i % 4]()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            for i in range(n):
                sets[i % 4]()
            b.record(s)
            s.synchronize()
            rot4[str(T)] = round(a.elapsed_time(b) * 1e3 / n, 3)
            del sets
            # cold rotation: R = max(4, ceil(4 L2 / state bytes per call)) state sets cycled, no flush,
            # so every call reads state that is not in L2 and nothing dirty is left to write back
            nb = p.state.shape[0]
            R = max(4, min(1024, -(-4 * l2 // (nb * p.state.shape[1] * p.state.shape[2] * 4))))
            if R == 4:
                cold[str(T)] = rot4[str(T)]
            else:
                big = inputs.draw_state(3000 + T, R * nb, str(dev))
                sets = [binding.PreparedCall(d["token_to_req"], d["positions"], d["slot_mapping"], d["block_table"],
                                             big[k * nb:(k + 1) * nb], d["rms_w"], p.eps, d["cos_sin"], d["k_cache"],
                                             d["kv_slot_mapping"], p.kv_block_size, stream=s) for k in range(R)]
                for i in range(max(R, args.sweep_warmup)):
                    sets[i % R]()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(s)
                for i in range(n):
                    sets[i % R]()
                b.record(s)
                s.synchronize()
                cold[str(T)] = round(a.elapsed_time(b) * 1e3 / n, 3)
                del sets, big
            for mode, fn in (("eager", call), ("graph", g.replay)):
                evs = []
                for _ in range(n):
                    flush.fill_(1.0)
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(s)
                    fn()
                    b.record(s)
                    evs.append((a, b))
                s.synchronize()
                us = statistics.mean(a.elapsed_time(b) * 1e3 for a, b in evs)
                (eager if mode == "eager" else graph)[str(T)] = round(us, 3)
            assert binding.device_errors(s, clear=True) == 0
        del d, p, g, call
    return {"eager": eager, "graph": graph, "rotate4_no_flush": rot4, "rotate_cold_no_flush": cold,
            "l2_hot_same_inputs": hot,
            "timing": f"{args.sweep_warmup} warm-up calls, then {args.sweep_calls} timed calls per column and "
                      f"token_num (mean; CUDA events around the timed calls, or around each call in the flush "
                      f"columns)"}


def next_algorithmic_bytes(p, pos):
    """Bytes a window at each position in `pos` must move: the kv and score half-rows of its
    unmasked rows (rows at negative positions are masked), one 4-byte block id per distinct state
    block, the 64 fp32 cos/sin values and the cache slot."""
    n = (1 + p.overlap) * p.ratio
    rows = np.minimum(n, pos + 1)
    first = np.maximum(pos - n + 1, 0)
    sb = int(p.state.shape[1])
    blocks = pos // sb - first // sb + 1
    slot = {0: 584, 1: 132, 2: 68}[p.fmt]
    return int((rows * 2 * p.head * 4 + blocks * 4 + 256 + slot).sum())


def bench_next(args, dev):
    """The other configurations of the pages' fused kernels through compress_norm_rope_store_ex
    (C4 overlap with the sparse-attention cache; the head-128 indexer with FP8 or MXFP4 caches at
    ratios 4 and 128), each on a prefill batch with about a quarter million tokens whose state is
    larger than L2: µs per call, windows/s, and the gather kernel's algorithmic GB/s."""
    import torch
    from deepseek_v4_sparse_c128_gb300 import binding
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    peak = float(peaks.get("hbm_gbs", 6800.0))
    try:
        traffic = json.load(open(OTHER_TRAFFIC_FILE))
    except (OSError, ValueError):
        traffic = {}
    res = {}
    for name, scale in NEXT_SCALES.items():
        p = inputs.make_next_problem(name, state_device=str(dev), scale=scale)
        to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        d = {k: to(getattr(p, k)) for k in ("token_to_req", "positions", "slot_mapping", "block_table", "rms_w",
                                            "cos_sin", "k_cache", "kv_slot_mapping")}
        cfg = binding.config(p.head, p.ratio, p.overlap, p.state_width, p.fmt)
        stream = torch.cuda.current_stream()
        call = binding.PreparedCall(d["token_to_req"], d["positions"], d["slot_mapping"], d["block_table"], p.state,
                                    d["rms_w"], p.eps, d["cos_sin"], d["k_cache"], d["kv_slot_mapping"],
                                    p.kv_block_size, stream=stream, cfg=cfg)
        binding.reserve_workspace(p.num_tokens)
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        n = 20
        # call time as a caller sees it (the planning kernel overlapped by PDL), then the compress
        # kernel alone from the library's timer (events around it, which turn PDL off)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            call()
        b.record(stream)
        torch.cuda.synchronize()
        with binding.KernelTimer() as kt:
            for _ in range(n):
                call()
            torch.cuda.synchronize()
        assert binding.device_errors(clear=True) == 0
        active = (p.positions >= 0) & ((p.positions + 1) % p.ratio == 0)   # every token here has a slot
        A = int(active.sum())
        total_bytes = next_algorithmic_bytes(p, p.positions[active])
        per_window = total_bytes / max(A, 1)
        kus = kt.total_ms * 1e3 / kt.launches
        achieved = total_bytes / (kus * 1e-6) / 1e9
        res[name] = {"tokens": p.num_tokens, "windows": A, "us_per_call": round(a.elapsed_time(b) * 1e3 / n, 2),
                     "windows_per_s": A / (a.elapsed_time(b) / n * 1e-3), "kernel_us": round(kus, 2),
                     "algorithmic_bytes_per_window": round(per_window, 1), "achieved_gbs": round(achieved, 1),
                     "frac_of_measured_hbm": round(achieved / peak, 3)}
        rec = current_traffic_record(traffic.get(name)) if isinstance(traffic.get(name), dict) else None
        res[name]["ncu_dram_bytes_per_window"] = None if rec is None else rec["dram_bytes_per_window"]
        del d, p, call
        torch.cuda.empty_cache()
    return res


WORKLOADS = ("tiny", "decode", "mixed", "varlen", "varlen16k")
META_BYTES_PER_TOKEN = 4 + 8 + 8 + 8   # token_to_req (int32), positions, slot_mapping, kv_slot_mapping (int64)


def active_windows(p) -> np.ndarray:
    """Tokens that store a window: slot >= 0, position >= 0 at a window end, kv slot >= 0."""
    return ((p.slot_mapping >= 0) & (p.positions >= 0) & ((p.positions + 1) % inputs.RATIO == 0)
            & (p.kv_slot_mapping >= 0))


def workload_bytes(p) -> int:
    """Algorithmic bytes of one call: 525,192 per active window (its 128 state rows, 16 block ids,
    the cos/sin row and the 584-byte slot) + 28 per token of metadata + the 2 KiB RMSNorm weight."""
    return int(active_windows(p).sum()) * ALGO_BYTES_PER_WINDOW + META_BYTES_PER_TOKEN * p.num_tokens + 4 * 512


def bench_workloads(args, dev, peak: float, probe_gbs):
    """The five synthetic workloads (tiny, decode, mixed, varlen, varlen16k) through the public call:
    µs per call (mean of the timed calls, and min / median over ten chunks of them), compressed
    windows/s, algorithmic GB/s and its fraction of the measured copy bandwidth and of the read
    probe, in two columns: cold (R state sets in rotation, R x state bytes >= 4 x L2, so no call
    finds its state in L2) and L2-hot (one input set back to back). Beside them, the CPU oracle
    over all host threads on the same workload (state copied to the host)."""
    import dataclasses
    import torch
    from deepseek_v4_sparse_c128_gb300 import binding
    import oracle
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 129 * 1024 * 1024))
    threads = os.cpu_count() or 1
    oracle.build()
    res = {}
    for name in WORKLOADS:
        p = inputs.make_problem(name, state_device=str(dev))
        to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        d = {k: to(getattr(p, k)) for k in ("token_to_req", "positions", "slot_mapping", "block_table", "rms_w",
                                            "cos_sin", "k_cache", "kv_slot_mapping")}
        A = int(active_windows(p).sum())
        nbytes = workload_bytes(p)
        state_bytes = p.state.numel() * 4
        R = max(1, -(-4 * l2 // state_bytes))
        states = [p.state] + [inputs.draw_state(7000 + 31 * k + inputs.CONFIG_SEEDS[name], p.state.shape[0], str(dev))
                              for k in range(1, R)]
        s = torch.cuda.Stream(device=dev)
        binding.reserve_workspace(p.num_tokens, s)
        calls = [binding.PreparedCall(d["token_to_req"], d["positions"], d["slot_mapping"], d["block_table"], st,
                                      d["rms_w"], p.eps, d["cos_sin"], d["k_cache"], d["kv_slot_mapping"],
                                      p.kv_block_size, stream=s) for st in states]
        n = args.workload_calls
        row = {"tokens": p.num_tokens, "windows": A, "algorithmic_bytes_per_call": nbytes,
               "state_sets": R, "state_bytes_per_set": state_bytes}
        for col, rot in (("cold", len(calls)), ("l2_hot", 1)):
            for i in range(max(50, rot)):
                calls[i % rot]()
            chunk = max(1, n // 10)
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(n // chunk + 1)]
            evs[0].record(s)
            for i in range(n // chunk * chunk):
                calls[i % rot]()
                if (i + 1) % chunk == 0:
                    evs[(i + 1) // chunk].record(s)
            s.synchronize()
            per = [evs[k].elapsed_time(evs[k + 1]) * 1e3 / chunk for k in range(len(evs) - 1)]
            us = evs[0].elapsed_time(evs[-1]) * 1e3 / (chunk * len(per))
            gbs = nbytes / (us * 1e-6) / 1e9
            row[col] = {"us_per_call": round(us, 3), "us_min_chunk": round(min(per), 3),
                        "us_median_chunk": round(statistics.median(per), 3), "calls": chunk * len(per),
                        "windows_per_s": A / (us * 1e-6), "algorithmic_gbs": round(gbs, 1),
                        "frac_of_measured_hbm": round(gbs / peak, 3),
                        "frac_of_read_probe": round(gbs / probe_gbs, 3) if probe_gbs else None}
        assert binding.device_errors(s, clear=True) == 0, f"device error in workload {name}"
        # the CPU oracle on the same workload (the first state set, copied to the host)
        if not args.no_cpu_baseline:
            host = dataclasses.replace(p, state=p.state.cpu().numpy())
            passes, t0 = 0, time.perf_counter()
            while True:
                oracle.forward(host, k_cache=p.k_cache.copy(), threads=threads)
                passes += 1
                if time.perf_counter() - t0 > 1.0 or passes >= 20:
                    break
            wall = time.perf_counter() - t0
            row["oracle"] = {"windows_per_s": A * passes / wall, "cores": threads, "passes": passes,
                             "kind": "oracle", "sample": "the whole workload"}
            del host
        res[name] = row
        s.synchronize()
        binding.release_stream(s)
        del calls, states, d, p
        torch.cuda.empty_cache()
    return res


# --------------------------------------------------------------------------- reference arm
def run_reference(args, ws, rank):
    """The CPU oracle as it stands, on the host cores, over a bounded sample of the same workload."""
    if rank != 0:
        return
    T = args.tokens
    # metadata of the full workload; the state is drawn only for the sampled windows' blocks
    p = inputs.make_problem("sweep", tokens=T, state_device="none")
    rng = np.random.default_rng(12)
    S = min(T, 256)
    sample = np.sort(rng.choice(T, size=S, replace=False))
    st = inputs.draw_state(99, 16 * S, "cpu")
    sub = oracle_sample_problem(p, sample, st)
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    for _ in range(args.warmup):
        oracle.forward(sub, k_cache=sub.k_cache.copy(), threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.forward(sub, k_cache=sub.k_cache.copy(), threads=threads)
    wall = time.perf_counter() - t0
    value = S * args.steps / wall
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": wall * 1e3 / args.steps, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
           "config": workload_config(T, ws),
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                            "sample": f"each step: {S} random windows of sweep{T} (state of their 16 blocks "
                                      f"each), oracle over {threads} host threads"},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


NEXT_SCALES = {"c4_sparse": 64, "idx_c4_fp8": 64, "idx_c4_mxfp4": 64, "idx_c128_fp8": 16, "idx_c128_mxfp4": 16}


def run_case(args):
    """One workload alone, `--warmup` + `--steps` calls on one stream with nothing else around
    them (the command the ncu summaries under profiles/ are taken with): `sweep` (the headline
    layout at --tokens) or one of the other configurations at its bench size."""
    import torch
    from deepseek_v4_sparse_c128_gb300 import binding, build
    build.build()
    binding.load()
    dev = torch.device("cuda", 0)
    if args.case == "read_probe":
        # the read probe alone over a 1 GiB buffer (8x L2), in the shape that led the bench's sweep
        buf = torch.randint(-2**31, 2**31 - 1, (1 << 28,), dtype=torch.int32, device=dev)
        word = torch.zeros(1, dtype=torch.int32, device=dev)
        stream = torch.cuda.current_stream()
        run = lambda: binding.read_probe(buf, word, 512, 4, 4, stream=stream)
        for _ in range(args.warmup):
            run()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            run()
        b.record(stream)
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / max(args.steps, 1)
        print(json.dumps({"case": args.case, "bytes": buf.numel() * 4, "calls": args.steps, "us_per_call": us,
                          "gbs": buf.numel() * 4 / (us * 1e-6) / 1e9, "device_errors": 0}), flush=True)
        return
    if args.case == "sweep":
        p = inputs.make_problem("sweep", tokens=args.tokens, state_device=str(dev))
        cfg = None
    else:
        p = inputs.make_next_problem(args.case, state_device=str(dev), scale=args.scale or NEXT_SCALES[args.case])
        cfg = binding.config(p.head, p.ratio, p.overlap, p.state_width, p.fmt)
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    d = {k: to(getattr(p, k)) for k in ("token_to_req", "positions", "slot_mapping", "block_table", "rms_w",
                                        "cos_sin", "k_cache", "kv_slot_mapping")}
    stream = torch.cuda.current_stream()
    call = binding.PreparedCall(d["token_to_req"], d["positions"], d["slot_mapping"], d["block_table"], p.state,
                                d["rms_w"], p.eps, d["cos_sin"], d["k_cache"], d["kv_slot_mapping"], p.kv_block_size,
                                stream=stream, cfg=cfg)
    binding.reserve_workspace(p.num_tokens)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(args.warmup):
        call()
    a.record(stream)
    for _ in range(args.steps):
        call()
    b.record(stream)
    torch.cuda.synchronize()
    errs = binding.device_errors(clear=True)
    us = a.elapsed_time(b) * 1e3 / max(args.steps, 1)
    out = {"case": args.case, "tokens": p.num_tokens, "calls": args.steps, "us_per_call": us, "device_errors": errs}
    if args.case != "sweep":
        active = (p.positions >= 0) & ((p.positions + 1) % p.ratio == 0)   # every token here has a slot
        out.update(windows=int(active.sum()),
                   algorithmic_gbs=round(next_algorithmic_bytes(p, p.positions[active]) / (us * 1e-6) / 1e9, 1))
    print(json.dumps(out), flush=True)
    if errs:
        raise SystemExit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--tokens", type=int, default=HEADLINE_T)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-next", action="store_true")
    ap.add_argument("--no-read-probe", action="store_true")
    ap.add_argument("--no-workloads", action="store_true")
    ap.add_argument("--sweep-warmup", type=int, default=50, help="warm-up calls per token_num of the sweep")
    ap.add_argument("--sweep-calls", type=int, default=1000, help="timed calls per token_num and column")
    ap.add_argument("--workload-calls", type=int, default=1000,
                    help="timed calls per workload in the five-workload table")
    ap.add_argument("--scale", type=int, default=None,
                    help="with --case and another configuration: request-count scale (default: the bench size)")
    ap.add_argument("--case", choices=["sweep", "read_probe"] + list(NEXT_SCALES),
                    help="run one workload alone (no JSON bench line); used for profiling")
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return
    ws, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, ws, rank)
        else:
            run_ours(args, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
