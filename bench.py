"""Benchmark of the KV relocation + rank-m patch path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config I] [--impl ours|reference]

One step = one pass of the whole operator over one workload: every chunk,
every layer, K and V (one relocation kernel launch through the C ABI, preceded
for a batch by the small copy launches that carry its plan).  The default
workload is the largest: the sliding-window survival + recall batch of a
Qwen2.5-VL-7B-shaped model (28 layers, 4 KV heads x 128; 8 requests x 32
chunks x 1024 tokens, 224 chunks moved by R(delta) alone and 32 recalled with
rank-64 patches; 16-token pages through shuffled block tables; one
kv_relocate_batch launch).  --config picks another of the measured workloads
(1: the single-chunk Qwen2.5-VL-shaped GQA video segment).

Prints one JSON line: tokens/s (chunk tokens per second, all layers, K and V),
the dominant kernel's roofline (algorithmic bytes / mean launch time against
the measured HBM copy bandwidth), a parity block on what the timed launches
wrote (whole-output placement and byte-copy checks on the device, and sampled
rows against the fp64 oracle), an end-to-end figure through the C ABI with
host buffers (inputs copied in and results copied out every step), the fp64
oracle timed on the host cores (one core and all cores), and the SM clocks
sampled during the timed region.  Under torchrun each rank runs its own replica of the workload (the
path shards into independent chunks; there is no exchange step): weak scaling.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "relocated+patched KV tokens/s and HBM GB/s (fraction of GB300 roofline), 1 GPU"
KERNEL_SOURCES = ["position_invariant_kv_gb300/csrc/kvrp_kernel.cu", "position_invariant_kv_gb300/csrc/kvrp_plan.h",
                  "position_invariant_kv_gb300/csrc/kvrp_host.cpp", "position_invariant_kv_gb300/csrc/kvrp_ptx.h"]
L2_BYTES = 129 * 2 ** 20


def kernel_hash(sources=None) -> str:
    h = hashlib.sha256()
    for p in sources or KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, p), "rb").read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


ATTEND_SOURCES = ["position_invariant_kv_gb300/csrc/kvrp_attend.cu", "position_invariant_kv_gb300/csrc/kvrp_ptx.h"]


def profiled_traffic(workload: str, summary: str = "relocate_kernel_dram.json", sources=None):
    """DRAM bytes per launch from the committed ncu summary of a kernel, if it
    was taken on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("kernel_hash") != kernel_hash(sources):
        return None
    ent = d.get("per_launch", {}).get(workload)
    return None if ent is None else ent.get("dram_bytes")


def workload_text(wl) -> str:
    chunks = len(wl.chunks)
    ranks = sorted({c.rank for c in wl.chunks})
    dst = "paged 16-token pages via shuffled block table" if wl.paged else "contiguous"
    if wl.family == "mla":
        shape = f"MLA rows {wl.kv_lora_dim}+{wl.rope_dim}"
    else:
        shape = f"{wl.n_heads} KV heads x {wl.head_dim}"
    return (f"{wl.name}: {wl.n_layers} layers, {shape}, {chunks} chunk(s), {wl.n_chunk_tokens} tokens, "
            f"rank {'/'.join(map(str, ranks))}, theta {wl.theta:g}, {dst}")


# --------------------------------------------------------------------------- #
# clocks sampled during the timed region
# --------------------------------------------------------------------------- #
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except FileNotFoundError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        mhz, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        mhz.sort()
        return {"sm_mhz": mhz[len(mhz) // 2] if mhz else None, "sm_max_mhz": mx, "samples": len(mhz),
                "reasons": sorted(reasons)}


# --------------------------------------------------------------------------- #
# CPU baseline: the fp64 oracle on a bounded sample, in a fresh process
# --------------------------------------------------------------------------- #
class OracleSampler:
    """The fp64 oracle, as it stands, on token rows of one layer of the
    workload: one representative chunk of each distinct rank (c4: a surviving
    chunk at rank 0 and a recalled one at rank 64), each evaluated in
    proportion to the workload's tokens of that kind.  A step over n rows of
    one (layer, tensor) slice stands for n / (layers x tensors) chunk tokens."""

    def __init__(self, cfg: int, seed_offset: int = 0):
        import workloads as W
        from oracle import operator_rows, round_to_bf16_bits, row_layout
        self._op, self._round = operator_rows, round_to_bf16_bits
        wl = W.config(cfg)
        self.wl = wl
        kinds = {}
        for c in wl.chunks:
            kinds.setdefault(c.rank, [c, 0])[1] += c.n_tokens
        chunks, row = [], 0
        for c, _ in kinds.values():
            chunks.append(W.Chunk(row, c.n_tokens, c.delta, c.rank, 0, row))
            row += c.n_tokens
        total = sum(t for _, t in kinds.values())
        self.share = [t / total for _, t in kinds.values()]
        self.slice_wl = W.Workload(wl.name, wl.family, 1, wl.n_heads, wl.head_dim, wl.kv_lora_dim, wl.rope_dim,
                                   wl.theta, row, (row + W.PAGE - 1) // W.PAGE, False, chunks, None,
                                   wl.seed + seed_offset, "numpy", mrope_sections=wl.mrope_sections)
        self.host = W.host_inputs(self.slice_wl)
        self.layouts = {n: row_layout(wl.family, n, n_heads=wl.n_heads, head_dim=wl.head_dim,
                                      kv_lora_dim=wl.kv_lora_dim, rope_dim=wl.rope_dim) for n in wl.tensors}
        self.layer_tensors = wl.n_layers * len(wl.tensors)
        self.n_tokens = max(c.n_tokens for c in chunks)
        self.kinds = "; ".join(f"{share:.1%} of rows at rank {c.rank}" for c, share in zip(chunks, self.share))
        self.i = 0

    def step(self, n_rows: int):
        """(seconds of oracle time, rows evaluated) for about n_rows rows, split
        over the chunk kinds by their share of the workload's tokens."""
        import numpy as np
        secs, done = 0.0, 0
        for ci, (c, share) in enumerate(zip(self.slice_wl.chunks, self.share)):
            n = max(1, int(round(n_rows * share)))
            toks = (self.i + np.arange(n)) % c.n_tokens
            name = self.wl.tensors[self.i % len(self.wl.tensors)]
            x = self.host["rows"][name][0, c.src_row0 + toks]
            u = self.host["u"][name][ci][0, toks] if c.rank else None
            w = self.host["w"][name][ci][0] if c.rank else None
            t0 = time.perf_counter()
            self._round(self._op(x, u, w, c.delta, self.wl.theta, self.layouts[name], self.wl.mrope_sections))
            secs += time.perf_counter() - t0
            done += n
        self.i += 1 + n_rows
        return secs, done

    def tokens(self, n_rows: int) -> float:
        return n_rows / self.layer_tensors


def _oracle_rate(cfg: int, seconds: float, seed_offset: int, barrier=None, out=None):
    """Rows/s of the oracle on one core for about `seconds` of wall time (after
    an optional start barrier shared with the other cores' processes)."""
    o = OracleSampler(cfg, seed_offset)
    if barrier is not None:
        barrier.wait()
    t0 = time.perf_counter()
    rows, busy = 0, 0.0
    while time.perf_counter() - t0 < seconds:
        s, n = o.step(o.n_tokens)
        busy += s
        rows += n
    wall = time.perf_counter() - t0
    res = (rows, wall, busy)
    if out is not None:
        out.put(res)
    return res


def cpu_baseline_worker(cfg: int, budget_s: float) -> dict:
    """The oracle on one host core, then on every host core at once (one
    process per core, started with spawn, all timed over the same window)."""
    import multiprocessing as mp
    o = OracleSampler(cfg)
    cores = os.cpu_count() or 1
    rows1, wall1, busy1 = _oracle_rate(cfg, budget_s / 2, 0)
    one = o.tokens(rows1) / busy1
    ctx = mp.get_context("spawn")
    barrier, q = ctx.Barrier(cores), ctx.Queue()
    procs = [ctx.Process(target=_oracle_rate, args=(cfg, budget_s / 2, 1 + i, barrier, q)) for i in range(cores)]
    for p in procs:
        p.start()
    res = [q.get(timeout=600) for _ in procs]
    for p in procs:
        p.join(timeout=60)
    rows_all = sum(r[0] for r in res)
    wall = max(r[1] for r in res)
    every = o.tokens(rows_all) / wall
    return {"value": every, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "single_core_value": one, "os_cpu_count": cores,
            "sample": f"fp64 NumPy oracle on rows of one layer of {o.wl.name} ({o.kinds}); one chunk token = "
                      f"{o.layer_tensors} such rows. value: {cores} processes, one per host core (os.cpu_count() = "
                      f"{cores}), one BLAS thread each, {rows_all} rows in {wall:.1f} s of wall time; "
                      f"single_core_value: one process, {rows1} rows in {busy1:.1f} s of oracle time"}


def parity_worker(path: str) -> dict:
    """The parity rule of the oracle on output rows sampled from the device
    (see collect_parity_sample): the report summed over every sampled row."""
    import pickle
    from oracle import conditioning, operator_rows, row_layout
    from oracle.compare import parity_report
    with open(path, "rb") as f:
        groups = pickle.load(f)
    total = {}
    for g in groups:
        lay = row_layout(g["family"], g["tensor"], n_heads=g["n_heads"], head_dim=g["head_dim"],
                         kv_lora_dim=g["kv_lora_dim"], rope_dim=g["rope_dim"])
        ref = operator_rows(g["x"], g["u"], g["w"], g["delta"], g["theta"], lay, g["sections"])
        cond = conditioning(g["x"], g["u"], g["w"], g["delta"], g["theta"], lay, g["sections"])
        r = parity_report(g["got"], ref, cond)
        for k, v in r.items():
            total[k] = max(total.get(k, 0), v) if k.startswith("max") else total.get(k, 0) + v
    total["rows"] = sum(len(g["got"]) for g in groups)
    return total


def _worker_env() -> dict:
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    return env


def run_cpu_baseline(cfg: int, budget_s: float, parity_path: str = None) -> dict:
    """Runs the CPU-baseline worker (and, given a sample file, the oracle's
    parity check of the bench's own output) in a fresh process without a GPU."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--cpu-baseline-worker", "--config", str(cfg),
           "--budget", str(budget_s)]
    if parity_path:
        cmd += ["--parity-sample", parity_path]
    res = subprocess.run(cmd, capture_output=True, text=True, env=_worker_env(), timeout=1200)
    if res.returncode != 0:
        tail = res.stderr.strip().splitlines()[-1] if res.stderr.strip() else "no output"
        return {"value": None, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": "failed: " + tail}
    return json.loads(res.stdout.strip().splitlines()[-1])


def collect_parity_sample(wl, dwl, path: str, n_groups: int = 512, per_group: int = 4, seed: int = 12345) -> int:
    """Copies to the host, for randomly chosen (chunk, tensor, layer) groups of
    a few tokens each, the inputs the oracle needs and the rows the device
    wrote into the destination pools, and pickles them to `path`.  Returns the
    number of rows.  No arithmetic of the operator happens here."""
    import pickle
    import numpy as np
    import torch
    rng = np.random.default_rng(seed)
    dev = dwl.pools[wl.tensors[0]].device

    def bits(t):
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

    groups = []
    for _ in range(n_groups):
        ci = int(rng.integers(len(wl.chunks)))
        c = wl.chunks[ci]
        name = wl.tensors[int(rng.integers(len(wl.tensors)))]
        layer = int(rng.integers(wl.n_layers))
        toks = np.unique(rng.integers(0, c.n_tokens, size=per_group))
        ti = torch.as_tensor(toks, device=dev)
        q = c.dst_start + toks
        page = wl.block_tables[c.seq][q // 16] if wl.paged else q // 16
        got = dwl.pools[name][layer, torch.as_tensor(page, device=dev), torch.as_tensor(q % 16, device=dev)]
        groups.append({
            "family": wl.family, "tensor": name, "n_heads": wl.n_heads, "head_dim": wl.head_dim,
            "kv_lora_dim": wl.kv_lora_dim, "rope_dim": wl.rope_dim, "delta": c.delta, "theta": wl.theta,
            "sections": wl.mrope_sections, "x": bits(dwl.rows[name][layer, c.src_row0 + ti]),
            "u": bits(dwl.u[name][ci][layer, ti]) if c.rank else None,
            "w": bits(dwl.w[name][ci][layer]) if c.rank else None, "got": bits(got)})
    with open(path, "wb") as f:
        pickle.dump(groups, f)
    return sum(len(g["got"]) for g in groups)


def device_properties(wl, dwl) -> dict:
    """Checks of the whole output that hold at any size, evaluated on the
    device one layer at a time: every slot no token targets keeps its sentinel
    (and every targeted slot was written), and the values of unpatched GQA/MHA
    chunks and the c_KV part of unpatched MLA rows are byte copies."""
    import torch
    import workloads as W
    untouched = sum(int((p[l].view(torch.int16) == -1).all(dim=-1).sum())
                    for p in dwl.pools.values() for l in range(wl.n_layers))
    want_untouched = len(wl.tensors) * wl.n_layers * (wl.num_pages * W.PAGE - wl.n_chunk_tokens)
    copies_ok, copied_rows = True, 0
    plain = [c for c in wl.chunks if c.rank == 0]
    if plain:
        name = "kv" if wl.family == "mla" else "v"
        cols = slice(0, wl.kv_lora_dim) if wl.family == "mla" else slice(None)
        dev = dwl.pools[name].device
        q = torch.cat([torch.arange(c.dst_start, c.dst_start + c.n_tokens) for c in plain]).to(dev)
        seq = torch.cat([torch.full((c.n_tokens,), c.seq) for c in plain]).to(dev)
        src = torch.cat([torch.arange(c.src_row0, c.src_row0 + c.n_tokens) for c in plain]).to(dev)
        page = dwl.block_tables.long()[seq, q // 16] if wl.paged else q // 16
        for l in range(wl.n_layers):
            out = dwl.pools[name][l, page, q % 16, cols]
            copies_ok &= bool(torch.equal(out.view(torch.int16), dwl.rows[name][l, src, cols].view(torch.int16)))
        copied_rows = int(q.numel()) * wl.n_layers
    return {"untouched_slots": untouched, "untouched_slots_expected": want_untouched,
            "placement_ok": untouched == want_untouched, "byte_copy_rows": copied_rows, "byte_copies_ok": copies_ok}


# --------------------------------------------------------------------------- #
# our arm
# --------------------------------------------------------------------------- #
def max_over_ranks(value: float, device) -> float:
    """The largest of each rank's value (the slowest rank's time); identity on one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, total_ms: float, steps: int) -> float:
    """Whole-job tokens/s: every rank moves its own replica each step, and the
    job's step time is the slowest rank's."""
    return tokens_per_rank * world / (total_ms / 1e3 / steps)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def bench_config(wl, world: int) -> dict:
    """The `config` object of the JSON line, the same for both arms."""
    nbytes = wl.algorithmic_bytes()
    return {"workload": workload_text(wl), "tokens_per_step": wl.n_chunk_tokens,
            "algorithmic_bytes_per_step": nbytes["total"],
            "l2": f"inputs larger than L2 ({nbytes['total'] / 1e6:.0f} MB moved per step vs 129 MB L2)"
            if nbytes["total"] > 2 * L2_BYTES else "L2-resident workload (smaller than L2)",
            "parallelism": f"replicas x{world}"}


def default_steps(wl, peak_gbs: float) -> int:
    """Launches that keep the timed region near ten seconds at ~90% of peak."""
    t = wl.algorithmic_bytes()["total"] / (0.9 * peak_gbs * 1e9)
    return int(min(20000, max(20, 10.0 / max(t, 1e-6))))


def bench_ours(args) -> dict:
    import tempfile
    import torch
    import harness
    import workloads as W
    import position_invariant_kv_gb300 as kvrp

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    from position_invariant_kv_gb300.build import build
    if rank == 0 or world == 1:
        build()
    if world > 1:
        torch.distributed.barrier()
    kvrp.lib()

    wl = W.config(args.config)
    if args.layers:
        wl.n_layers = min(wl.n_layers, args.layers)   # a smaller copy of the workload for profiler captures
    dwl = harness.DeviceWorkload(wl, f"cuda:{local}")
    stream = torch.cuda.current_stream()
    nbytes = wl.algorithmic_bytes()
    tokens = wl.n_chunk_tokens
    peaks = measured_peaks()
    steps = args.steps if args.steps else default_steps(wl, peaks["hbm_gbs"])
    args.steps = steps

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # One event pair brackets the timed region; the launches inside it run back
    # to back, as a caller's loop would issue them (an event recorded between two
    # launches would stop the next one's set-up from overlapping the previous one).
    # The warm-up launches run right before it, once the clock sampler is up, so
    # the GPU does not sit idle between them and the timed launches.
    with ClockSampler(local) as clocks:
        for _ in range(args.warmup):
            dwl.run(stream=stream)
        # the timed launches alone write the pools checked below
        dwl.reset_pools()
        dwl.status.zero_()
        barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(steps):
            dwl.run(stream=stream)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier()
    total_ms = t0.elapsed_time(t1)
    mean_launch_ms = total_ms / steps      # one step = the plan upload (batches) + relocate_kernel
    launches_per_step = kvrp.kvrp_last_launch_count()   # the library's count for the last timed call
    status = dwl.status_value()

    total_ms = max_over_ranks(total_ms, f"cuda:{local}")
    ms_per_step = total_ms / steps
    value = job_throughput(tokens, world, total_ms, steps)

    # parity of what the timed launches wrote: properties of the whole output on
    # the device, and sampled rows for the oracle (checked in the CPU-baseline
    # process, the only place this script runs the oracle)
    props = device_properties(wl, dwl)
    parity_path = None
    if rank == 0 and not args.no_cpu_baseline:
        parity_path = os.path.join(tempfile.mkdtemp(prefix="kvrp_parity_"), "sample.pkl")
        n_rows = collect_parity_sample(wl, dwl, parity_path)

    # end to end through the C ABI with host buffers: copy the step's inputs in
    # from pinned memory, run, copy the destination pools out, every step
    # (--e2e-steps 0 leaves it out: profiler captures only)
    e2e = bench_e2e_bounded(dwl, wl, args, stream, f"cuda:{local}") if args.e2e_steps > 0 else None

    achieved = nbytes["total"] / (mean_launch_ms / 1e3) / 1e9
    traffic = profiled_traffic(wl.name)
    out = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": bench_config(wl, world),
        "hbm_gbs": nbytes["total"] / (ms_per_step / 1e3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "kernel": "relocate_kernel", "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)"
                     if peaks["source"] == "measured" else "fallback 6.8 TB/s",
                     "mean_launch_us": mean_launch_ms * 1e3,
                     "launch_timing": "CUDA events around the whole timed region / steps (a step of a batch "
                                      "also holds its plan-upload copy kernels)"},
        "e2e": e2e,
        "gpu_launches": steps * launches_per_step,
        "clocks": clocks.summary(),
        "device_status": status,
        "patch_tflops": wl.patch_flops() / (mean_launch_ms / 1e3) / 1e12,
    }
    if rank == 0 and not args.no_cpu_baseline:
        cb = run_cpu_baseline(args.config, args.budget, parity_path)
        par = cb.pop("parity", None)
        out["cpu_baseline"] = cb
        out["parity"] = dict(par or {"error": "parity check did not run"}, **props,
                             of="the destination pools as the last timed launch left them (reset to a "
                                "sentinel before the timed region)",
                             rule="within 1 bf16 ulp of the fp64 oracle rounded once; a mismatch (> 1 ulp) "
                                  "must stay within ulp(ref) + 2^-20 x the conditioning sum, else a violation")
    else:
        out["parity"] = props
    if world > 1:
        torch.distributed.destroy_process_group()
    return out if rank == 0 else None


def host_budget_bytes() -> int:
    """Pinned host memory one process may take for the end-to-end leg: half of
    the host's available memory, shared by the processes of this node."""
    avail = 0
    try:
        for ln in open("/proc/meminfo"):
            if ln.startswith("MemAvailable:"):
                avail = int(ln.split()[1]) * 1024
    except OSError:
        pass
    local_world = int(os.environ.get("LOCAL_WORLD_SIZE", os.environ.get("WORLD_SIZE", "1")))
    return int(0.5 * avail / max(1, local_world)) if avail else 1 << 62


def e2e_layers(wl, budget: int) -> int:
    """Layers the end-to-end leg can move within `budget` bytes of pinned host
    memory (inputs in, pools out): all of them when they fit."""
    per_layer = (wl.algorithmic_bytes()["total"] + wl.n_layers * wl.num_pages * 16 * wl.row_width * 2
                 * len(wl.tensors)) / wl.n_layers
    return max(1, min(wl.n_layers, int(budget // max(per_layer, 1))))


def bench_e2e_bounded(dwl, wl, args, stream, device) -> dict:
    """The end-to-end leg on the whole workload when its pinned host buffers
    fit this process's share of host memory; otherwise on a copy of the
    workload cut to its first layers (every layer does the same work), its
    rate scaled to the full layer count and labelled so."""
    import harness
    import workloads as W
    n = e2e_layers(wl, host_budget_bytes())
    if n >= wl.n_layers:
        return bench_e2e(dwl, wl, args, stream)
    sub = W.config(args.config)
    sub.n_layers = n
    out = bench_e2e(harness.DeviceWorkload(sub, device), sub, args, stream)
    out["value"] *= n / wl.n_layers
    out["layers_moved"] = n
    out["note"] = (f"host memory: the step moved {n} of {wl.n_layers} layers (inputs in, pools out); value is that "
                   f"rate scaled by {n}/{wl.n_layers} to the full model")
    return out


def bench_e2e(dwl, wl, args, stream) -> dict:
    """End to end through the C ABI with host buffers: every step copies its
    inputs in from pinned host memory, runs the operator and copies every
    destination pool out.  Steps are pipelined the way a serving loop would
    run them: the upload of step i+1, the kernel of step i and the download
    of step i-1 proceed on three streams over two device buffer sets."""
    import torch
    sets = [dwl, dwl.replica()]

    def inputs(d):
        out = []
        for n in wl.tensors:
            out.append(d.rows[n])
            out += [t for t in d.u[n] + d.w[n] if t is not None]
        if d.block_tables is not None:
            out.append(d.block_tables)
        return out

    dev_in = [inputs(d) for d in sets]
    host_in = []
    for t in dev_in[0]:
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        host_in.append(h)
    host_out = [torch.empty(p.shape, dtype=p.dtype, pin_memory=True) for p in dwl.pools.values()]
    bi = sum(t.numel() * t.element_size() for t in host_in)
    bo = sum(t.numel() * t.element_size() for t in host_out)
    steps = max(3, min(args.e2e_steps, args.steps))
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event() for _ in sets] for k in ("in", "run", "out")}
    used = [False, False]

    def one(i):
        b = i % 2
        d = sets[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev["run"][b])          # the previous kernel on this set has read its inputs
            for h, t in zip(host_in, dev_in[b]):
                t.copy_(h, non_blocking=True)
            ev["in"][b].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(ev["in"][b])
            if used[b]:
                s_run.wait_event(ev["out"][b])         # the previous result of this set has left
            d.run(stream=s_run)
            ev["run"][b].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["run"][b])
            for h, p in zip(host_out, d.pools.values()):
                h.copy_(p, non_blocking=True)
            ev["out"][b].record(s_out)
        used[b] = True

    for i in range(4):
        one(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        one(i)
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / steps
    del sets[1]
    return {"value": wl.n_chunk_tokens / dt, "unit": "tokens/s", "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "ms_per_step": dt * 1e3, "steps": steps,
            "pipeline": "upload / kernel / download on three streams, two device buffer sets"}


# --------------------------------------------------------------------------- #
# reference arm: the oracle on the host cores
# --------------------------------------------------------------------------- #
def bench_reference(args) -> dict:
    """The oracle timed on the host cores: each step evaluates a bounded number
    of rows, sized so the whole run stays within about two minutes."""
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    o = OracleSampler(args.config)
    probe, n_probe = o.step(256)
    rows_per_s = n_probe / max(probe, 1e-6)
    per_step = max(8, min(o.n_tokens, int(rows_per_s * 100.0 / (args.steps + args.warmup))))
    for _ in range(args.warmup):
        o.step(per_step)
    secs, rows = 0.0, 0
    for _ in range(args.steps):
        s_, n_ = o.step(per_step)
        secs += s_
        rows += n_
    value = o.tokens(rows) / secs
    sample = (f"{rows // args.steps} rows per step of one layer of {o.wl.name} ({o.kinds}), fp64 NumPy, one "
              f"thread; one chunk token = {o.layer_tensors} rows")
    return {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(o.wl, world),
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample,
                             "os_cpu_count": os.cpu_count()},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# --------------------------------------------------------------------------- #
# patch formation (and the orbit patch): the factors of one chunk's deficit
# --------------------------------------------------------------------------- #
PATCH_METRIC = "patch formation: chunk tokens/s (rank-m K and V factors of one chunk, all layers)"


def patch_form_setup(wl, orbit: int, device):
    """Seeded synthetic caches of the workload's first chunk: canonical K and V
    rows and `orbit` conditioned copies (canonical plus a conditioning term)."""
    import torch
    c = wl.chunks[0]
    L, T, D = wl.n_layers, c.n_tokens, wl.row_width
    g = torch.Generator(device=device).manual_seed(wl.seed + 101)
    canon = {n: torch.randn((L, T, D), generator=g, device=device).to(torch.bfloat16) for n in wl.tensors}
    cond = {n: [(canon[n].float() + 0.1 * torch.randn((L, T, D), generator=g, device=device)).to(torch.bfloat16)
                for _ in range(orbit)] for n in wl.tensors}
    deltas = [int(c.delta) + 977 * i for i in range(orbit)]
    return canon, cond, deltas


def patch_bytes(L, T, D, m, p, q, orbit) -> int:
    """Bytes this method moves per tensor: read the caches (bf16), write the
    deficit twice (bf16 rows and transposed rows), 2q + 3 tensor-core passes
    over it (bf16), the small fp32 operands (each pass's output, and the Gram's
    and the apply's reads in each of the 2q + 2 orthonormalisation rounds), and
    the factors."""
    kp = (m + p + 15) // 16 * 16
    n = L * T * D
    skinny = L * (T + D) * kp * 4
    return (n * 2 * (1 + orbit) + n * 4 + (2 * q + 3) * n * 2 + ((2 * q + 3) + 2 * (2 * q + 2)) * skinny
            + L * (T + D) * m * 2)


def patch_form_jobs(tensors, n_layers: int, streams: int):
    """The calls of one patch-formation step: (tensor, first layer, end layer)
    for each tensor, its layers cut into max(1, streams // len(tensors)) nearly
    equal ranges (empty ranges dropped), and that range count."""
    per = max(1, streams // len(tensors))
    bounds = [n_layers * i // per for i in range(per + 1)]
    jobs = [(n, bounds[i], bounds[i + 1]) for n in tensors for i in range(per) if bounds[i + 1] > bounds[i]]
    return jobs, per


def bench_patch_form(args) -> dict:
    import torch
    import workloads as W
    import position_invariant_kv_gb300 as kvrp
    rank, world, local = dist_env()
    if rank != 0:
        return None
    torch.cuda.set_device(local)
    from position_invariant_kv_gb300.build import build
    build()
    kvrp.lib()
    wl = W.config(args.config)
    if args.layers:
        wl.n_layers = min(wl.n_layers, args.layers)
    device = f"cuda:{local}"
    c = wl.chunks[0]
    L, T, D = wl.n_layers, c.n_tokens, wl.row_width
    m = c.rank if c.rank else 32
    p, q, orbit = args.oversample, args.power_iters, args.orbit
    canon, cond, deltas = patch_form_setup(wl, orbit, device)
    g = torch.Generator(device=device).manual_seed(wl.seed + 202)
    omega = torch.randn((D, m + p), generator=g, device=device)
    fac = {n: (torch.empty((L, T, m), dtype=torch.bfloat16, device=device),
               torch.empty((L, D, m), dtype=torch.bfloat16, device=device)) for n in wl.tensors}
    d_status = torch.zeros(1, dtype=torch.int32, device=device)
    # a graph is captured on a stream of its own (never the legacy default stream)
    stream = torch.cuda.Stream(device=device) if args.graph else torch.cuda.current_stream()
    if wl.family == "mla":
        kinds = {"kv": (kvrp.KVRP_ROPE_MLA_TAIL, wl.rope_dim)}
    else:
        kinds = {"k": (kvrp.KVRP_ROPE_HEADS, wl.head_dim), "v": (kvrp.KVRP_ROPE_NONE, 0)}
    # The calls of a step (one per tensor, or per tensor and range of layers) each run on
    # a stream of their own with their own workspace: one call's k x k solves (one CTA per
    # layer) overlap another's passes over the deficit.
    jobs, per = patch_form_jobs(wl.tensors, L, args.streams)
    streams = [torch.cuda.Stream(device=device) for _ in jobs] if args.streams > 1 else [stream] * len(jobs)
    wss = [torch.empty(kvrp.kv_patch_form_workspace_size(l1 - l0, T, D, m, p), dtype=torch.uint8, device=device)
           for (_, l0, l1) in (jobs if args.streams > 1 else jobs[:1])]
    fork = torch.cuda.Event()
    joins = [torch.cuda.Event() for _ in jobs]

    def fork_all():
        fork.record(stream)
        for s in set(streams):
            if s is not stream:
                s.wait_event(fork)

    def join_all():
        for j, s in enumerate(streams):
            joins[j].record(s)
            stream.wait_event(joins[j])

    def step():
        # Steps are independent chunks: each stream runs its calls back to back (its
        # workspace and outputs are only reused in its own order) unless --join-steps
        # makes every step wait for the previous one on all streams.
        if args.join_steps:
            fork_all()
        for j, (n, l0, l1) in enumerate(jobs):
            kind, rot = kinds[n]
            kvrp.kv_patch_form_orbit([x[l0:l1] for x in cond[n]], deltas, canon[n][l0:l1], n_layers=l1 - l0,
                                     n_tokens=T, row_width=D, rope_kind=kind, rot_dim=rot, rope_theta=wl.theta,
                                     rank=m, oversample=p, power_iters=q, omega=omega, u_out=fac[n][0][l0:l1],
                                     v_out=fac[n][1][l0:l1], workspace=wss[min(j, len(wss) - 1)],
                                     d_status=d_status, stream=streams[j])
        if args.join_steps:
            join_all()

    fork_all()
    for _ in range(args.warmup):
        step()
    join_all()
    torch.cuda.synchronize()
    graph = None
    if args.graph:
        # one step (its calls on their streams, forked from and joined to the capture stream)
        # recorded once into a CUDA graph and replayed: the library calls are capturable
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            fork_all()
            step()
            join_all()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                graph.replay()
        torch.cuda.synchronize()
    steps = args.steps
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        if graph is not None:
            with torch.cuda.stream(stream):
                for _ in range(steps):
                    graph.replay()
        else:
            fork_all()
            for _ in range(steps):
                step()
            join_all()
        t1.record(stream)
        torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    nb = patch_bytes(L, T, D, m, p, q, orbit) * len(wl.tensors)
    peaks = measured_peaks()
    achieved = nb / (ms / 1e3) / 1e9
    out = {
        "metric": PATCH_METRIC, "value": T / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "row": "patch_form",
        "config": {"workload": f"{wl.name} first chunk: {L} layers x {T} tokens x {D} features, tensors "
                               f"{'/'.join(wl.tensors)}, rank {m}, oversample {p}, {q} subspace iterations, "
                               f"orbit of {orbit} ordering(s), "
                               f"{len(jobs)} call(s) per step ({per} layer range(s) per tensor), "
                               f"{'each on its own stream' if args.streams > 1 else 'in turn on one stream'}"
                               f"{', every step joined' if args.join_steps else ''}"
                               f"{', the step replayed from a CUDA graph' if args.graph else ''}",
                   "tokens_per_step": T, "method_bytes_per_step": nb,
                   "l2": f"inputs larger than L2 ({nb / 1e6:.0f} MB moved per step vs 129 MB L2)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": None,
                     "kernel": "kv_patch_form_orbit, whole call (delta, tensor-core passes, k x k solves)",
                     "peak_source": peaks["source"]},
        # per call: deficit, Omega transpose, 2q + 3 passes over the deficit, 2q + 2 orthonormalisation
        # rounds of (Gram, Cholesky, apply), the projected Gram, Jacobi, the B^T W apply, U and V writers
        "gpu_launches": steps * len(jobs) * (2 + (2 * q + 3) + 3 * (2 * q + 2) + 5),
        "clocks": clocks.summary(),
        "device_status": int(d_status.item()),
    }
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = run_patch_cpu_baseline(args.config, args.budget)
    return out


def patch_cpu_worker(cfg: int, budget_s: float) -> dict:
    """The oracle's patch formation (fp64 deficit + exact truncated SVD) on
    whole (layer, tensor) slices of the chunk until the budget is spent."""
    import numpy as np
    import workloads as W
    from oracle import conditioning_deficit, row_layout, svd_patch
    wl = W.config(cfg)
    c = wl.chunks[0]
    T, D = c.n_tokens, wl.row_width
    m = c.rank if c.rank else 32
    rng = np.random.default_rng(wl.seed + 303)
    elapsed, n = 0.0, 0
    while elapsed < budget_s:
        name = wl.tensors[n % len(wl.tensors)]
        lay = row_layout(wl.family, name, n_heads=wl.n_heads, head_dim=wl.head_dim, kv_lora_dim=wl.kv_lora_dim,
                         rope_dim=wl.rope_dim)
        canon = rng.standard_normal((T, D))
        cond = canon + 0.1 * rng.standard_normal((T, D))
        t0 = time.perf_counter()
        svd_patch(conditioning_deficit(cond, canon, c.delta, wl.theta, lay), m)
        elapsed += time.perf_counter() - t0
        n += 1
    slices = wl.n_layers * len(wl.tensors)
    return {"value": T * n / slices / elapsed, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} (layer, tensor) slices of {T} x {D} ({wl.name}; fp64 deficit and exact SVD, NumPy, "
                      f"one thread, {elapsed:.1f} s); one chunk = {slices} slices"}


def run_patch_cpu_baseline(cfg: int, budget_s: float) -> dict:
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--cpu-baseline-worker", "--row",
                          "patch_form", "--config", str(cfg), "--budget", str(budget_s)],
                         capture_output=True, text=True, env=env, timeout=900)
    if res.returncode != 0:
        tail = res.stderr.strip().splitlines()[-1] if res.stderr.strip() else "no output"
        return {"value": None, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": "failed: " + tail}
    return json.loads(res.stdout.strip().splitlines()[-1])


# --------------------------------------------------------------------------- #
# fused read: decode attention over relocated, patched chunks (no relocated cache)
# --------------------------------------------------------------------------- #
ATTN_METRIC = "relocated-chunk decode attention: context tokens/s (one query token per sequence, one layer)"
ATTN_SHAPE = dict(seqs=16, chunks=4, tokens=4096, Hq=28, Hkv=4, d=128, rank=32, theta=1e6)


def attn_text(a) -> str:
    return (f"one layer of a Qwen2.5-VL-shaped GQA model ({a['Hq']} query / {a['Hkv']} KV heads x {a['d']}): "
            f"{a['seqs']} sequences, each {a['chunks']} relocated chunks x {a['tokens']} tokens with rank-{a['rank']} "
            f"K and V patches, theta {a['theta']:g}; canonical K, V in a shuffled 16-token paged pool")


def attn_bytes(a) -> int:
    n_chunks = a["seqs"] * a["chunks"]
    D = a["Hkv"] * a["d"]
    per_chunk = a["tokens"] * D * 2 * 2 + a["tokens"] * a["rank"] * 2 * 2 + D * a["rank"] * 2 * 2
    return n_chunks * per_chunk + a["seqs"] * a["Hq"] * a["d"] * 2 * 2


def attend_workload(a, dev, seed: int = 4242):
    """The attention row's seeded synthetic inputs on the device: (tensors kept
    alive, AttnChunk list, q [seqs][Hq][d], seq_chunks).  The canonical K and V
    of all chunks sit in one paged pool per tensor ([pages][16][H_kv d], pages
    handed out by a seeded shuffle, as a serving cache holds them); each chunk
    reads its pages through its block table.  bf16 N(0,1) K, V and queries,
    U_k, U_v N(0, 0.3^2), V_k, V_v N(0, 0.1^2); chunk i shifted by
    (7919 i mod 65536) - 32768."""
    import torch
    import position_invariant_kv_gb300 as kvrp
    g = torch.Generator(device=dev).manual_seed(seed)
    D = a["Hkv"] * a["d"]
    n_chunks = a["seqs"] * a["chunks"]
    per = (a["tokens"] + 15) // 16
    n_pages = n_chunks * per

    def rnd(*shape, std=1.0):
        return (std * torch.randn(shape, generator=g, device=dev)).to(torch.bfloat16)

    pool_k, pool_v = rnd(n_pages, 16, D), rnd(n_pages, 16, D)
    perm = torch.randperm(n_pages, generator=g, device=dev).to(torch.int32)
    keep, chunks = [pool_k, pool_v, perm], []
    for i in range(n_chunks):
        t = [rnd(a["tokens"], a["rank"], std=0.3), rnd(D, a["rank"], std=0.1), rnd(a["tokens"], a["rank"], std=0.3),
             rnd(D, a["rank"], std=0.1)]
        keep += t
        chunks.append(kvrp.AttnChunk(k=pool_k, v=pool_v, n_tokens=a["tokens"], delta=(i * 7919) % 65536 - 32768,
                                     rank=a["rank"], uk=t[0], vk=t[1], uv=t[2], vv=t[3],
                                     block_table=perm[i * per:(i + 1) * per], num_pages=n_pages))
    seq_chunks = [s * a["chunks"] for s in range(a["seqs"] + 1)]
    q = rnd(a["seqs"], a["Hq"], a["d"])
    return keep, chunks, q, seq_chunks


def bench_attend(args) -> dict:
    import torch
    import position_invariant_kv_gb300 as kvrp
    rank, world, local = dist_env()
    if rank != 0:
        return None
    torch.cuda.set_device(local)
    from position_invariant_kv_gb300.build import build
    build()
    kvrp.lib()
    a = dict(ATTN_SHAPE)
    dev = f"cuda:{local}"
    n_chunks = a["seqs"] * a["chunks"]
    keep, chunks, q, seq_chunks = attend_workload(a, dev)
    arr = kvrp.attn_chunk_array(chunks)
    out = torch.empty_like(q)
    ws = torch.empty(kvrp.kv_attend_relocated_workspace_size([a["tokens"]] * n_chunks, a["Hq"], a["Hkv"], a["d"]),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        kvrp.kv_attend_relocated(q, arr, seq_chunks, n_q_heads=a["Hq"], n_kv_heads=a["Hkv"], head_dim=a["d"],
                                 rope_theta=a["theta"], softmax_scale=a["d"] ** -0.5, out=out, workspace=ws,
                                 d_status=status, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"kv_attend_relocated reported device status {int(status.item()):#x}")
    ms = t0.elapsed_time(t1) / args.steps
    nb = attn_bytes(a)
    peaks = measured_peaks()
    achieved = nb / (ms / 1e3) / 1e9
    ctx = a["seqs"] * a["chunks"] * a["tokens"]
    out_line = {
        "metric": ATTN_METRIC, "value": ctx / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic", "row": "attend",
        "config": {"workload": attn_text(a), "context_tokens_per_step": ctx, "algorithmic_bytes_per_step": nb,
                   "l2": f"inputs larger than L2 ({nb / 1e6:.0f} MB read per step vs 129 MB L2)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "traffic": profiled_traffic("attend", "attend_dram.json", ATTEND_SOURCES),
                     "kernel": "kv_attend_relocated, whole call (block and combine kernels); traffic is "
                               "block_kernel's DRAM bytes per launch",
                     "peak_source": peaks["source"]},
        "gpu_launches": kvrp.kvrp_last_launch_count() * args.steps,
        "clocks": clocks.summary(),
    }
    if not args.no_cpu_baseline:
        out_line["cpu_baseline"] = run_attn_cpu_baseline(args.budget)
    return out_line


def attn_cpu_worker(budget_s: float) -> dict:
    """The fp64 oracle (materialised K^, V^ and softmax) on whole sequences of
    the bench shape until the budget is spent."""
    import numpy as np
    from oracle import attend_relocated, round_to_bf16_bits
    a = dict(ATTN_SHAPE)
    rng = np.random.default_rng(4242)
    D = a["Hkv"] * a["d"]
    elapsed, n = 0.0, 0
    while elapsed < budget_s:
        cs = []
        for i in range(a["chunks"]):
            cs.append({"k": round_to_bf16_bits(rng.standard_normal((a["tokens"], D))),
                       "v": round_to_bf16_bits(rng.standard_normal((a["tokens"], D))), "delta": 1000 * i,
                       "uk": round_to_bf16_bits(0.3 * rng.standard_normal((a["tokens"], a["rank"]))),
                       "vk": round_to_bf16_bits(0.1 * rng.standard_normal((D, a["rank"]))),
                       "uv": round_to_bf16_bits(0.3 * rng.standard_normal((a["tokens"], a["rank"]))),
                       "vv": round_to_bf16_bits(0.1 * rng.standard_normal((D, a["rank"])))})
        q = round_to_bf16_bits(rng.standard_normal(a["Hq"] * a["d"]))
        t0 = time.perf_counter()
        attend_relocated(q, cs, a["Hq"], a["Hkv"], a["d"], a["theta"], a["d"] ** -0.5)
        elapsed += time.perf_counter() - t0
        n += 1
    ctx = n * a["chunks"] * a["tokens"]
    return {"value": ctx / elapsed, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} sequences of {a['chunks']} x {a['tokens']} tokens (fp64 NumPy, one thread, "
                      f"{elapsed:.1f} s)"}


def run_attn_cpu_baseline(budget_s: float) -> dict:
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--cpu-baseline-worker", "--row",
                          "attend", "--budget", str(budget_s)], capture_output=True, text=True, env=env, timeout=900)
    if res.returncode != 0:
        tail = res.stderr.strip().splitlines()[-1] if res.stderr.strip() else "no output"
        return {"value": None, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": "failed: " + tail}
    return json.loads(res.stdout.strip().splitlines()[-1])


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0,
                    help="timed steps; 0 (default) picks a count that keeps the timed region near ten seconds")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", type=int, default=4,
                    help="workload: 4 (default) is the sliding-window survival + recall batch, the largest")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20,
                    help="end-to-end steps (host copies in the loop); 0 skips that leg (profiler captures only)")
    ap.add_argument("--layers", type=int, default=0, help="use only the first N layers (profiling captures)")
    ap.add_argument("--budget", type=float, default=15.0, help="seconds of oracle time for the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-baseline-worker", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--parity-sample", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--row", choices=["relocate", "patch_form", "attend"], default="relocate",
                    help="relocate: the reuse operator (the headline); patch_form: forming the patch factors; "
                         "attend: decode attention over relocated chunks without materialising them")
    ap.add_argument("--orbit", type=int, default=1, help="patch_form: conditioned caches averaged (orbit patch)")
    ap.add_argument("--oversample", type=int, default=16, help="patch_form: range-finder oversampling")
    ap.add_argument("--power-iters", type=int, default=2, help="patch_form: subspace iterations")
    ap.add_argument("--join-steps", type=int, default=0,
                    help="patch_form: 1 makes each step wait for the previous one on every stream")
    ap.add_argument("--graph", type=int, default=0,
                    help="patch_form: 1 records one step into a CUDA graph and times its replays")
    ap.add_argument("--streams", type=int, default=4,
                    help="patch_form: concurrent calls per step, one stream each (tensors first, then layer "
                         "ranges of each tensor); 1 runs the tensors in turn on one stream")
    args = ap.parse_args()
    if args.cpu_baseline_worker:
        if args.row == "attend":
            print(json.dumps(attn_cpu_worker(args.budget)))
            return
        if args.row == "patch_form":
            print(json.dumps(patch_cpu_worker(args.config, args.budget)))
            return
        out = cpu_baseline_worker(args.config, args.budget)
        if args.parity_sample:
            out["parity"] = parity_worker(args.parity_sample)
        print(json.dumps(out))
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if not args.steps and (args.impl == "reference" or args.row != "relocate"):
        args.steps = 20 if args.impl == "reference" else {"patch_form": 200, "attend": 2000}[args.row]
    if args.impl == "reference":
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[k] = "1"
    if args.row == "attend":
        if args.impl == "reference":
            rank, world, _ = dist_env()
            if rank != 0:
                return
            cb = attn_cpu_worker(args.budget)
            out = {"metric": ATTN_METRIC, "value": cb["value"], "unit": "tokens/s", "n_gpus": world,
                   "impl": "reference", "higher_is_better": True, "dtype": "f64", "data": "synthetic", "row": "attend",
                   "config": {"workload": attn_text(ATTN_SHAPE)}, "cpu_baseline": cb,
                   "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        else:
            out = bench_attend(args)
        if out is not None:
            print(json.dumps(out))
        return
    if args.row == "patch_form":
        if args.impl == "reference":
            rank, world, _ = dist_env()
            if rank != 0:
                return
            cb = patch_cpu_worker(args.config, args.budget)
            out = {"metric": PATCH_METRIC, "value": cb["value"], "unit": "tokens/s", "n_gpus": world, "impl": "reference",
                   "higher_is_better": True, "dtype": "f64", "data": "synthetic", "row": "patch_form",
                   "config": {"workload": cb["sample"]}, "cpu_baseline": cb,
                   "e2e": {"value": cb["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        else:
            out = bench_patch_form(args)
        if out is not None:
            print(json.dumps(out))
        return
    out = bench_reference(args) if args.impl == "reference" else bench_ours(args)
    if out is not None:
        print(json.dumps(out))


if __name__ == "__main__":
    main()
