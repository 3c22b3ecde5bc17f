"""Benchmark of one paged-KV decode step on GB300: slot-mapped KV write + split-K paged decode
attention (split kernel + merge kernel), through the C ABI, on a seeded synthetic workload.

Prints one JSON line. `value` is algorithmic KV GB/s of the whole step (bytes the step must move
divided by device time), `tokens_per_s` the decoded tokens per second of that one attention
layer. L2 is flushed before every step (a 512 MB write, then a 1 GB read so that no dirty line
of the flush is written back during the timed kernels), outside the timed events. The flush keeps
the GPU busy for ~0.2 ms per step, long enough that the host has queued the step's launches
before the first timed event runs: the events then hold device time only (with a 256 MB read the
Llama-3-8B-shaped step measures ~4 % slower, host launch time leaking into the events).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--chunk T]
    python bench.py --impl reference ...   # the fp64 oracle on the host cores, same metric

For N > 1 it runs under torchrun, one rank per GPU; every rank decodes its own batch (a seed
of its own: weak scaling, no data-path collective); the barrier, the max over ranks and the
sum of bytes are the only communication.
"""
import argparse
import contextlib
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged decode attn: KV GB/s vs GB300 HBM peak; decoded tokens/s per step"
DEFAULT_CONFIG = 3          # long-context split-K decode (B=8, 32k-131k): the largest workload
MIN_LOOP_MS = 1000.0        # the roofline and e2e loops run at least this much GPU time
SECONDARY_LOOP_MS = 300.0   # each secondary workload's attention loop
FALLBACK_HBM_GBS = 6800.0   # used only when MEASURED_PEAKS.json is absent
L2_FLUSH_BYTES = 512 << 20
PROFILES = os.path.join(ROOT, "profiles")
CSRC = os.path.join(ROOT, "paged_kv_decode_reshape_gb300", "csrc")


# ------------------------------------------------------------------------------------------
# host-side pieces (no GPU needed; covered by tests/test_bench_host.py)
# ------------------------------------------------------------------------------------------

def dist_env():
    """(rank, world_size, local_rank) from the torchrun environment (1 process otherwise)."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def rank_seed(cfg: int, rank: int) -> int:
    """Each rank decodes its own batch: the config's seed for rank 0, distinct ones after."""
    return cfg + 1000 * rank


def aggregate(local_bytes: float, local_ms: float, group=None):
    """Whole-job (bytes, ms): bytes summed over ranks, time the max over ranks."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return local_bytes, local_ms
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([local_bytes], dtype=torch.float64, device=dev)
    m = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    dist.all_reduce(m, op=dist.ReduceOp.MAX, group=group)
    return float(t.item()), float(m.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# the sources the dominant (split) kernel is built from: a change to any of them makes the
# committed ncu traffic figure stale
SPLIT_KERNEL_SOURCES = ("decode_mma.cuh", "decode_mma.cu", "pkv_device.cuh", "pkv_internal.h")


def source_code_only(text: str) -> str:
    """C/C++ source with its comments removed (string and character literals kept) and every run of
    whitespace collapsed to one space: what the compiler sees, so an edit of comments or layout does
    not mark the ncu figures of unchanged code as stale."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in SPLIT_KERNEL_SOURCES:
        with open(os.path.join(CSRC, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + source_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the split kernel for this workload from profiles/traffic.json (a
    single-pass ncu capture), if the kernel sources are unchanged since the capture (else None)."""
    path = os.path.join(PROFILES, "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        entry = json.load(f).get("split_kernel", {}).get(workload)
    if not entry or entry.get("kernel_source_sha") != kernel_source_hash():
        return None
    try:
        return int(entry["traffic_bytes_per_launch"])
    except (KeyError, TypeError, ValueError):
        return None


@contextlib.contextmanager
def nvtx_range(name: str):
    """An NVTX range around a bench region (for ncu --nvtx or nsys); nothing if NVTX is not
    available."""
    pushed = False
    try:
        import torch
        torch.cuda.nvtx.range_push(name)
        pushed = True
    except Exception:
        pass
    try:
        yield
    finally:
        if pushed:
            try:
                torch.cuda.nvtx.range_pop()
            except Exception:
                pass


def timed_loop(untimed, timed, min_ms: float, first: int, stream):
    """Per iteration k: untimed(k) (the L2 flush), then timed(k) between a CUDA event pair on
    `stream`. Runs in batches until the events add up to at least min_ms of GPU time and at least
    `first` iterations ran. Returns (total ms inside the events, iterations)."""
    import torch
    total, n = 0.0, 0
    while n < first or total < min_ms:
        if n < first:
            batch = first - n
        else:  # enough iterations for the remaining time at the average so far, at most 2000
            batch = max(1, min(2000, int((min_ms - total) / max(total / n, 1e-3)) + 1))
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(batch)]
        for i in range(batch):
            untimed(n + i)
            ev[i][0].record(stream)
            timed(n + i)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        total += sum(e[0].elapsed_time(e[1]) for e in ev)
        n += batch
    return total, n


def attention_bytes(w: W.DecodeWorkload) -> int:
    """Algorithmic bytes of the attention call alone (KV + scales + q + out + tables)."""
    elem = {"f32": 4, "bf16": 2, "i8": 1}[w.kv_dtype]
    per_tok = w.Hkv * w.D * elem * 2 + (w.Hkv * 8 if w.kv_dtype == "i8" else 0)
    written = int((w.slot_mapping >= 0).sum())
    wr = written * per_tok * 2 + 8 * w.T
    return W.kv_bytes(w) - wr


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.gpu = gpu_index

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as f:
            rows = [r.strip() for r in f if r.strip()]
        os.unlink(self.path)
        return parse_clock_rows(rows)


def parse_clock_rows(rows):
    sm, mx, reasons = [], None, set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for r in rows:
        parts = [p.strip() for p in r.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            mx = float(parts[2])
        except ValueError:
            continue
        for name, val in zip(names, parts[5:9]):
            if val.lower().startswith("active"):
                reasons.add(name)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
            "samples": len(sm)}


def stage_buffers(dev, tensors):
    """Copy `tensors` into one uint8 device buffer (each at a 256-byte-aligned offset) and return
    (buffer, {name: view of the buffer with the tensor's dtype and shape})."""
    import torch
    offs, total = {}, 0
    for n, t in tensors.items():
        offs[n] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(max(total, 256), dtype=torch.uint8, device=dev)
    views = {}
    for n, t in tensors.items():
        nb = t.numel() * t.element_size()
        v = buf[offs[n]:offs[n] + nb].view(t.dtype).view(t.shape)
        v.copy_(t)
        views[n] = v
    return buf, views


def cuda_launches_per_step(w: W.DecodeWorkload, chunk_used: int, cascade: bool = False) -> int:
    """Kernels of this library one step launches: write, split, and merge when any split; a
    shared-prefix (cascade) step adds the prefix kernel and always merges."""
    if cascade:
        return 4
    splits = max(1, w.max_context_len // chunk_used)
    return 2 + (1 if splits > 1 else 0)


# ------------------------------------------------------------------------------------------
# the fp64 oracle on the host cores (cpu_baseline and --impl reference)
# ------------------------------------------------------------------------------------------

def oracle_step_seconds(w: W.DecodeWorkload, rows, threads: int, keep=None) -> float:
    """Seconds of one oracle step (write + attention) over `rows`; with `keep` (a dict), also
    keeps the rows and the fp64 output there."""
    import oracle
    kp, vp = w.k_pool, w.v_pool
    ks, vs = w.k_scales, w.v_scales
    rows = np.asarray(rows)
    t0 = time.perf_counter()
    oracle.kv_cache_write(w.k_new[rows], w.v_new[rows], kp, vp, w.slot_mapping[rows],
                          None if w.k_new_scales is None else w.k_new_scales[rows],
                          None if w.v_new_scales is None else w.v_new_scales[rows],
                          ks, vs, inplace=True)
    out = oracle.paged_decode_attention(w.q[rows], kp, vp, w.block_tables[rows], w.context_lens[rows],
                                        w.scale, ks, vs, num_threads=threads)
    dt = time.perf_counter() - t0
    if keep is not None:
        keep["rows"], keep["out"] = rows, out
    return dt


def accuracy_vs_oracle(gpu_out, ref, rows) -> dict:
    """Max and mean |GPU - oracle| over the checked rows (the GPU output cast up to fp64)."""
    got = np.asarray(gpu_out, dtype=np.float64)[np.asarray(rows)]
    d = np.abs(got - ref)
    finite = np.isfinite(d)
    fin = lambda v: float(v) if np.isfinite(v) else None
    return {"max_abs_err": fin(d[finite].max()) if finite.any() else None,
            "mean_abs_err": fin(d[finite].mean()) if finite.any() else None,
            "max_abs_ref": fin(np.abs(ref).max()), "nonfinite": int((~finite).sum()),
            "rows_checked": int(len(rows)), "elements_checked": int(d.size)}


def sample_rows(w: W.DecodeWorkload, cpu_budget_s: float):
    """A prefix of the batch whose oracle step costs about cpu_budget_s seconds of CPU time,
    from a single-thread probe of the first sequence."""
    t0 = oracle_step_seconds(w, [0], 1)
    per_tok = t0 / max(1, int(w.context_lens[0]))
    n, cost = 0, 0.0
    while n < w.B and cost + int(w.context_lens[n]) * per_tok <= cpu_budget_s:
        cost += int(w.context_lens[n]) * per_tok
        n += 1
    return list(range(max(1, n)))


def sample_bytes(w: W.DecodeWorkload, rows) -> int:
    rows = np.asarray(rows)
    sub = W.DecodeWorkload(**{**w.__dict__, "B": len(rows), "q": w.q[rows],
                              "block_tables": w.block_tables[rows],
                              "context_lens": w.context_lens[rows],
                              "slot_mapping": w.slot_mapping[rows], "k_new": w.k_new[rows],
                              "v_new": w.v_new[rows], "shared_prefix_blocks": 0})
    if w.shared_prefix_blocks and len(rows) > 1:
        sub.shared_prefix_blocks = w.shared_prefix_blocks
    return W.kv_bytes(sub)


# Arm (implementer, part) codes of /proc/cpuinfo with a known core name
ARM_CORES = {(0x41, 0xd4f): "Arm Neoverse-V2", (0x41, 0xd40): "Arm Neoverse-V1",
             (0x41, 0xd0c): "Arm Neoverse-N1", (0x41, 0xd49): "Arm Neoverse-N2"}


def parse_cpu_model(cpuinfo: str, machine: str) -> str:
    """The CPU model from /proc/cpuinfo text: x86 kernels give a 'model name' line; Arm kernels
    give implementer and part codes, named from ARM_CORES when known."""
    impl = part = None
    for ln in cpuinfo.splitlines():
        key, _, val = ln.partition(":")
        key, val = key.strip().lower(), val.strip()
        if key == "model name" and val:
            return val
        try:
            if key == "cpu implementer" and impl is None:
                impl = int(val, 16)
            elif key == "cpu part" and part is None:
                part = int(val, 16)
        except ValueError:
            pass
    if impl is not None and part is not None:
        return ARM_CORES.get((impl, part), f"{machine} implementer 0x{impl:x} part 0x{part:x}")
    return machine or "unknown"


def host_cpu_model() -> str:
    try:
        with open("/proc/cpuinfo", errors="replace") as f:
            return parse_cpu_model(f.read(), platform.machine())
    except Exception:  # a descriptive field only: never fail the bench over it
        return platform.machine() or "unknown"


def cpu_baseline(w: W.DecodeWorkload, cpu_budget_s: float = 20.0, keep=None):
    """The oracle on a bounded sample: a prefix of the batch costing <= cpu_budget_s CPU
    seconds per step, repeated until about 10 CPU seconds have been spent (`keep`: see
    oracle_step_seconds)."""
    threads = os.cpu_count() or 1
    rows = sample_rows(w, cpu_budget_s)
    secs, reps = 0.0, 0
    while reps == 0 or (secs * threads < 10.0 and reps < 50):
        secs += oracle_step_seconds(w, rows, threads, keep)
        reps += 1
    gbs = sample_bytes(w, rows) * reps / secs / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "cpu_model": host_cpu_model(),
            "sample": f"{len(rows)} of {w.B} sequences of the {w.name} step (write + attention, "
                      f"all {w.Hq} heads) x {reps} repetitions, fp64 C oracle, {threads} threads, "
                      f"{secs:.2f} s wall"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return  # the oracle leg runs on rank 0 only
    w = W.make_config(args.config, seed=rank_seed(args.config, 0))
    threads = os.cpu_count() or 1
    steps = max(1, args.steps)
    # the whole run stays near two minutes of wall time on `threads` cores
    rows = sample_rows(w, max(0.05, 120.0 * threads / (steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_step_seconds(w, rows, threads)
    secs = sum(oracle_step_seconds(w, rows, threads) for _ in range(steps))
    nbytes = sample_bytes(w, rows)
    gbs = nbytes * steps / secs / 1e9
    ms = secs / steps * 1e3
    sample = (f"{len(rows)} of {w.B} sequences of the {w.name} step per timed step "
              f"(write + attention, all heads), fp64 C oracle, {threads} threads")
    line = {"metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "impl": "reference",
            "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "description": W.CONFIGS[args.config]},
            "tokens_per_s": round(len(rows) * steps / secs, 2),
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "cpu_model": host_cpu_model(), "sample": sample},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
# the CUDA path
# ------------------------------------------------------------------------------------------

class DecodeRun:
    """One decode workload resident on the device, with the calls a step makes: the L2 flush
    (untimed), the KV write and the attention call."""

    def __init__(self, pkv, w, dev, chunk_req=0, no_cascade=False):
        import torch
        self.pkv, self.w = pkv, w

        def up(a):
            if a is None:
                return None
            a = np.ascontiguousarray(a)
            if a.dtype == np.uint16:
                return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
            return torch.from_numpy(a).to(dev)

        self.kp, self.vp = up(w.k_pool), up(w.v_pool)
        self.ks, self.vs = up(w.k_scales), up(w.v_scales)
        # the step's own inputs (q, tables, lengths, slots, new K/V rows) live in one device
        # buffer, 256-byte aligned segments, so a step fed from the host needs a single copy
        self.stage, views = stage_buffers(dev, {n: up(a) for n, a in dict(
            q=w.q, bt=w.block_tables, cl=w.context_lens, sm=w.slot_mapping, kn=w.k_new, vn=w.v_new,
            kns=w.k_new_scales, vns=w.v_new_scales).items() if a is not None})
        self.q, self.bt, self.cl, self.sm, self.kn, self.vn = (
            views[n] for n in ("q", "bt", "cl", "sm", "kn", "vn"))
        self.kns, self.vns = views.get("kns"), views.get("vns")
        self.out = torch.empty_like(self.q)
        self.maxc = maxc = w.max_context_len
        self.chunk_req = chunk_req
        # a batch whose sequences share a prefix runs through the shared-prefix (cascade) call
        self.prefix = prefix = w.shared_prefix_blocks * w.BS
        self.cascade = prefix > 0 and not no_cascade
        self.chunk = pkv.decode_split_chunk(w.B, w.Hkv, w.D, maxc - (prefix if self.cascade else 0),
                                            chunk_req, {"f32": pkv.F32, "bf16": pkv.BF16, "i8": pkv.I8}[w.kv_dtype])
        nws = (pkv.decode_shared_prefix_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, maxc, prefix, chunk_req)
               if self.cascade else pkv.decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, maxc, chunk_req))
        self.ws = torch.empty(nws, dtype=torch.uint8, device=dev) if nws else None
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.clean = torch.zeros(L2_FLUSH_BYTES // 2, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.current_stream()

    def flush_l2(self, k):
        # write a buffer 4x the L2, then read a 1 GB one, so the step starts with a cold L2 holding
        # clean lines (no write-back of the flush's dirty lines charged to the timed kernels)
        self.flush.fill_(k & 0xFF)
        self.clean.max()

    def write(self):
        self.pkv.kv_cache_write(self.kn, self.vn, self.kp, self.vp, self.sm, self.kns, self.vns, self.ks,
                                self.vs, status=self.status, stream=self.stream)

    def attend(self):
        pkv, w = self.pkv, self.w
        if self.cascade:
            pkv.paged_decode_attention_shared_prefix(self.out, self.q, self.kp, self.vp, self.bt, self.cl,
                                                     self.maxc, w.scale, self.prefix, self.chunk_req,
                                                     self.ws, self.status, self.stream)
        elif w.kv_dtype == "i8":
            pkv.paged_decode_attention_int8(self.out, self.q, self.kp, self.vp, self.ks, self.vs, self.bt,
                                            self.cl, self.maxc, w.scale, self.chunk_req, self.ws,
                                            self.status, self.stream)
        else:
            pkv.paged_decode_attention(self.out, self.q, self.kp, self.vp, self.bt, self.cl, self.maxc,
                                       w.scale, self.chunk_req, self.ws, self.status, self.stream)


def measure_attention(pkv, cfg: int, dev, min_ms: float, warmup: int = 5) -> dict:
    """The attention call alone on config `cfg` (L2 flushed before each call, CUDA events around
    it, at least min_ms of GPU time), as a roofline record: a secondary measurement next to the
    headline line."""
    import torch
    w = W.make_config(cfg, seed=rank_seed(cfg, 0))
    run = DecodeRun(pkv, w, dev)
    for _ in range(max(3, warmup)):
        run.flush_l2(1)
        run.write()
        run.attend()
    torch.cuda.synchronize()
    if int(run.status.item()) != 0:
        raise RuntimeError(f"{w.name}: kernels flagged bad inputs: status {int(run.status.item())}")
    total_ms, n = timed_loop(run.flush_l2, lambda k: run.attend(), min_ms, 20, run.stream)
    hbm, peak_kind = measured_peaks()
    nbytes = attention_bytes(w)
    avg_s = total_ms / n / 1e3
    achieved = nbytes / avg_s / 1e9
    rec = {"workload": w.name, "description": W.CONFIGS[cfg], "dtype": w.kv_dtype,
           "attention_call_us": round(avg_s * 1e6, 3), "achieved_gbs": round(achieved, 2),
           "peak_gbs": hbm, "frac": round(achieved / hbm, 4), "peak_kind": f"of {peak_kind}",
           "algorithmic_bytes_per_launch": nbytes, "split_chunk": run.chunk,
           "shared_prefix_call": bool(run.cascade), "launches_timed": n,
           "timed_ms": round(total_ms, 2), "traffic": profiled_traffic(w.name)}
    del run
    torch.cuda.empty_cache()
    return rec


def run_ours(args):
    import torch
    import torch.distributed as dist

    import paged_kv_decode_reshape_gb300 as pkv

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    pkv.load(build_if_missing=False)
    dev = torch.device("cuda", local)

    w = W.make_config(args.config, seed=rank_seed(args.config, rank))
    run = DecodeRun(pkv, w, dev, args.chunk, getattr(args, "no_cascade", False))
    stage, out, status, stream = run.stage, run.out, run.status, run.stream
    maxc, chunk, cascade = run.maxc, run.chunk, run.cascade
    flush_l2, write, attend = run.flush_l2, run.write, run.attend

    # nvidia-smi samples the clocks from before the warm-up to the end of the e2e loop: the K timed
    # steps alone can be shorter than one sampling interval, the roofline and e2e loops are not
    clocks = ClockSampler(local)
    clocks.start()
    for _ in range(max(3, args.warmup)):
        flush_l2(1)
        write()
        attend()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"kernels flagged bad inputs: status {int(status.item())}")

    K = args.steps
    # one event pair per step: nothing between the write and the attention call, so the kernels
    # keep their programmatic-dependent-launch overlap
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    with nvtx_range("timed steps (write + attention)"):
        for k in range(K):
            flush_l2(k)                      # evict the previous step's lines (not timed)
            ev[k][0].record(stream)
            write()
            attend()
            ev[k][1].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall_s = time.perf_counter() - t_wall
    step_ms = sum(e[0].elapsed_time(e[1]) for e in ev)
    # the dominant kernels alone (the attention call: split + merge), for the roofline: at least
    # MIN_LOOP_MS of GPU time whatever K is
    with nvtx_range("attention calls (roofline loop)"):
        attn_total_ms, KA = timed_loop(flush_l2, lambda k: attend(), args.min_loop_ms, K, stream)

    step_bytes = W.kv_bytes(w)
    total_bytes, max_ms = aggregate(step_bytes * K, step_ms)
    ms_per_step = max_ms / K
    value = total_bytes / (max_ms / 1e3) / 1e9
    tokens_per_s = w.B * world * K / (max_ms / 1e3)

    # e2e through the public API: the step's inputs from pinned host memory each step (one copy of
    # the staging buffer), out read back; also at least MIN_LOOP_MS of GPU time
    host_stage = stage.cpu().pin_memory()
    host_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = host_stage.numel()
    d2h = out.numel() * out.element_size()
    torch.cuda.synchronize()

    def e2e_step(k):
        stage.copy_(host_stage, non_blocking=True)
        write()
        attend()
        host_out.copy_(out, non_blocking=True)
    with nvtx_range("e2e steps (host copies + write + attention)"):
        e2e_ms, KE = timed_loop(flush_l2, e2e_step, args.min_loop_ms, K, stream)
    e2e_bytes, e2e_max = aggregate(step_bytes * KE, e2e_ms)
    e2e_value = e2e_bytes / (e2e_max / 1e3) / 1e9
    clk = clocks.stop()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    hbm, peak_kind = measured_peaks()
    attn_bytes = attention_bytes(w)
    attn_avg_s = attn_total_ms / KA / 1e3
    achieved = attn_bytes / attn_avg_s / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": max(3, args.warmup), "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"bf16": "bf16", "f32": "f32", "i8": "i8"}[w.kv_dtype], "data": "synthetic",
        "config": {"workload": w.name, "description": W.CONFIGS[args.config],
                   "batch": w.B, "q_heads": w.Hq, "kv_heads": w.Hkv, "head_dim": w.D,
                   "block_size": w.BS, "mean_context": float(w.context_lens.mean()),
                   "max_context": maxc, "split_chunk": chunk,
                   "shared_prefix_call": bool(cascade),
                   "l2": f"flushed before every step ({L2_FLUSH_BYTES >> 20} MB write, then a "
                         f"{(L2_FLUSH_BYTES // 2) * 4 >> 20} MB read so no dirty line is left; untimed)",
                   "bytes_per_step": step_bytes, "parallelism": f"replicas x{world}",
                   "seed": rank_seed(args.config, rank)},
        "tokens_per_s": round(tokens_per_s, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "peak_kind": f"of {peak_kind}",
                     "kernel": ("paged decode attention call: " +
                                ("prefix (tcgen05) + split + merge kernels" if cascade
                                 else "split kernel + merge kernel") +
                                " (CUDA events around the call); traffic: split kernel (ncu)"),
                     "traffic": profiled_traffic(w.name),
                     "algorithmic_bytes_per_launch": attn_bytes,
                     "avg_launch_us": round(attn_avg_s * 1e6, 3), "launches_timed": KA,
                     "timed_ms": round(attn_total_ms, 2)},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": KE, "timed_ms": round(e2e_ms, 2)},
        "gpu_launches": cuda_launches_per_step(w, chunk, cascade) * K,
        "wall_s": round(wall_s, 3),
    }
    if clk is not None:
        clk["window"] = ("nvidia-smi every 100 ms from the warm-up to the end of the e2e loop "
                         "(the timed steps, the roofline loop and the e2e loop)")
        line["clocks"] = clk
    if not args.no_cpu and world == 1:
        # the last e2e step's output (the same inputs every step), against the oracle on the rows
        # the baseline leg computes anyway
        gpu_out = host_out.float().numpy()
        kept = {}
        line["cpu_baseline"] = cpu_baseline(w, keep=kept)
        line["accuracy"] = {**accuracy_vs_oracle(gpu_out, kept["out"], kept["rows"]),
                            "reference": "fp64 oracle on the cpu_baseline sample's rows",
                            "output_dtype": str(out.dtype).replace("torch.", "")}
    if world == 1 and not args.no_secondary:
        # the other workloads, each as its own record (the headline keys above stay as they are):
        # the Llama-3-8B GQA batch, the INT8 batch, the shared-prefix batch, and the paged prefill
        # over a bf16 and an INT8 cache
        del run, stage, out, status, flush_l2, write, attend
        torch.cuda.empty_cache()
        clocks2 = ClockSampler(local)
        clocks2.start()
        rec = {}
        for cfg in (2, 4, 5):
            r = measure_attention(pkv, cfg, dev, SECONDARY_LOOP_MS)
            rec[r["workload"]] = r
        for kv in ("bf16", "i8"):
            p = measure_prefill(pkv, kv, 60, 5)
            rec[p["config"]["workload"]] = {
                "metric": p["metric"], "tflops": p["value"], "ms_per_call": p["ms_per_step"],
                "peak_tflops": p["roofline"]["peak"], "frac": p["roofline"]["frac"],
                "peak_kind": p["roofline"]["peak_kind"], "calls_timed": p["steps"],
                "flops_per_call": p["config"]["flops_per_step"]}
        clk2 = clocks2.stop()
        line["secondary"] = {"note": ("separate workloads measured after the headline, each on its "
                                      "own: decode attention calls (L2 flushed before each call, at "
                                      f"least {SECONDARY_LOOP_MS:.0f} ms of GPU time) and paged "
                                      "prefill calls"),
                             "workloads": rec, "clocks": clk2}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def prefill_flops(w) -> int:
    """Algorithmic FLOPs of a causal paged prefill: per query head and row i of sequence b,
    2 * D for each visible key in Q K^T and again in P V."""
    vis = 0
    for b in range(w.B):
        L = int(w.query_start[b + 1] - w.query_start[b])
        n = int(w.context_lens[b])
        vis += sum(n - L + 1 + i for i in range(L))
    return 4 * w.D * w.Hq * vis


def run_multi(args):
    """Multi-token decode (MTP verification): every sequence of config --config gets its last L
    context positions as new query tokens, attending causally. Times the attention call
    (pkv_paged_decode_attention_multi) with a flushed L2 and reports KV GB/s against the measured
    HBM peak; the KV bytes are those of the one-token step (the L tokens share the context)."""
    import torch

    import paged_kv_decode_reshape_gb300 as pkv
    pkv.load(build_if_missing=False)
    L = args.multi
    w = W.make_multi_token(W.make_config(args.config), L, seed=3)

    def up(a):
        if a is None:
            return None
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
        return torch.from_numpy(a).cuda()
    q, kp, vp = up(w.q), up(w.k_pool), up(w.v_pool)
    ks, vs = up(w.k_scales), up(w.v_scales)
    bt, cl = up(w.block_tables), up(w.context_lens)
    out = torch.empty_like(q)
    maxc = w.max_context_len
    nb = pkv.decode_workspace_bytes(w.B * L, w.Hq, w.Hkv, w.D, maxc, args.chunk)
    ws = torch.empty(max(nb, 256), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    clean = torch.zeros(L2_FLUSH_BYTES // 2, dtype=torch.int32, device="cuda")

    def call():
        pkv.paged_decode_attention_multi(out, q, kp, vp, bt, cl, maxc, w.scale, ks, vs, args.chunk,
                                         ws, status)
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"kernels flagged bad inputs: status {int(status.item())}")
    K = max(1, min(args.steps, 500))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    clocks = ClockSampler(0)
    clocks.start()
    for k in range(K):
        flush.fill_(k & 0xFF)
        clean.max()
        ev[k][0].record()
        call()
        ev[k][1].record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    kvb = attention_bytes(W.make_config(args.config))
    gbs = kvb / (ms / 1e3) / 1e9
    hbm, peak_kind = measured_peaks()
    line = {"metric": "multi-token decode attention KV GB/s (L query tokens per sequence)",
            "value": round(gbs, 2), "unit": "GB/s", "n_gpus": 1, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": round(ms, 5), "higher_is_better": True,
            "dtype": w.kv_dtype, "data": "synthetic",
            "config": {"workload": w.name, "tokens_per_sequence": L, "batch": w.B,
                       "q_heads": w.Hq, "kv_heads": w.Hkv, "head_dim": w.D,
                       "l2": "flushed before every call (untimed)"},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": hbm, "unit": "GB/s",
                         "frac": round(gbs / hbm, 4), "peak_kind": f"of {peak_kind}"},
            "tokens_per_s": round(w.B * L / (ms / 1e3), 1)}
    if clk is not None:
        line["clocks"] = clk
    print(json.dumps(line), flush=True)


def measure_prefill(pkv, kv: str, steps: int, warmup: int) -> dict:
    """Paged chunked prefill on tcgen05: 4 sequences x 4096 new prompt tokens after 2048 cached
    tokens, Llama-3-8B heads (32 q / 8 kv, D = 128), over a bf16 or an INT8 cache. Returns the
    JSON line: TFLOP/s against the measured dense bf16 tensor peak."""
    import torch
    i8 = kv == "i8"
    w = W.make_prefill(name="prefill_llama3_8b" + ("_int8" if i8 else ""), query_lens=[4096] * 4,
                       cached_lens=[2048] * 4, Hq=32, Hkv=8, D=128, seed=7,
                       kv_dtype="i8" if i8 else "bf16")

    def up(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
        return torch.from_numpy(a).cuda()
    q, kp, vp = up(w.q), up(w.k_pool), up(w.v_pool)
    bt, cl, qs = up(w.block_tables), up(w.context_lens), up(w.query_start)
    ks = up(w.k_scales) if i8 else None
    vs = up(w.v_scales) if i8 else None
    out = torch.empty_like(q)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def step():
        if i8:
            pkv.paged_prefill_attention_int8(out, q, kp, vp, ks, vs, bt, cl, qs, w.max_query_len, w.scale)
        else:
            pkv.paged_prefill_attention(out, q, kp, vp, bt, cl, qs, w.max_query_len, w.scale)
    for _ in range(max(3, warmup)):
        step()
    torch.cuda.synchronize()
    K = max(1, min(steps, 200))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    clocks = ClockSampler(0)
    clocks.start()
    clean = torch.zeros(L2_FLUSH_BYTES // 2, dtype=torch.int32, device="cuda")
    for k in range(K):
        flush.fill_(k & 0xFF)
        clean.max()
        ev[k][0].record()
        step()
        ev[k][1].record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    flops = prefill_flops(w)
    tflops = flops / (ms / 1e3) / 1e12
    peak = 1925.2
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            peak = float(json.load(f).get("bf16_tflops", peak))
    line = {"metric": "paged prefill attention TFLOP/s (causal, tcgen05)" + (", INT8 KV cache" if i8 else ""),
            "value": round(tflops, 2),
            "unit": "TFLOP/s", "n_gpus": 1, "steps": K, "warmup": max(3, warmup),
            "ms_per_step": round(ms, 4), "higher_is_better": True, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.name, "sequences": w.B, "new_tokens": 4096, "cached_tokens": 2048,
                       "q_heads": w.Hq, "kv_heads": w.Hkv, "head_dim": w.D, "flops_per_step": flops,
                       "l2": "flushed before every step (untimed)"},
            "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                         "peak_kind": "of measured (cuBLAS bf16 burst)"},
            "tokens_per_s": round(int(w.query_start[-1]) / (ms / 1e3), 1)}
    if clk is not None:
        line["clocks"] = clk
    del q, kp, vp, out, flush, clean
    torch.cuda.empty_cache()
    return line


def run_prefill(args):
    import paged_kv_decode_reshape_gb300 as pkv
    pkv.load(build_if_missing=False)
    print(json.dumps(measure_prefill(pkv, getattr(args, "prefill_kv", "bf16"), args.steps, args.warmup)),
          flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=8000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG, choices=sorted(W.CONFIGS))
    ap.add_argument("--chunk", type=int, default=0, help="split chunk in tokens (0 = auto)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle cpu_baseline leg")
    ap.add_argument("--min-loop-ms", type=float, default=MIN_LOOP_MS,
                    help="GPU time the roofline and e2e loops run at least (0: exactly --steps "
                         "iterations each, e.g. under a profiler)")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the secondary workloads (configs 2, 4, 5 and the paged prefill) "
                         "measured after the headline and reported in its line")
    ap.add_argument("--no-cascade", action="store_true",
                    help="run a shared-prefix workload through the plain decode call instead of "
                         "the shared-prefix (cascade) call")
    ap.add_argument("--multi", type=int, default=0, metavar="L",
                    help="time multi-token decode (L new tokens per sequence, e.g. MTP "
                         "verification) on the chosen config instead of the decode step")
    ap.add_argument("--prefill", action="store_true",
                    help="time the paged prefill kernel instead of the decode step")
    ap.add_argument("--prefill-kv", choices=["bf16", "i8"], default="bf16",
                    help="K/V cache type of the --prefill workload")
    args = ap.parse_args(argv)
    if args.prefill:
        run_prefill(args)
    elif args.multi:
        run_multi(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
