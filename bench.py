"""Benchmark of the three sequence-head relayouts on GB300.

One step = QKV destination pack + attention-result split + returned-head
merge over one batch of synthetic input at the pages' shape (T=55,414,
H=28, D=128, P=2, C=4, bf16 moved as raw 16-bit patterns; pack source with
row stride 3*H*D+64, split source head-major).  The metric is effective HBM
GB/s: algorithmic bytes read + written (2 x elements moved x 2 B) over time.

Default arm: the CUDA library.  W untimed warm-up steps, then exactly K steps
bracketed by a barrier and a device synchronise, timed with CUDA events on
the launching stream (max over ranks), inputs larger than L2 and two
rotating buffer sets.  The JSON line also carries the per-op breakdown, the
roofline of the dominant kernel, the SM clocks sampled during the timed
region, an end-to-end figure through the public API with pinned host buffers
(host-to-device copies of the inputs and device-to-host copies of the
outputs inside the timed region), and the CPU oracle timed on host cores.

``--impl reference``: the CPU oracle, unmodified, on the host cores, timed
on a bounded token sample of the same workload each step.

Several GPUs (torchrun): every rank runs an independent replica of the
workload on its own GPU (the relayouts have no exchange step on one rank);
``value`` is the bytes of all ranks over the slowest rank's time.
"""
import argparse
import hashlib
import json
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "effective HBM GB/s (read+write) and % of GB300 peak per relayout op"
UNIT = "GB/s"
WORKLOAD = "pages"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900
# what the GPU executes: the kernel and its launch policy (not the ABI's checks)
KERNEL_SOURCES = ["sequence_head_relayout_gb300/csrc/relayout_kernel.cuh",
                  "sequence_head_relayout_gb300/csrc/launch.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic_pages.txt")


def kernel_source_hash() -> str:
    """Hash of the kernel sources with comments and whitespace removed, so that
    a recorded ncu traffic figure stays attached to the code it measured."""
    import re
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def max_over_ranks(x: float, device="cpu") -> float:
    """Maximum of a per-rank scalar over all ranks (identity on one rank)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: the bytes every rank moved over the slowest rank's time."""
    return world * steps * bytes_per_rank_step / (max_ms / 1e3) / 1e9


def op_elements(cfg):
    T, H, D = cfg.T, cfg.H, cfg.D
    return {"qkv_pack": 3 * T * H * D, "attn_split": T * H * D, "head_merge": T * H * D,
            "qkv_unpack": 3 * T * (H // cfg.P) * D}


def alg_bytes(elems: int) -> int:
    return 2 * 2 * elems            # read once + written once, 2 bytes each


def lossy_bytes(elems: int, D: int) -> int:
    """Lossy transport: 2 B bf16 + 1 B code per element, plus one 4 B scale
    per D-element head row (read or written once each)."""
    return 3 * elems + 4 * (elems // D)


# ----------------------------------------------------------------------------
# CPU oracle (reported baseline and reference arm); runs in spawned workers
# ----------------------------------------------------------------------------

def _oracle_inputs(T, H, D, pad, seed):
    import numpy as np
    rng = np.random.default_rng(seed)
    return {
        "pack_src": rng.integers(0, 1 << 16, size=T * (3 * H * D + pad), dtype=np.uint16),
        "split_src": rng.integers(0, 1 << 16, size=T * H * D, dtype=np.uint16),  # [H][T][D]
        "merge_src": rng.integers(0, 1 << 16, size=T * H * D, dtype=np.uint16),
        "pack_dst": np.empty(3 * T * H * D, dtype=np.uint16),
        "split_dst": np.empty(T * H * D, dtype=np.uint16),
        "merge_dst": np.empty(T * H * D, dtype=np.uint16),
    }


def _oracle_proc(rank, shape, passes, barrier, results):
    """One host core: build a token sample of the workload once, then run the
    C oracle's pack, split and merge over it `passes` times, each pass
    started together with the other processes (barrier) and timed alone."""
    import ctypes

    from oracle import build
    T, H, D, P, C, pad = shape
    lib = ctypes.CDLL(build.LIB)
    I64 = ctypes.c_int64
    x = _oracle_inputs(T, H, D, pad, 1000 + rank)
    ptr = {k: ctypes.c_void_p(v.ctypes.data) for k, v in x.items()}
    ps = (I64 * 4)(3 * H * D + pad, H * D, D, 1)
    ss = (I64 * 3)(D, T * D, 1)
    ms = (I64 * 3)(H * D, D, 1)
    dims = (I64(T), I64(H), I64(D), I64(P), I64(C))
    for f in (lib.oracle_qkv_pack, lib.oracle_attn_split, lib.oracle_head_merge):
        f.restype = I64
    times = []
    for _ in range(passes):
        barrier.wait()
        t0 = time.perf_counter()
        lib.oracle_qkv_pack(ptr["pack_src"], ps, *dims, ptr["pack_dst"])
        lib.oracle_attn_split(ptr["split_src"], ss, *dims, ptr["split_dst"])
        lib.oracle_head_merge(ptr["merge_src"], *dims, ptr["merge_dst"], ms)
        times.append(time.perf_counter() - t0)
    results.put((rank, times))


def _collect(results, n: int, procs, timeout_s: float = 900.0):
    """n results from spawned workers; raises if a worker died or the
    results do not arrive within timeout_s."""
    import queue
    got, t0 = [], time.monotonic()
    while len(got) < n:
        try:
            got.append(results.get(timeout=2.0))
        except queue.Empty:
            dead = [pr.exitcode for pr in procs if pr.exitcode not in (None, 0)]
            if dead or time.monotonic() - t0 > timeout_s:
                for pr in procs:
                    if pr.is_alive():
                        pr.terminate()
                raise RuntimeError("CPU oracle workers failed (exit codes %s)" % dead)
    return got


def run_oracle(cfg, tokens: int, passes: int, cores: int):
    """Per-pass times (the slowest core's) of `cores` processes, each moving
    its own `tokens`-token sample; and the bytes all cores move per pass."""
    from oracle import build
    build.build()
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(cores)
    results = ctx.Queue()
    shape = (tokens, cfg.H, cfg.D, cfg.P, cfg.C, cfg.pad)
    procs = [ctx.Process(target=_oracle_proc, args=(r, shape, passes, barrier, results))
             for r in range(cores)]
    for pr in procs:
        pr.start()
    got = _collect(results, cores, procs)
    for pr in procs:
        pr.join()
    per_pass = [max(t[i] for _, t in got) for i in range(passes)]
    return per_pass, cores * alg_bytes(5 * tokens * cfg.H * cfg.D)


SAMPLE_BYTES_PER_CORE = 1 << 30        # host memory one oracle process may hold


def calibrate_tokens(cfg, seconds_per_pass: float):
    """Token count whose oracle pass takes about `seconds_per_pass` on a core,
    within SAMPLE_BYTES_PER_CORE of inputs and outputs; and the estimated
    seconds of one pass at that count."""
    probe = min(cfg.T, 2048)
    times, _ = run_oracle(cfg, probe, 2, 1)
    per_token = max(min(times) / probe, 1e-9)
    bytes_per_token = 2 * ((3 * cfg.H * cfg.D + cfg.pad) + 5 * cfg.H * cfg.D + 2 * cfg.H * cfg.D)
    cap = max(16, SAMPLE_BYTES_PER_CORE // bytes_per_token)
    tokens = int(max(16, min(cfg.T, cap, seconds_per_pass / per_token)))
    return tokens, tokens * per_token


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def lossy_cpu_baseline(cfg, tokens: int = 2048, passes: int = 2):
    """The lossy-transport oracle on one host core, on a token sample of the
    workload: GB/s per op with the lossy byte count (3 B per element + 4 B
    per head row), best of `passes`."""
    import torch

    from oracle import loops
    from sequence_head_relayout_gb300 import workloads as W
    T, H, D, P, C = min(tokens, cfg.T), cfg.H, cfg.D, cfg.P, cfg.C
    x4 = W.finite_rows_(torch.empty((T, 3, H, D), dtype=torch.int16), 1)
    x3 = W.finite_rows_(torch.empty((T, H, D), dtype=torch.int16), 2)
    ops = {}

    def timed(name, elems, fn):
        best = min(_wall(fn) for _ in range(passes))
        ops[name] = round(lossy_bytes(elems, D) / best / 1e9, 3)

    codes, scales = loops.qkv_pack_q(x4, P, C, loops.INT8)
    fcodes, fscales = loops.attn_split_q(x3, P, C, loops.E4M3)
    n_unpack = 3 * T * (H // P) * D
    timed("qkv_pack_int8", 3 * T * H * D, lambda: loops.qkv_pack_q(x4, P, C, loops.INT8))
    timed("qkv_unpack_int8", n_unpack, lambda: loops.qkv_unpack_q(
        codes[:n_unpack], scales[:n_unpack // D], T, H, D, P, C, loops.INT8))
    timed("attn_split_e4m3", T * H * D, lambda: loops.attn_split_q(x3, P, C, loops.E4M3))
    timed("head_merge_e4m3", T * H * D, lambda: loops.head_merge_q(
        fcodes, fscales, T, H, D, P, C, loops.E4M3))
    return {"unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "%d of %d tokens (H=%d, D=%d, P=%d, C=%d), finite bf16 rows, best of %d"
                      % (T, cfg.T, H, D, P, C, passes),
            "ops": ops}


def _wall(fn) -> float:
    t0 = time.perf_counter()
    fn()
    return time.perf_counter() - t0


def cpu_baseline(cfg, budget_s: float = 10.0, cores: int = None):
    """The oracle on all host cores for about budget_s of wall time, then on
    one core (two passes of the same per-core sample)."""
    cores = cores or os.cpu_count() or 1
    tokens, est = calibrate_tokens(cfg, budget_s / 3)
    passes = int(max(3, min(30, budget_s / max(est, 1e-3))))
    per_pass, nbytes = run_oracle(cfg, tokens, passes, cores)
    total = sum(per_pass)
    one, one_bytes = run_oracle(cfg, tokens, 3, 1)
    return {"value": round(nbytes / statistics.median(per_pass) / 1e9, 3), "unit": UNIT,
            "cores": cores, "kind": "oracle",
            "single_core_value": round(one_bytes / statistics.median(one) / 1e9, 3),
            "cpu_model": cpu_model(),
            "statistic": "median pass",
            "sample": "%d of %d tokens (H=%d, D=%d, P=%d, C=%d, padded-row pack source, "
                      "head-major split source) per core, one process per core, %d timed "
                      "passes of pack+split+merge started together, %.1f s; single core: "
                      "3 passes of the same sample"
                      % (tokens, cfg.T, cfg.H, cfg.D, cfg.P, cfg.C, passes, total)}


CPU_OPS = ("qkv_pack", "attn_split", "head_merge", "qkv_unpack")
CPU_SAMPLE_BYTES = 256 << 20     # inputs + outputs of the four ops held by one process
CPU_MIN_PASS_ELEMS = 1 << 22     # elements one timed pass moves at least (repeating the op)


def cpu_sample_tokens(cfg, cap_bytes: int = CPU_SAMPLE_BYTES) -> int:
    """Tokens of a per-process sample of `cfg`: the whole workload when its
    four ops' inputs and outputs fit in cap_bytes, else the first tokens that
    do."""
    H, D, Hp = cfg.H, cfg.D, cfg.H // cfg.P
    per_token = 2 * ((3 * H * D + cfg.pad) + 3 * H * D + 4 * H * D + 6 * Hp * D)
    return int(max(1, min(cfg.T, cap_bytes // per_token)))


def _cpu_op_inputs(shape, T, seed):
    """numpy buffers and element strides of the four ops on a T-token sample,
    in the workload's own layouts (padded or head-major pack source,
    head-major split source, head-major merge destination)."""
    import numpy as np
    H, D, P, C, pad, pack_src, split_src, merge_dst = shape
    Hp = H // P
    rng = np.random.default_rng(seed)

    def bits(n):
        return rng.integers(0, 1 << 16, size=n, dtype=np.uint16)

    row = 3 * H * D + pad
    x = {"pack_src": bits(T * row), "pack_dst": np.empty(3 * T * H * D, np.uint16),
         "split_src": bits(T * H * D), "split_dst": np.empty(T * H * D, np.uint16),
         "merge_src": bits(T * H * D), "merge_dst": np.empty(T * H * D, np.uint16),
         "recv": bits(3 * T * Hp * D)}
    for k in ("q", "k", "v"):
        x[k] = np.empty(T * Hp * D, np.uint16)
    st = {"pack": (row, H * D, D, 1) if pack_src != "head_major" else (row, D, 3 * D, 1),
          "split": (D, T * D, 1) if split_src == "bhtd" else (H * D, D, 1),
          "merge": (D, T * D, 1) if merge_dst == "head_major" else (H * D, D, 1),
          "unpack": (Hp * D, D, 1)}
    return x, st


def _cpu_op_worker(rank, tasks, barrier, results):
    """One host process: for every task (a workload sample), build its inputs
    once, then time each op `passes` times, every pass started together with
    the other processes (barrier)."""
    import ctypes

    from oracle import build
    lib = ctypes.CDLL(build.LIB)
    I64 = ctypes.c_int64
    for f in (lib.oracle_qkv_pack, lib.oracle_attn_split, lib.oracle_head_merge,
              lib.oracle_qkv_unpack_recv):
        f.restype = I64
    while True:
        task = tasks.get()
        if task is None:
            return
        key, shape, T, passes, reps = task
        H, D, P, C = shape[:4]
        x, st = _cpu_op_inputs(shape, T, 5000 + rank)
        ptr = {k: ctypes.c_void_p(v.ctypes.data) for k, v in x.items()}
        arr = {k: (I64 * len(v))(*v) for k, v in st.items()}
        dims = (I64(T), I64(H), I64(D), I64(P), I64(C))
        run = {
            "qkv_pack": lambda: lib.oracle_qkv_pack(ptr["pack_src"], arr["pack"], *dims,
                                                    ptr["pack_dst"]),
            "attn_split": lambda: lib.oracle_attn_split(ptr["split_src"], arr["split"], *dims,
                                                        ptr["split_dst"]),
            "head_merge": lambda: lib.oracle_head_merge(ptr["merge_src"], *dims,
                                                        ptr["merge_dst"], arr["merge"]),
            "qkv_unpack": lambda: lib.oracle_qkv_unpack_recv(ptr["recv"], *dims, ptr["q"],
                                                             ptr["k"], ptr["v"], arr["unpack"]),
        }
        times = {}
        for op in CPU_OPS:
            times[op] = []
            for _ in range(passes):
                barrier.wait()
                t0 = time.perf_counter()
                for _ in range(reps[op]):
                    n = run[op]()
                times[op].append(time.perf_counter() - t0)
                if n < 0:
                    raise RuntimeError("oracle %s rejected the sample" % op)
        del x, ptr
        results.put((rank, key, times))


def cpu_per_config(names, cores: int = None, passes: int = 3):
    """The C oracle, unmodified, timed per op at every workload: on all host
    cores (one spawned process per core, each moving its own sample, every
    pass started together; a pass takes the slowest process's time) and on one
    core; median of `passes`.  GB/s counts the same algorithmic bytes as the
    GPU figures (4 B per element moved), summed over processes."""
    from oracle import build
    from sequence_head_relayout_gb300 import workloads as W
    build.build()
    cores = cores or os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    table = {name: {} for name in names}
    samples = {}
    t_all = time.perf_counter()
    for nproc in (cores, 1):
        barrier = ctx.Barrier(nproc)
        tasks, results = ctx.Queue(), ctx.Queue()
        procs = [ctx.Process(target=_cpu_op_worker, args=(r, tasks, barrier, results))
                 for r in range(nproc)]
        for pr in procs:
            pr.start()
        for name in names:
            cfg = W.CONFIGS[name]
            T = cpu_sample_tokens(cfg)
            samples[name] = T
            shape = (cfg.H, cfg.D, cfg.P, cfg.C, cfg.pad, cfg.pack_src, cfg.split_src,
                     cfg.merge_dst)
            sample_cfg = W.Config(name, T, cfg.H, cfg.D, cfg.P, cfg.C)
            elems = op_elements(sample_cfg)
            # small samples repeat the op inside a pass (about 4 M elements moved)
            reps = {op: max(1, CPU_MIN_PASS_ELEMS // max(1, elems[op])) for op in CPU_OPS}
            for _ in range(nproc):
                tasks.put((name, shape, T, passes, reps))
            got = _collect(results, nproc, procs)
            for op in CPU_OPS:
                per_pass = [max(t[op][i] for _, _, t in got) for i in range(passes)]
                med = statistics.median(per_pass)
                gbs = nproc * reps[op] * alg_bytes(elems[op]) / med / 1e9
                key = "cpu_gbs" if nproc == cores else "cpu_gbs_1core"
                table[name].setdefault(op, {})[key] = round(gbs, 3)
        for _ in range(nproc):
            tasks.put(None)
        for pr in procs:
            pr.join()
    desc = {name: "%d of %d tokens per process%s" % (samples[name], W.CONFIGS[name].T,
                                                    "" if samples[name] == W.CONFIGS[name].T
                                                    else " (sampled)")
            for name in names}
    return {"cores": cores, "cpu_model": cpu_model(), "kind": "oracle",
            "statistic": "median of %d passes; an all-core pass is timed from a common "
                         "start to the slowest process's end" % passes,
            "parallelism": "one spawned process per core, each moving its own sample "
                           "(the oracle has no threading of its own)",
            "sample": desc, "seconds": round(time.perf_counter() - t_all, 1),
            "table": table}


# ----------------------------------------------------------------------------
# Clocks sampled during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(self.REASONS, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for key in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
            if key in d and d[key]:
                return float(d[key]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic():
    """ncu DRAM bytes per launch (read + write) recorded for the current kernel
    source, as {op: bytes}; None when absent or taken on other kernel code."""
    d = {}
    try:
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if line.startswith("#") or ":" not in line:
                    continue
                k, _, v = line.partition(":")
                d[k.strip()] = v.strip()
    except OSError:
        return None
    if d.get("kernel_source_sha") != kernel_source_hash():
        return None
    return {k: int(v) for k, v in d.items() if k in ("qkv_pack", "attn_split", "head_merge")}


def make_set(cfg, dev, seed_shift, ops=("qkv_pack", "attn_split", "head_merge")):
    import torch

    from sequence_head_relayout_gb300 import workloads as W
    n = op_elements(cfg)
    s = {}
    if "qkv_pack" in ops:
        s["pack_src"], s["pack_base"] = W.pack_source(cfg, device=dev, seed=cfg.seed + seed_shift)
        s["pack_dst"] = torch.empty(n["qkv_pack"], dtype=torch.int16, device=dev)
    if "attn_split" in ops:
        s["split_src"], s["split_base"] = W.split_source(cfg, device=dev,
                                                         seed=cfg.seed + seed_shift)
        s["split_dst"] = torch.empty(n["attn_split"], dtype=torch.int16, device=dev)
    if "head_merge" in ops:
        s["merge_src"] = W.merge_source(cfg, device=dev, seed=cfg.seed + seed_shift)
        s["merge_dst"] = torch.empty((cfg.T, cfg.H, cfg.D), dtype=torch.int16, device=dev)
    if "qkv_unpack" in ops:
        Hp = cfg.H // cfg.P
        s["recv"] = torch.empty(3 * cfg.T * Hp * cfg.D, dtype=torch.int16, device=dev)
        W.fill_(s["recv"], cfg.payload, cfg.seed + seed_shift + 3000)
        s["qkv_out"] = tuple(torch.empty((cfg.T, Hp, cfg.D), dtype=torch.int16, device=dev)
                             for _ in range(3))
    return s


def run_op(vf, cfg, s, name):
    """Enqueue one relayout of the step on the current stream."""
    if name == "qkv_pack":
        vf.qkv_pack(s["pack_src"], cfg.P, cfg.C, out=s["pack_dst"])
    elif name == "attn_split":
        vf.attn_split(s["split_src"], cfg.P, cfg.C, out=s["split_dst"])
    elif name == "head_merge":
        vf.head_merge(s["merge_src"], cfg.T, cfg.H, cfg.D, cfg.P, cfg.C, out=s["merge_dst"])
    else:
        vf.qkv_unpack(s["recv"], cfg.T, cfg.H, cfg.D, cfg.P, cfg.C, outs=s["qkv_out"])


def back_to_back(vf, cfg, sets, ops_run, launches: int = 100, reps: int = 3):
    """Per op: `launches` launches of that op alone, back to back on the
    rotating buffer sets, with events only before the first and after the
    last, so consecutive launches overlap as they do in the timed step; the
    median over `reps` of total / launches, in microseconds."""
    import torch
    out = {}
    for name in ops_run:
        ts = []
        for rep in range(reps + 1):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            for i in range(launches):
                run_op(vf, cfg, sets[i % len(sets)], name)
            b.record()
            if rep:
                ts.append((a, b))
        torch.cuda.synchronize()
        out[name] = statistics.median(x.elapsed_time(y) for x, y in ts) * 1e3 / launches
    return out


def run_step(vf, cfg, s, events=None):
    """Enqueue the step's relayouts; events[i] is recorded before op i and
    events[-1] after the last one."""
    k = 0
    if events:
        events[0].record()
    if "pack_src" in s:
        vf.qkv_pack(s["pack_src"], cfg.P, cfg.C, out=s["pack_dst"])
        k += 1
        if events:
            events[k].record()
    if "split_src" in s:
        vf.attn_split(s["split_src"], cfg.P, cfg.C, out=s["split_dst"])
        k += 1
        if events:
            events[k].record()
    if "merge_src" in s:
        vf.head_merge(s["merge_src"], cfg.T, cfg.H, cfg.D, cfg.P, cfg.C, out=s["merge_dst"])
        k += 1
        if events:
            events[k].record()
    if "recv" in s:
        vf.qkv_unpack(s["recv"], cfg.T, cfg.H, cfg.D, cfg.P, cfg.C, outs=s["qkv_out"])
        k += 1
        if events:
            events[k].record()


def split_per_chunk_calls(vf, cfg, s, reps=50):
    """The attention-result split issued as one call per overlap chunk (as
    the pages timed it, and as an overlap pipeline issues it): the median of
    C back-to-back chunk calls, divided by C, in microseconds."""
    import torch
    ts = []
    for rep in range(reps + 3):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for c in range(cfg.C):
            vf.attn_split(s["split_src"], cfg.P, cfg.C, out=s["split_dst"], chunks=(c, 1))
        b.record()
        if rep >= 3:
            ts.append((a, b))
    torch.cuda.synchronize()
    return round(statistics.median(x.elapsed_time(y) for x, y in ts) * 1e3 / cfg.C, 2)


def launches_per_step(cfg, ops) -> int:
    """Kernel launches of one step: one per 128 pieces; a piece is one (chunk,
    destination) block, times the q/k/v slabs for the pack and the unpack."""
    per_launch = 128
    slabs = {"qkv_pack": 3, "qkv_unpack": 3, "attn_split": 1, "head_merge": 1}
    return sum(-(-slabs[o] * cfg.P * cfg.C // per_launch) for o in ops)


def gpu_arm(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import sequence_head_relayout_gb300 as vf
    from sequence_head_relayout_gb300 import workloads as W

    cfg = W.CONFIGS[args.config]
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    vf.lib()

    order = ("qkv_pack", "attn_split", "head_merge", "qkv_unpack")
    ops_run = tuple(o for o in order[:3] if not args.only) or tuple(
        o for o in order if o in args.only)
    sets = [make_set(cfg, dev, 17 * i, ops_run) for i in range(args.sets)]
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    K = args.steps
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    # the clock sampler needs a moment to start; the warm-up steps come after
    # that pause, right before the timed region, so that it starts warm
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    for i in range(args.warmup):
        run_step(vf, cfg, sets[i % len(sets)])
    barrier()
    start.record()
    for i in range(K):
        run_step(vf, cfg, sets[i % len(sets)])
    end.record()
    barrier()
    # Per-op durations: an instrumented pass right after the timed region, with
    # events around every op of every step (events between two kernels stop
    # the next launch from overlapping the previous one's tail, so the timed
    # region itself carries none).  Its first step is dropped; medians.
    n_ev = max(50, args.event_steps) + 1
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ops_run) + 1)]
          for _ in range(n_ev)]
    for i in range(n_ev):
        run_step(vf, cfg, sets[i % len(sets)], ev[i])
    torch.cuda.synchronize()
    clock_info = clocks.stop()

    b2b = back_to_back(vf, cfg, sets, ops_run)

    total_ms = start.elapsed_time(end)
    per_op_ms = {name: [e[j].elapsed_time(e[j + 1]) for e in ev[1:]]
                 for j, name in enumerate(ops_run)}
    inst_step_ms = [e[0].elapsed_time(e[-1]) for e in ev[1:]]

    max_ms = max_over_ranks(total_ms, dev)

    elems = op_elements(cfg)
    step_bytes = sum(alg_bytes(elems[n]) for n in ops_run)
    value = job_gbs(step_bytes, K, world, max_ms)
    peak, peak_kind = measured_peak()

    step_us = max_ms / K * 1e3
    ops = {}
    for name, ts in per_op_ms.items():
        med = statistics.median(ts)
        b = alg_bytes(elems[name])
        gbs = b / (med / 1e3) / 1e9
        ops[name] = {"bytes": b, "median_us": round(med * 1e3, 2),
                     "mean_us": round(statistics.fmean(ts) * 1e3, 2),
                     "min_us": round(min(ts) * 1e3, 2),
                     "p90_us": round(sorted(ts)[int(0.9 * (len(ts) - 1))] * 1e3, 2),
                     "samples": len(ts),
                     "gbs": round(gbs, 1),
                     "frac_of_peak": round(gbs / peak, 4),
                     "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
                     "share_of_step": round(med * 1e3 / step_us, 4),
                     "back_to_back_us": round(b2b[name], 2),
                     "back_to_back_gbs": round(b / (b2b[name] / 1e6) / 1e9, 1)}
    if "attn_split" in ops:
        ops["attn_split"]["per_chunk_call_us"] = split_per_chunk_calls(vf, cfg, sets[0])
    inst_med = statistics.median(inst_step_ms) * 1e3
    per_op_summary = {
        "method": "events around every op of %d instrumented steps run right after the "
                  "timed region (first dropped); medians" % (n_ev - 1),
        "instrumented_step_us": round(inst_med, 2),
        "sum_of_op_medians_us": round(sum(o["median_us"] for o in ops.values()), 2),
        "back_to_back": "per op, 100 launches of that op alone on the rotating sets, events "
                        "only at the ends (launches overlap as in the timed step); median "
                        "of 3 of total / 100",
        "sum_of_back_to_back_us": round(sum(b2b.values()), 2),
        "timed_step_us": round(step_us, 2),
        "note": "the timed region has no events between ops, so consecutive launches "
                "overlap (programmatic dependent launch) and its step is shorter than "
                "an instrumented one; the back-to-back figures keep that overlap"}

    dominant = max(ops_run, key=lambda k: statistics.median(per_op_ms[k]))
    dom_s = statistics.median(per_op_ms[dominant]) / 1e3
    achieved = alg_bytes(elems[dominant]) / dom_s / 1e9
    traffic = recorded_traffic()
    roofline = {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 1),
                "peak": peak, "peak_source": peak_kind, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "nominal_peak": NOMINAL_HBM_GBS,
                "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                "traffic": (traffic or {}).get(dominant),
                "algorithmic_bytes": alg_bytes(elems[dominant]),
                "duration_us": round(dom_s * 1e6, 2),
                "duration_stat": per_op_summary["method"],
                "share_of_step": round(dom_s * 1e6 / step_us, 4)}
    target = None
    if cfg.name == "pages":
        worst = min(ops[o]["frac_of_nominal"] for o in ("qkv_pack", "attn_split", "head_merge")
                    if o in ops)
        target = {"rule": "each relayout sustains >= 0.80 of GB300 HBM peak at the pages' "
                          "shape",
                  "judged_against": "the nominal %d GB/s (the stricter of the two; the "
                                    "measured copy peak is %.1f GB/s)" % (NOMINAL_HBM_GBS, peak),
                  "worst_op_frac_of_nominal": worst, "met": worst >= 0.80}

    e2e = None
    if not args.no_e2e and not args.only:
        del sets
        torch.cuda.empty_cache()
        e2e = e2e_arm(args, cfg, dev, world)

    configs = per_config(args, dev) if args.configs else None
    lossy = None
    if configs and cfg.name in configs["table"]:
        row = configs["table"][cfg.name]
        lossy = {k: row[k] for k in ("qkv_pack_int8", "qkv_unpack_int8", "attn_split_e4m3",
                                     "head_merge_e4m3")}
        lossy["note"] = ("opt-in INT8 QKV / E4M3 attention-output transport at the bench "
                         "workload; GB/s counts 3 B per element + 4 B per head row")
        lossy["quality"] = lossy_quality(dev)
    chain_aba = None if args.no_chain else torch_chain_aba(cfg, dev)

    line = None
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(max_ms / K, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16 bit patterns)",
            "config": {"workload": "%s: T=%d H=%d D=%d P=%d C=%d" % (cfg.name, cfg.T, cfg.H,
                                                                    cfg.D, cfg.P, cfg.C),
                       "pack_source": "row stride %d elements (3*H*D+%d)" % (
                           3 * cfg.H * cfg.D + cfg.pad, cfg.pad),
                       "split_source": "head-major [H,T,D] viewed as [T,H,D]",
                       "merge_destination": "contiguous [T,H,D]",
                       "step": " + ".join(ops_run),
                       "kernel_source_sha": kernel_source_hash(),
                       "l2": "inputs larger than L2 (each op reads >= 397 MB), "
                             "%d rotating buffer set(s)" % args.sets,
                       "per_op_events": "%d instrumented steps after the timed region"
                                        % (n_ev - 1),
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "ops": ops,
            "per_op_timing": per_op_summary,
            "target": target,
            "roofline": roofline,
            "clocks": clock_info,
            "gpu_launches": K * launches_per_step(cfg, ops_run),
            "e2e": e2e,
            "per_config": configs,
            "lossy_transport": lossy,
            "vs_torch_chain": chain_aba,
        }
    return line


def e2e_arm(args, cfg, dev, world):
    """Same metric through the public API from pinned host buffers.

    Every step copies its inputs host->device, runs the three relayouts and
    copies the outputs device->host.  The step is pipelined over the C overlap
    chunks on three streams (copy in, relayout, copy out) with the chunk-range
    entry points, so the two copy directions and the kernels overlap; events
    order chunk c of step i+1 after chunk c of step i.  A serial variant (one
    stream, whole tensors) is reported beside it."""
    import torch

    import sequence_head_relayout_gb300 as vf

    T, H, D, P, C = cfg.T, cfg.H, cfg.D, cfg.P, cfg.C
    d = make_set(cfg, dev, 33)
    keys_in = ("pack_base", "split_base", "merge_src")
    keys_out = ("pack_dst", "split_dst", "merge_dst")
    host = {k: torch.empty(d[k].shape, dtype=torch.int16, pin_memory=True)
            for k in keys_in + keys_out}
    for k in keys_in:
        host[k].copy_(d[k])
    torch.cuda.synchronize()
    h2d = sum(host[k].numel() * 2 for k in keys_in)
    d2h = sum(host[k].numel() * 2 for k in keys_out)

    def token_major(dv, hv):
        """Buffers whose outermost axis is the token: rows [t0, t1)."""
        a, b = dv.view(T, -1), hv.view(T, -1)
        return lambda t0, t1: [(a[t0:t1], b[t0:t1])]

    def head_major(dv, hv):
        """[X, T, D] buffers: rows [t0, t1) of every head plane."""
        a, b = dv.view(-1, T, D), hv.view(-1, T, D)
        return lambda t0, t1: [(a[x, t0:t1], b[x, t0:t1]) for x in range(a.shape[0])]

    pack_in = token_major(d["pack_base"], host["pack_base"])
    split_in = (head_major if cfg.split_src == "bhtd" else token_major)(d["split_base"],
                                                                         host["split_base"])
    merge_out = token_major(d["merge_dst"], host["merge_dst"])    # make_set: contiguous
    pk = vf.piece_table(vf.OP_QKV_PACK, T, H, D, P, C)
    sp = vf.piece_table(vf.OP_ATTN_SPLIT, T, H, D, P, C)
    mg = vf.piece_table(vf.OP_HEAD_MERGE, T, H, D, P, C)

    def slab(table, c, total):
        a = table[2][c * P]
        b = table[2][(c + 1) * P] if c + 1 < C else total
        return a, b

    n_pack, n_split = d["pack_dst"].numel(), d["split_dst"].numel()
    n_merge = d["merge_src"].numel()
    s_in, s_k, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    done_k = [None] * C       # relayout of chunk c finished (inputs free)
    done_out = [None] * C     # copy-out of chunk c finished (outputs free)

    def pipelined_step():
        for c in range(C):
            t0 = mg[0][c * P]
            t1 = t0 + mg[1][c * P]
            with torch.cuda.stream(s_in):
                if done_k[c] is not None:
                    s_in.wait_event(done_k[c])
                for dv, hv in pack_in(t0, t1):
                    dv.copy_(hv, non_blocking=True)
                for p in range(P):
                    e = c * P + p
                    for dv, hv in split_in(sp[0][e], sp[0][e] + sp[1][e]):
                        dv.copy_(hv, non_blocking=True)
                a, b = slab(mg, c, n_merge)
                d["merge_src"][a:b].copy_(host["merge_src"][a:b], non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(s_in)
            s_k.wait_event(ready)
            if done_out[c] is not None:
                s_k.wait_event(done_out[c])
            vf.qkv_pack(d["pack_src"], P, C, out=d["pack_dst"], stream=s_k, chunks=(c, 1))
            vf.attn_split(d["split_src"], P, C, out=d["split_dst"], stream=s_k, chunks=(c, 1))
            vf.head_merge(d["merge_src"], T, H, D, P, C, out=d["merge_dst"], stream=s_k,
                          chunks=(c, 1))
            done_k[c] = torch.cuda.Event()
            done_k[c].record(s_k)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done_k[c])
                a, b = slab(pk, c, n_pack)
                host["pack_dst"][a:b].copy_(d["pack_dst"][a:b], non_blocking=True)
                a, b = slab(sp, c, n_split)
                host["split_dst"][a:b].copy_(d["split_dst"][a:b], non_blocking=True)
                for dv, hv in merge_out(t0, t1):
                    hv.copy_(dv, non_blocking=True)
                done_out[c] = torch.cuda.Event()
                done_out[c].record(s_out)

    def serial_step():
        for k in keys_in:
            d[k].copy_(host[k], non_blocking=True)
        run_step(vf, cfg, d)
        for k in keys_out:
            host[k].copy_(d[k], non_blocking=True)

    step_bytes = sum(alg_bytes(op_elements(cfg)[x])
                     for x in ("qkv_pack", "attn_split", "head_merge"))
    n = max(3, min(args.steps, 20))

    def timed(step, streams):
        for _ in range(2):
            step()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(streams[0])
        for st in streams[1:]:
            st.wait_event(a)
        for _ in range(n):
            step()
        for st in streams[:-1]:
            ev = torch.cuda.Event()
            ev.record(st)
            streams[-1].wait_event(ev)
        b.record(streams[-1])
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    # zero copy: the kernels read the pinned host inputs and write the pinned
    # host outputs directly over the host link, one pass, no staging copies
    def host_view(dev_view, base):
        return torch.as_strided(host[base], dev_view.size(), dev_view.stride(),
                                dev_view.storage_offset())

    hz_pack = host_view(d["pack_src"], "pack_base")
    hz_split = host_view(d["split_src"], "split_base")

    def zero_copy_step():
        vf.qkv_pack(hz_pack, P, C, out=host["pack_dst"])
        vf.attn_split(hz_split, P, C, out=host["split_dst"])
        vf.head_merge(host["merge_src"], T, H, D, P, C, out=host["merge_dst"])

    def outputs_match():
        return bool(torch.equal(host["pack_dst"], d["pack_dst"].cpu())
                    and torch.equal(host["split_dst"], d["split_dst"].cpu())
                    and torch.equal(host["merge_dst"], d["merge_dst"].cpu()))

    cur = torch.cuda.current_stream(dev)
    modes = {}
    for name, fn, streams in (
            ("pipelined", pipelined_step, [s_in, s_k, s_out]),
            ("zero_copy", zero_copy_step, [cur]),
            ("serial", serial_step, [cur])):
        for k in keys_out:
            host[k].fill_(0)
        ms = timed(fn, streams)
        # the last outputs on the host must be the relayouts of the inputs
        modes[name] = {"value": round(world * n * step_bytes / (ms / 1e3) / 1e9, 1),
                       "ms_per_step": round(ms / n, 3), "outputs_checked": outputs_match()}
    desc = {"pipelined": "copies pipelined over the %d overlap chunks on 3 streams "
                         "(copy in, chunk-range relayouts, copy out)" % C,
            "zero_copy": "kernels read pinned host inputs and write pinned host outputs "
                         "directly over the host link",
            "serial": "whole-tensor copy in, relayouts, copy out on one stream"}
    best = max((m for m in modes if modes[m]["outputs_checked"]),
               key=lambda m: modes[m]["value"])
    return {"value": modes[best]["value"], "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "ms_per_step": modes[best]["ms_per_step"], "mode": best,
            "mode_description": desc[best], "modes": modes}


class TorchChain:
    """The materialisation chains the direct relayouts replace, on the GPU with
    PyTorch ops ("Sol-Engine alignment on SM86 and SM89", section "What is
    enabled": stack/permute/contiguous for the pack, cat/permute/contiguous
    for the merge; the split copies each token shard's chunk once).  A
    comparison arm only: the library never runs these."""

    def __init__(self, cfg):
        import sequence_head_relayout_gb300 as vf
        self.cfg = cfg
        T, H, D, P, C = cfg.T, cfg.H, cfg.D, cfg.P, cfg.C
        self.pack_tab = vf.piece_table(vf.OP_QKV_PACK, T, H, D, P, C)
        self.split_tab = vf.piece_table(vf.OP_ATTN_SPLIT, T, H, D, P, C)
        self.merge_tab = vf.piece_table(vf.OP_HEAD_MERGE, T, H, D, P, C)

    def qkv_pack(self, src):
        import torch
        cfg = self.cfg
        P, C, Hp = cfg.P, cfg.C, cfg.H // cfg.P
        stacked = torch.stack(src.unbind(1))                       # [3, T, H, D]
        out = torch.empty(3 * cfg.T * cfg.H * cfg.D, dtype=src.dtype, device=src.device)
        tok, length, off = self.pack_tab
        for c in range(C):
            t0, L = tok[c * P], length[c * P]
            blk = out[off[c * P]:off[c * P] + P * 3 * L * Hp * cfg.D].view(P, 3, L, Hp, cfg.D)
            blk.copy_(stacked[:, t0:t0 + L].unflatten(2, (P, Hp)).permute(2, 0, 1, 3, 4))
        return out

    def attn_split(self, src):
        import torch
        cfg = self.cfg
        out = torch.empty(cfg.T * cfg.H * cfg.D, dtype=src.dtype, device=src.device)
        tok, length, off = self.split_tab
        for e in range(len(tok)):
            n = length[e] * cfg.H * cfg.D
            out[off[e]:off[e] + n].view(length[e], cfg.H, cfg.D).copy_(
                src[tok[e]:tok[e] + length[e]])
        return out

    def head_merge(self, flat):
        import torch
        cfg = self.cfg
        P, C, Hp, D = cfg.P, cfg.C, cfg.H // cfg.P, cfg.D
        tok, length, off = self.merge_tab
        slabs = [flat[off[c * P]:off[c * P] + P * length[c * P] * Hp * D].view(
            P, length[c * P], Hp, D) for c in range(C)]
        slot_major = torch.cat(slabs, 1)                          # [P, T, Hp, D]
        return slot_major.permute(1, 0, 2, 3).contiguous().view(cfg.T, cfg.H, D)


def torch_chain_aba(cfg, dev, reps=20):
    """A/B/A against the torch chains at one workload: medians of the chain
    (A, before and after) and of the direct relayout (B), interleaved, each
    rep after an L2 flush; plus the incremental peak memory of each arm
    (the pages' allocation screen)."""
    import torch

    import sequence_head_relayout_gb300 as vf
    from sequence_head_relayout_gb300 import workloads as W

    chain = TorchChain(cfg)
    T, H, D, P, C = cfg.T, cfg.H, cfg.D, cfg.P, cfg.C
    pack_src, _ = W.pack_source(cfg, device=dev)
    split_src, _ = W.split_source(cfg, device=dev)
    merge_src = W.merge_source(cfg, device=dev)
    flush = torch.empty(128 << 20, dtype=torch.int16, device=dev)
    arms = {
        "qkv_pack": (lambda: chain.qkv_pack(pack_src), lambda: vf.qkv_pack(pack_src, P, C)),
        "attn_split": (lambda: chain.attn_split(split_src),
                       lambda: vf.attn_split(split_src, P, C)),
        "head_merge": (lambda: chain.head_merge(merge_src),
                       lambda: vf.head_merge(merge_src, T, H, D, P, C)),
    }
    out = {}
    for op, (a_fn, b_fn) in arms.items():
        same = torch.equal(a_fn().view(-1), b_fn().view(-1))

        def med(fn):
            ts = []
            for _ in range(reps):
                flush.fill_(1)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                ts.append((e0, e1))
            torch.cuda.synchronize()
            return statistics.median(x.elapsed_time(y) for x, y in ts)

        def peak(fn):
            torch.cuda.synchronize()
            torch.cuda.reset_peak_memory_stats(dev)
            base = torch.cuda.memory_allocated(dev)
            r = fn()
            torch.cuda.synchronize()
            p = torch.cuda.max_memory_allocated(dev) - base
            del r
            return p

        for _ in range(3):
            a_fn(), b_fn()
        a1, b, a2 = med(a_fn), med(b_fn), med(a_fn)
        out[op] = {"chain_us": [round(a1 * 1e3, 1), round(a2 * 1e3, 1)],
                   "direct_us": round(b * 1e3, 1),
                   "speedup": round((a1 + a2) / 2 / b, 3),
                   "chain_peak_bytes": peak(a_fn), "direct_peak_bytes": peak(b_fn),
                   "outputs_equal": bool(same)}
    return out


def lossy_quality(dev, T=4096, H=28, D=128, seed=11):
    """What the opt-in lossy transport costs in accuracy, on seeded N(0,1)
    activations at the pages' head count and head dim: the relative L2 error
    of a causal-free attention output when Q, K and V cross the exchange as
    INT8 (pack -> unpack, one destination), and of an attention output that
    crosses as E4M3 (split -> merge)."""
    import torch
    import torch.nn.functional as F

    import sequence_head_relayout_gb300 as vf
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    qkv = torch.randn((T, 3, H, D), generator=g, device=dev).to(torch.bfloat16)
    codes, scales = vf.qkv_pack_q(qkv, 1, 4, fmt="int8")
    q, k, v = vf.qkv_unpack_q(codes, scales, T, H, D, 1, 4, fmt="int8")

    def sdpa(a, b, c):                      # [T,H,D] -> [1,H,T,D]
        return F.scaled_dot_product_attention(*(t.permute(1, 0, 2)[None] for t in (a, b, c)))

    ref = sdpa(qkv[:, 0], qkv[:, 1], qkv[:, 2]).float()
    got = sdpa(q, k, v).float()
    attn = torch.randn((T, H, D), generator=g, device=dev).to(torch.bfloat16)
    fc, fs = vf.attn_split_q(attn, 1, 4, fmt="e4m3")
    back = vf.head_merge_q(fc, fs, T, H, D, 1, 4, fmt="e4m3").float()

    def rel(x, y):
        return float((x - y).norm() / y.norm())
    qkv_f = qkv.float()
    return {"shape": "T=%d H=%d D=%d, N(0,1) bf16" % (T, H, D),
            "int8_qkv_rel_err": round(rel(torch.stack((q, k, v), 1).float(), qkv_f), 6),
            "int8_qkv_attention_out_rel_err": round(rel(got, ref), 6),
            "e4m3_attention_out_rel_err": round(rel(back, attn.float()), 6)}


def per_config(args, dev):
    """Median time and effective GB/s of every relayout at every workload.

    The small workloads fit in L2, so every rep is preceded by a write of a
    256 MB buffer (twice the 129 MB L2) outside the timed region; the events
    bracket the relayout alone, on its launching stream."""
    import torch

    import sequence_head_relayout_gb300 as vf
    from sequence_head_relayout_gb300 import workloads as W

    peak, _ = measured_peak()
    flush = torch.empty(128 << 20, dtype=torch.int16, device=dev)
    reps = max(5, args.config_reps)
    table = {}
    for name in args.configs:
        cfg = W.CONFIGS[name]
        T, H, D, P, C = cfg.T, cfg.H, cfg.D, cfg.P, cfg.C
        Hp = H // P
        pack_src, _ = W.pack_source(cfg, device=dev)
        split_src, _ = W.split_source(cfg, device=dev)
        merge_src = W.merge_source(cfg, device=dev)
        merge_dst, _ = W.merge_destination(cfg, device=dev)
        recv = torch.empty(3 * T * Hp * D, dtype=torch.int16, device=dev)
        W.fill_(recv, cfg.payload, cfg.seed + 3000)
        outs = tuple(torch.empty((T, Hp, D), dtype=torch.int16, device=dev) for _ in range(3))
        pack_dst = torch.empty(3 * T * H * D, dtype=torch.int16, device=dev)
        split_dst = torch.empty(T * H * D, dtype=torch.int16, device=dev)
        n_pack, n_split, n_unpack = 3 * T * H * D, T * H * D, 3 * T * Hp * D
        # opt-in lossy transport: codes + one float scale per head row
        q_pack = torch.empty(n_pack, dtype=torch.int8, device=dev)
        q_pack_s = torch.empty(n_pack // D, dtype=torch.float32, device=dev)
        q_split = torch.empty(n_split, dtype=torch.float8_e4m3fn, device=dev)
        q_split_s = torch.empty(n_split // D, dtype=torch.float32, device=dev)
        vf.qkv_pack_q(pack_src, P, C, fmt="int8", codes=q_pack, scales=q_pack_s)
        vf.attn_split_q(split_src, P, C, fmt="e4m3", codes=q_split, scales=q_split_s)
        q_recv, q_recv_s = q_pack[:n_unpack], q_pack_s[:n_unpack // D]
        merge_bf16 = merge_dst.view(torch.bfloat16)
        outs_bf16 = tuple(o.view(torch.bfloat16) for o in outs)
        ops = {
            "qkv_pack": (alg_bytes(n_pack),
                         lambda: vf.qkv_pack(pack_src, P, C, out=pack_dst)),
            "attn_split": (alg_bytes(n_split),
                           lambda: vf.attn_split(split_src, P, C, out=split_dst)),
            "head_merge": (alg_bytes(n_split), lambda: vf.head_merge(merge_src, T, H, D, P, C,
                                                                     out=merge_dst)),
            "qkv_unpack": (alg_bytes(n_unpack), lambda: vf.qkv_unpack(recv, T, H, D, P, C,
                                                                      outs=outs)),
            "qkv_pack3": (alg_bytes(n_pack), lambda: vf.qkv_pack3(
                pack_src[:, 0], pack_src[:, 1], pack_src[:, 2], P, C, out=pack_dst)),
            "qkv_pack_slot_major": (alg_bytes(n_pack), lambda: vf.qkv_pack(
                pack_src, P, C, out=pack_dst, order="slot_major")),
            "head_merge_slot_major": (alg_bytes(n_split), lambda: vf.head_merge(
                merge_src, T, H, D, P, C, out=merge_dst, order="slot_major")),
            "qkv_pack_int8": (lossy_bytes(n_pack, D), lambda: vf.qkv_pack_q(
                pack_src, P, C, fmt="int8", codes=q_pack, scales=q_pack_s)),
            "qkv_unpack_int8": (lossy_bytes(n_unpack, D), lambda: vf.qkv_unpack_q(
                q_recv, q_recv_s, T, H, D, P, C, fmt="int8", outs=outs_bf16)),
            "attn_split_e4m3": (lossy_bytes(n_split, D), lambda: vf.attn_split_q(
                split_src, P, C, fmt="e4m3", codes=q_split, scales=q_split_s)),
            "head_merge_e4m3": (lossy_bytes(n_split, D), lambda: vf.head_merge_q(
                q_split, q_split_s, T, H, D, P, C, fmt="e4m3", out=merge_bf16)),
        }
        row = {}
        for op, (nbytes, fn) in ops.items():
            for _ in range(3):
                fn()
            ts = []
            for _ in range(reps):
                flush.fill_(1)
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record()
                fn()
                b.record()
                ts.append((a, b))
            torch.cuda.synchronize()
            med = statistics.median(x.elapsed_time(y) for x, y in ts)
            gbs = nbytes / (med / 1e3) / 1e9
            row[op] = {"us": round(med * 1e3, 2), "gbs": round(gbs, 1),
                       "frac_of_peak": round(gbs / peak, 4),
                       "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4)}
        table[name] = row
        del pack_src, split_src, merge_src, merge_dst, recv, outs, pack_dst, split_dst
        del q_pack, q_pack_s, q_split, q_split_s, q_recv, q_recv_s, merge_bf16, outs_bf16
        torch.cuda.empty_cache()
    return {"reps": reps, "l2": "256 MB buffer written between reps, outside the events",
            "bytes": "exact ops: 4 B per element (2 read, 2 written); *_int8 / *_e4m3 "
                     "(opt-in lossy transport): 3 B per element plus one 4 B scale per "
                     "D-element head row",
            "table": table}


# ----------------------------------------------------------------------------
# Reference arm: the oracle on host cores
# ----------------------------------------------------------------------------

def reference_arm(args, world):
    """The CPU oracle on the host cores: W warm-up and K timed passes over a
    token sample per core, sized so the whole run takes a few minutes."""
    from sequence_head_relayout_gb300 import workloads as W
    cfg = W.CONFIGS[args.config]
    cores = args.cpu_cores or os.cpu_count() or 1
    budget = max(0.02, min(2.0, 150.0 / max(1, args.steps + args.warmup)))
    tokens, _ = calibrate_tokens(cfg, budget)
    per_pass, nbytes = run_oracle(cfg, tokens, args.warmup + args.steps, cores)
    timed = per_pass[args.warmup:]
    total = sum(timed)
    value = nbytes * len(timed) / total / 1e9
    sample = ("%d of %d tokens per core per step (H=%d, D=%d, P=%d, C=%d), pack+split+merge, "
              "one process per core, steps started together" % (tokens, cfg.T, cfg.H, cfg.D,
                                                                cfg.P, cfg.C))
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / max(1, len(timed)) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded uniform 16-bit patterns)",
        "config": {"workload": "%s (sampled: %d of %d tokens per core per step): T=%d H=%d "
                               "D=%d P=%d C=%d" % (cfg.name, tokens, cfg.T, cfg.T, cfg.H, cfg.D,
                                                   cfg.P, cfg.C),
                   "step": "qkv_pack + attn_split + head_merge (CPU oracle)",
                   "parallelism": "%d host processes" % cores},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-cores", type=int, default=0)
    ap.add_argument("--only", nargs="+",
                    choices=["qkv_pack", "attn_split", "head_merge", "qkv_unpack"],
                    help="time only these relayouts (profiling runs); the receive-side "
                         "unpack runs only when named here")
    ap.add_argument("--sets", type=int, default=2, help="rotating input/output buffer sets")
    ap.add_argument("--configs", nargs="*", default=["tiny", "4k", "pages", "ragged", "large"],
                    help="workloads for the per-op, per-workload table (none to skip)")
    ap.add_argument("--config-reps", type=int, default=30)
    ap.add_argument("--event-steps", type=int, default=200,
                    help="instrumented steps (at least 50) run after the timed region for "
                         "the per-op durations")
    ap.add_argument("--no-chain", action="store_true",
                    help="skip the A/B/A comparison with the PyTorch materialisation chains")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(args, world)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    line = gpu_arm(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            from sequence_head_relayout_gb300 import workloads as W
            line["cpu_baseline"] = cpu_baseline(W.CONFIGS[args.config],
                                                cores=args.cpu_cores or None)
            line["cpu_baseline"]["lossy_single_core"] = lossy_cpu_baseline(
                W.CONFIGS[args.config])
            if line.get("per_config"):
                cpu = cpu_per_config(list(line["per_config"]["table"]),
                                     cores=args.cpu_cores or None)
                for name, row in cpu.pop("table").items():
                    for op, v in row.items():
                        line["per_config"]["table"][name][op].update(v)
                line["per_config"]["cpu"] = cpu
        else:
            line["cpu_baseline"] = None
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
