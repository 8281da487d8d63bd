"""Benchmark of the fusion-group hot path on GB300.

One step = one pass of every case of the hot path over its full-size
synthetic workload, each one launch through the C ABI:
  * the 64-node group over bf16 x [8192, 8192] with a row vector, a column
    vector and a scalar broadcast in (bf16 out);
  * the softmax region over bf16 logits [32768, 4096], once with the
    sequential order and once with interleaved(8) (exact exp);
  * the AdamW step over the 200 leaves (1,100,046,336 parameters) of a
    Llama-style 1.1B model (f32 params/m/v, bf16 grads).
metric: achieved HBM GB/s = algorithmic bytes of the step (every input read
once, every output written once) / step time.  Per-kernel figures are in
"kernels".  Inputs (15.9 GB) exceed L2 (129 MB), so no flush is needed.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]
Under torchrun each rank runs the whole workload on its own GPU (weak
scaling), or with --split its share of one workload (strong scaling): rows of
the group and the softmax, a range of the tree's parameters.  The cases shard
without exchange, so there is no collective on the data path.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)

L2_BYTES = 129 * 1024 * 1024


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffer) measurement")
    p.add_argument("--e2e-copy-streams", type=int, default=1,
                   help="streams per copy direction in the end-to-end leg (units alternate between them)")
    p.add_argument("--e2e-slices", type=int, default=10,
                   help="AdamW leaf slices of the end-to-end leg (smaller slices: shorter pipeline fill and drain)")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline sample")
    p.add_argument("--softmax-exp", choices=["exact", "fast"], default="fast",
                   help="exp of the softmax region inside the step (the other mode is timed beside it)")
    p.add_argument("--group-math", choices=["exact", "fast"], default="fast",
                   help="realization of the group's exp / erf / gelu nodes inside the step (the other mode is "
                        "timed beside it)")
    p.add_argument("--only", choices=["all", "group", "softmax", "adamw", "norm"], default="all",
                   help="time one case only (profiling captures)")
    p.add_argument("--split", action="store_true",
                   help="under torchrun, split one workload across the ranks (output rows of the group and the "
                        "softmax, the tree's parameters) instead of one full workload per rank: strong scaling")
    p.add_argument("--scale", type=float, default=1.0,
                   help="shrink the group rows, softmax rows and model layers (profiling captures only)")
    return p.parse_args()


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float) -> float:
    """The largest value of x across ranks (the job's time is its slowest
    rank's); identity without an initialised process group."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(bytes_per_rank_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job GB/s: the bytes every rank processed over the slowest rank's time."""
    return world * bytes_per_rank_step * steps / (max_ms / 1e3) / 1e9


def sum_over_ranks(x: int) -> int:
    """The sum of x across ranks (the bytes of one split workload); identity
    without an initialised process group."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return int(x)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([int(x)], dtype=torch.int64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return int(t.item())


def _peaks():
    try:
        with open(os.path.join(HERE, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ----------------------------------------------------------------- clocks
class NvmlSampler:
    """SM clock and clock-event reasons read through NVML (the library
    nvidia-smi reads), polled every 2 ms from a helper thread, so that a timed
    region of a few tens of milliseconds holds a dozen samples.  Read-only
    queries; nothing about the GPU is set."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_uuid: str, period: float = 0.002):
        import ctypes
        import threading

        self.ct = ctypes
        L = ctypes.CDLL("libnvidia-ml.so.1")
        if L.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.L, self.h = L, ctypes.c_void_p()
        if L.nvmlDeviceGetHandleByUUID(gpu_uuid.encode(), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle for " + gpu_uuid)
        self.reasons_fn = getattr(L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            L.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint(0)
        L.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))      # 1: the SM clock
        self.max_mhz = mx.value
        self.period, self.samples = period, []
        self.stop_ev, self.th = threading.Event(), threading.Thread(target=self._run, daemon=True)

    def _run(self):
        c, r = self.ct.c_uint(0), self.ct.c_ulonglong(0)
        while not self.stop_ev.is_set():
            t = time.perf_counter()
            if self.L.nvmlDeviceGetClockInfo(self.h, 1, self.ct.byref(c)) == 0:
                ok = self.reasons_fn(self.h, self.ct.byref(r)) == 0
                self.samples.append((t, c.value, r.value if ok else 0))
            time.sleep(self.period)

    def start(self):
        self.th.start()

    def stop(self, t0: float, t1: float):
        """Stop polling; the summary of the samples taken between host times t0
        and t1 (the timed region), or of all samples if none fell there."""
        self.stop_ev.set()
        self.th.join(timeout=5)
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        use = inside or self.samples
        if not use:
            return None
        bits = 0
        for s in use:
            bits |= s[2]
        return {"sm_mhz": statistics.median(s[1] for s in use), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for b, n in self.REASONS.items() if bits & b), "samples": len(inside),
                "source": "NVML, 2 ms polling" + ("" if inside else "; none inside the timed region, all shown")}


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = os.path.join("/tmp", f"psk_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", self.gpu_id], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, t0=None, t1=None):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        try:
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
            os.remove(self.path)
        except Exception:
            return None
        if not rows:
            return None

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def _gpu_uuid(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev)


# ------------------------------------------------------------ ncu counters
# the sources each kernel's device code is built from (the group kernel is
# generated from group.cu and compiled at run time from the device headers)
_KERNEL_SOURCES = {
    "adamw": ["adamw.cu"],
    "group": ["group.cu", "group_dev.cuh", "devcommon.cuh", "crmath.cuh", "crmath_tables.inc", "pair.cuh"],
    "softmax_sequential": ["lanes.cu", "rowmath.cuh", "pipe.cuh", "devcommon.cuh", "crmath.cuh", "crmath_tables.inc",
                           "pair.cuh"],
    "softmax_interleaved8": ["regions.cu", "rowmath.cuh", "pipe.cuh", "devcommon.cuh", "crmath.cuh",
                             "crmath_tables.inc", "pair.cuh"],
}


def _source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for f in _KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(HERE, "reduction_groups_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def _counter(kernel: str, name: str):
    """A per-launch counter of a kernel at full size from the committed ncu
    summaries (profiles/kernel_counters.txt), if the kernel's source is
    unchanged since the capture; else None."""
    path = os.path.join(HERE, "profiles", "kernel_counters.txt")
    if not os.path.exists(path) or kernel not in _KERNEL_SOURCES:
        return None
    h = _source_hash(kernel)
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == h and parts[2] == name:
            return int(parts[3])
    return None


def _issue_peak():
    """Warp-instruction issue peak: 152 SMs x 4 schedulers x 1 warp-instruction
    per cycle at the maximum SM clock."""
    try:
        with open(os.path.join(HERE, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f)["sm_max_mhz"])
    except Exception:
        mhz = 2070.0
    return 152 * 4 * mhz * 1e6 / 1e9, mhz


# --------------------------------------------------------------- CPU oracle
# The oracle, as it stands, timed on a bounded sample of each case: the
# 64-node group's rows, the softmax region's rows (both orders) and a stretch
# of AdamW parameters, drawn once on the host.  The sample lives in shared
# memory so that one leg runs it on one core and the other splits every case
# into disjoint parts (rows, parameter ranges) over a pool of worker
# processes, one per host core; the parts' outputs land in the same output
# buffers and must equal the one-core leg's bit for bit.

def _cpu_sample_arrays(scale: float):
    import numpy as np

    from synth import workloads as W

    rows_g = max(1, int(8 * scale))
    rows_s = max(1, int(24 * scale))
    n_adam = max(4096, int(4_000_000 * scale))
    wl = W.cap_group(rows_g, 8192)
    (gx, _), (grow, _), (gcol, _), (gsc, _) = wl.host_inputs()
    sx = W.softmax_rows(rows_s, 4096).host_x()
    rng = np.random.default_rng(0)
    th = (rng.standard_normal(n_adam) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n_adam) * 1e-3).astype(np.float32)
    v = np.abs(rng.standard_normal(n_adam) * 1e-4).astype(np.float32)
    g = ((rng.standard_normal(n_adam) * 1e-3).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    ins = {"gx": gx, "grow": grow, "gcol": gcol.reshape(-1), "gsc": gsc.reshape(1), "sx": sx,
           "th": th, "m": m, "v": v, "g": g}
    outs = {"gy": np.zeros((rows_g, 8192), np.uint16), "sy_seq": np.zeros(sx.shape, np.uint16),
            "sy_int": np.zeros(sx.shape, np.uint16), "th1": np.zeros_like(th), "m1": np.zeros_like(m),
            "v1": np.zeros_like(v)}
    nbytes = rows_g * 8192 * 4 + 2 * rows_s * 4096 * 4 + n_adam * 26
    desc = (f"{rows_g} rows of the 64-node group, {rows_s} rows of the softmax region in each order, "
            f"{n_adam} AdamW parameters")
    return ins, outs, {"rows_g": rows_g, "rows_s": rows_s, "n_adam": n_adam}, nbytes, desc


class _Shared:
    """Named arrays in POSIX shared memory (the parent's copies; workers attach
    by name)."""

    def __init__(self, arrays):
        from multiprocessing import shared_memory

        import numpy as np

        self.blocks, self.arrays, self.specs = [], {}, {}
        for k, a in arrays.items():
            blk = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
            view = np.ndarray(a.shape, a.dtype, buffer=blk.buf)
            view[...] = a
            self.blocks.append(blk)
            self.arrays[k] = view
            self.specs[k] = (blk.name, a.shape, a.dtype.str)

    def close(self):
        self.arrays.clear()
        for b in self.blocks:
            b.close()
            b.unlink()


def _attach(specs):
    from multiprocessing import shared_memory

    import numpy as np

    blocks, arrays = [], {}
    for k, (name, shape, dt) in specs.items():
        blk = shared_memory.SharedMemory(name=name)
        blocks.append(blk)
        arrays[k] = np.ndarray(shape, np.dtype(dt), buffer=blk.buf)
    return blocks, arrays


def _oracle_part(case: str, lo: int, hi: int, A: dict):
    """The oracle on rows (or parameters) [lo, hi) of one case of the sample,
    its outputs written into the output arrays of A."""
    import oracle.adamw as OA
    import oracle.group as OG
    import oracle.softmax as OS
    from synth import workloads as W

    if hi <= lo:
        return
    if case == "group":
        wl = W.cap_group(hi - lo, 8192)
        args = [(A["gx"][lo:hi], "bf16", (8192, 1)), (A["grow"], "bf16", (0, 1)), (A["gcol"][lo:hi], "bf16", (1, 0)),
                (A["gsc"], "bf16", (0, 0))]
        A["gy"][lo:hi] = OG.evaluate(wl.tokens, wl.imm, args, (hi - lo, 8192), "bf16")
    elif case == "softmax":
        A["sy_seq"][lo:hi] = OS.softmax_region(A["sx"][lo:hi], "bf16", "bf16", ("sequential",))
        A["sy_int"][lo:hi] = OS.softmax_region(A["sx"][lo:hi], "bf16", "bf16", ("interleaved", 8))
    else:
        hp = W.llama_adamw_leaves(layers=0, V=1).hp
        h = OA.hyper_f32(hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, hp.t)
        t1, m1, v1 = OA.step_leaf(A["th"][lo:hi], A["m"][lo:hi], A["v"][lo:hi], A["g"][lo:hi], "bf16", h)
        A["th1"][lo:hi], A["m1"][lo:hi], A["v1"][lo:hi] = t1, m1, v1


def _oracle_task(task):
    """Pool worker: one part of the sample, on the shared arrays."""
    case, lo, hi, specs = task
    blocks, A = _attach(specs)
    try:
        _oracle_part(case, lo, hi, A)
    finally:
        A.clear()
        for b in blocks:
            b.close()
    return case, lo, hi


def _digest(A, keys):
    h = hashlib.sha256()
    for k in keys:
        h.update(A[k].tobytes())
    return h.hexdigest()


def cpu_sample(scale: float = 1.0, min_seconds: float = 0.0, all_cores: bool = True):
    """Time the oracle, as it stands, on a bounded sample of each case: on one
    core, repeated until min_seconds have passed, then (all_cores) split over
    one worker process per host core, repeated likewise, its outputs checked
    bit for bit against the one-core leg's.  Returns a dict per leg
    ("one_core", "all_cores") of (algorithmic bytes, seconds), the core
    count, the sample's description and whether the legs' outputs agreed."""
    import multiprocessing as mp

    ins, outs, meta, nbytes, desc = _cpu_sample_arrays(scale)
    sh = _Shared({**ins, **outs})
    out_keys = list(outs)
    parts = {"group": meta["rows_g"], "softmax": meta["rows_s"], "adamw": meta["n_adam"]}
    res = {"description": desc}
    try:
        t0, reps = time.perf_counter(), 0
        while True:
            for case, n in parts.items():
                _oracle_part(case, 0, n, sh.arrays)
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= min_seconds:
                break
        res["one_core"] = (reps * nbytes, dt)
        if all_cores:
            ref = _digest(sh.arrays, out_keys)
            for k in out_keys:
                sh.arrays[k][...] = 0
            cores = os.cpu_count() or 1
            tasks = []
            for case, n in parts.items():
                for c in range(cores):
                    lo, hi = n * c // cores, n * (c + 1) // cores
                    if hi > lo:
                        tasks.append((case, lo, hi, sh.specs))
            os.environ.setdefault("OMP_NUM_THREADS", "1")
            with mp.get_context("spawn").Pool(cores) as pool:
                pool.map(_oracle_task, tasks[:cores], chunksize=1)      # start-up and imports, untimed
                t0, reps = time.perf_counter(), 0
                while True:
                    pool.map(_oracle_task, tasks, chunksize=1)
                    reps += 1
                    dt = time.perf_counter() - t0
                    if dt >= min_seconds:
                        break
            res["all_cores"] = (reps * nbytes, dt)
            res["cores"] = cores
            res["bit_identical"] = _digest(sh.arrays, out_keys) == ref
    finally:
        sh.close()
    return res


def cpu_gpt_tree_ms(reps: int = 20) -> float:
    """The oracle on the 28-leaf GPT tree (108,032 parameters), milliseconds
    per step on one host core."""
    import oracle.adamw as OA
    from synth import workloads as W

    tree = W.gpt_adamw_leaves()
    hl = [tree.host_leaf(i) for i in range(len(tree.leaves))]
    OA.step_tree(hl, tree.grad_dtype, tree.hp)
    t0 = time.perf_counter()
    for _ in range(reps):
        OA.step_tree(hl, tree.grad_dtype, tree.hp)
    return (time.perf_counter() - t0) * 1e3 / reps


def cpu_small_group_ms(reps: int = 20) -> float:
    """The oracle on the five-op group over 64x64 f32 (the launch-latency
    case), milliseconds per evaluation on one host core."""
    import oracle.group as OG
    from synth import workloads as W

    wl = W.small_group()
    args = [(a_, dt, s.strides) for (a_, dt), s in zip(wl.host_inputs(), wl.inputs)]
    OG.evaluate(wl.tokens, wl.imm, args, wl.out_shape, wl.out_dtype)
    t0 = time.perf_counter()
    for _ in range(reps):
        OG.evaluate(wl.tokens, wl.imm, args, wl.out_shape, wl.out_dtype)
    return (time.perf_counter() - t0) * 1e3 / reps


# ------------------------------------------------------------- our arm
def run_ours(a, ws, rank, local):
    import numpy as np
    import torch

    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import reduction_groups_gb300 as R
    from synth import workloads as W

    # workloads (drawn on the device; seeds shared, so every rank has the same data)
    sc = a.scale
    wl = W.cap_group(rows=max(1, int(8192 * sc)))
    g_in = wl.device_inputs()
    g_args = [(t, s.strides) for t, s in zip(g_in, wl.inputs)]
    g_out = torch.empty(wl.out_shape, dtype=torch.bfloat16, device="cuda")
    sw = W.softmax_rows(rows=max(1, int(32768 * sc)))
    sx = sw.device_x()
    sy = torch.empty_like(sx)
    tree = W.llama_adamw_leaves(layers=max(1, int(round(22 * sc))))
    leaves = [tree.device_leaf(i) for i in range(len(tree.leaves))]
    clip_leaves = leaves
    split = a.split and ws > 1
    if split:
        # this rank's share of one workload: output rows of the group (the
        # column vector from the same rows) and of the softmax region, a range
        # of the tree's parameters as pieces of leaves
        from reduction_groups_gb300 import shard as SH

        g0, g1 = SH.row_range(wl.out_shape[0], ws, rank)
        g_in = [g_in[0][g0:g1], g_in[1], g_in[2][g0:g1], g_in[3]]
        g_args = [(t, s_.strides) for t, s_ in zip(g_in, wl.inputs)]
        g_out = g_out[g0:g1]
        s0, s1 = SH.row_range(sw.rows, ws, rank)
        sx, sy = sx[s0:s1], sy[s0:s1]
        # the clipped step's share is cut on its squared-norm tree's group
        # boundaries (the group sums are gathered across the ranks)
        clip_leaves = [tuple(t[p0:p1] for t in leaves[i]) for i, p0, p1 in SH.clip_pieces(tree.numels, ws, rank)]
        leaves = [tuple(t[p0:p1] for t in leaves[i]) for i, p0, p1 in SH.param_pieces(tree.numels, ws, rank)]
    torch.cuda.synchronize()

    b_group = sum(t.numel() * t.element_size() for t in g_in) + g_out.numel() * g_out.element_size()
    b_soft = sx.numel() * sx.element_size() + sy.numel() * sy.element_size()
    n_adam = sum(leaf[0].numel() for leaf in leaves)
    b_adam = n_adam * tree.bytes_per_param()
    em = a.softmax_exp
    gm = a.group_math
    launches = {
        "group": lambda: R.psk_group_run(wl.tokens, wl.imm, g_args, g_out, math=gm),
        "softmax_sequential": lambda: R.psk_softmax_region(sx, sy, ("sequential",), em),
        "softmax_interleaved8": lambda: R.psk_softmax_region(sx, sy, ("interleaved", 8), em),
        "adamw": lambda: R.psk_adamw_tree(leaves, tree.hp),
    }
    b_all = {"group": b_group, "softmax_sequential": b_soft, "softmax_interleaved8": b_soft, "adamw": b_adam}
    # the normalization regions (rows beyond the step's path): timed beside
    # the step, or as the step itself under --only norm
    extra_launches, norm_rows = {}, 0
    if a.only in ("all", "norm"):
        for kind, label in (("rms", "rmsnorm"), ("layer", "layernorm")):
            nw = W.norm_rows(kind, rows=max(1, int(32768 * sc)))
            nx = nw.device_x()
            ny = torch.empty_like(nx)
            ng, nb = nw.device_params()
            for oname, order in (("sequential", ("sequential",)), ("interleaved8", ("interleaved", 8))):
                extra_launches[f"{label}_{oname}"] = (lambda nx=nx, ny=ny, kind=kind, eps=nw.eps, ng=ng, nb=nb,
                                                     order=order: R.psk_norm_region(nx, ny, kind, eps, ng, nb, order))
                b_all[f"{label}_{oname}"] = nw.algorithmic_bytes()
            norm_rows = nw.rows
        torch.cuda.synchronize()
    if a.only in ("all", "softmax"):
        # the masked softmax (one mask row for every row, 70 % allowed) and the
        # softmax backward on the softmax region's shape
        mrow = (torch.rand(sw.cols, device="cuda", generator=torch.Generator(device="cuda").manual_seed(7))
                < 0.7).to(torch.uint8)
        extra_launches["softmax_masked_interleaved8"] = lambda: R.psk_softmax_masked(sx, sy, mrow, ("interleaved", 8),
                                                                                     em)
        b_all["softmax_masked_interleaved8"] = b_soft
        bct = torch.empty_like(sx).normal_(generator=torch.Generator(device="cuda").manual_seed(8))
        bdx = torch.empty_like(sx)
        for oname, order in (("sequential", ("sequential",)), ("interleaved8", ("interleaved", 8))):
            extra_launches[f"softmax_backward_{oname}"] = (lambda order=order: R.psk_softmax_backward(sy, bct, bdx,
                                                                                                     order))
            b_all[f"softmax_backward_{oname}"] = 3 * sx.numel() * 2
    if a.only in ("all", "group"):
        # the 64-node group in the other math mode, beside the step
        g_other = "exact" if gm == "fast" else "fast"
        extra_launches[f"group_{g_other}_math"] = lambda: R.psk_group_run(wl.tokens, wl.imm, g_args, g_out,
                                                                          math=g_other)
        b_all[f"group_{g_other}_math"] = b_group
        # the same program, math mode and shape through the precompiled
        # interpreter kernel: the baseline of the program-specialised kernel
        extra_launches["group_interpreter"] = lambda: R.psk_group_run_interp(wl.tokens, wl.imm, g_args, g_out, math=gm)
        b_all["group_interpreter"] = b_group
        # the extended op set (LOG, TANH, RECIP, SELECT on an int32 mask) on the
        # group's shape
        xw = W.select_group(rows=max(1, int(8192 * sc)))
        x_in = xw.device_inputs()
        x_args = [(t, s_.strides) for t, s_ in zip(x_in, xw.inputs)]
        x_out = torch.empty(xw.out_shape, dtype=torch.bfloat16, device="cuda")
        extra_launches["group_select_log_tanh"] = lambda: R.psk_group_run(xw.tokens, xw.imm, x_args, x_out)
        b_all["group_select_log_tanh"] = xw.algorithmic_bytes()
    if a.only == "norm":
        launches = dict(extra_launches)
    kernels = [k for k in launches if a.only in ("all", "norm") or k.startswith(a.only)]
    bytes_step = sum(b_all[k] for k in kernels)
    # the job's bytes per step: every rank's own (a full workload each, or its
    # share of one split workload)
    job_bytes_step = sum_over_ranks(bytes_step) if split else ws * bytes_step

    def step(ev=None):
        for j, k in enumerate(kernels):
            if ev is not None:
                ev[j][0].record()
            launches[k]()
            if ev is not None:
                ev[j][1].record()

    # clocks sampled from before the warm-up (the sampler is running when the
    # timed region starts) to after the timed region
    try:
        sampler = NvmlSampler(_gpu_uuid(torch, local))
    except Exception:
        sampler = ClockSampler(_gpu_uuid(torch, local))
    sampler.start()
    for _ in range(a.warmup):
        step()
    torch.cuda.synchronize()

    def barrier():
        if ws > 1:
            import torch.distributed as dist

            dist.barrier()

    evs = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in kernels]
           for _ in range(a.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t_host0 = time.perf_counter()
    start.record()
    for i in range(a.steps):
        step(evs[i])
    end.record()
    torch.cuda.synchronize()
    t_host1 = time.perf_counter()
    barrier()
    clocks = sampler.stop(t_host0, t_host1)
    total_ms = start.elapsed_time(end)
    per_kernel_ms = {k: sum(evs[i][j][0].elapsed_time(evs[i][j][1]) for i in range(a.steps)) / a.steps
                     for j, k in enumerate(kernels)}
    total_ms = max_over_ranks(total_ms)

    # the softmax region in the other exp mode, timed beside the step (not in value)
    other = "exact" if em == "fast" else "fast"
    extra_ms = {}
    if "softmax_sequential" in kernels:
        for name, order in (("softmax_sequential", ("sequential",)), ("softmax_interleaved8", ("interleaved", 8))):
            for _ in range(2):
                R.psk_softmax_region(sx, sy, order, other)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(a.steps):
                R.psk_softmax_region(sx, sy, order, other)
            e1.record()
            torch.cuda.synchronize()
            extra_ms[f"{name}_{other}_exp"] = e0.elapsed_time(e1) / a.steps

    # the clipped step with a cosine schedule on the same tree (clipping reads
    # every gradient once more before the update), beside the step
    clip_ws = None
    if a.only in ("all", "adamw"):
        clip_ws = torch.empty(max(16, R.psk_adamw_workspace(clip_leaves, "cosine", 100, 5000, 1.0)),
                              dtype=torch.uint8, device="cuda")
        if split:
            # each rank's group sums of ||g||^2, all-gathered, then the scale
            # and the rank's pieces: the one-process step's bits
            from reduction_groups_gb300 import sharded as SHD

            extra_launches["adamw_clip_cosine"] = lambda: SHD.adamw_tree_clipped(
                clip_leaves, tree.numels, ws, rank, tree.hp, 1.0, clip_ws, "cosine", 100, 5000)
        else:
            extra_launches["adamw_clip_cosine"] = lambda: R.psk_adamw_tree_ex(leaves, tree.hp, "cosine", 100, 5000,
                                                                             1.0, clip_ws)
        n_clip = sum(leaf[0].numel() for leaf in clip_leaves)
        b_all["adamw_clip_cosine"] = n_clip * (tree.bytes_per_param() + (2 if tree.grad_dtype == "bf16" else 4))
    if a.only in ("all", "adamw", "softmax", "group"):
        for name, fn in extra_launches.items():
            for _ in range(2):
                fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(a.steps):
                fn()
            e1.record()
            torch.cuda.synchronize()
            extra_ms[name] = e0.elapsed_time(e1) / a.steps

    # the launch-latency cases beside the step: the five-op group on 64x64 f32
    # and the 28-leaf GPT tree (108,032 parameters) as one launch against one
    # launch per leaf
    latency = None
    if a.only == "all":
        def per_launch_us(fn, reps=200):
            for _ in range(10):
                fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                fn()
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) * 1e3 / reps

        import ctypes

        from reduction_groups_gb300 import _native as N
        from reduction_groups_gb300 import ops as O

        sg = W.small_group()
        sg_in = sg.device_inputs()
        sg_args = [(t, s_.strides) for t, s_ in zip(sg_in, sg.inputs)]
        sg_out = torch.empty(sg.out_shape, dtype=torch.float32, device="cuda")
        us_g = per_launch_us(lambda: R.psk_group_run(sg.tokens, sg.imm, sg_args, sg_out))
        # the same calls with the C structs built once (what a C caller pays)
        lib, st = N.lib(), O._stream_handle(None)
        p_, keep_ = O._program(sg.tokens, sg.imm)
        arr_, n_, o_ = O._group_args(sg_args, sg_out)
        us_g_c = per_launch_us(lambda: lib.psk_group_run_ex(ctypes.byref(p_), arr_, n_, ctypes.byref(o_), 0, st))
        gt = W.gpt_adamw_leaves()
        g_leaves = [gt.device_leaf(i) for i in range(len(gt.leaves))]
        us_tree = per_launch_us(lambda: R.psk_adamw_tree(g_leaves, gt.hp))
        us_per_leaf = per_launch_us(lambda: [R.psk_adamw_tree([lf], gt.hp) for lf in g_leaves], reps=50)
        tab_, nt_ = O._leaf_table(g_leaves)
        h_ = O._hparams(gt.hp)
        one_ = [O._leaf_table([lf]) for lf in g_leaves]
        us_tree_c = per_launch_us(lambda: lib.psk_adamw_tree(tab_, nt_, ctypes.byref(h_), st))
        us_per_leaf_c = per_launch_us(lambda: [lib.psk_adamw_tree(t_, k_, ctypes.byref(h_), st) for t_, k_ in one_],
                                      reps=50)
        latency = {
            "small_group_64x64_f32": {"us_per_call": round(us_g, 2), "us_per_call_c_abi": round(us_g_c, 2),
                                      "bytes": sg.algorithmic_bytes(),
                                      "gbs": round(sg.algorithmic_bytes() / (us_g_c * 1e3), 2)},
            "gpt_tree_28_leaves": {"us_one_launch": round(us_tree, 2), "us_one_launch_per_leaf": round(us_per_leaf, 2),
                                   "us_one_launch_c_abi": round(us_tree_c, 2),
                                   "us_one_launch_per_leaf_c_abi": round(us_per_leaf_c, 2),
                                   "launches": [1, len(g_leaves)], "params": gt.n_params,
                                   "params_per_s": round(gt.n_params / (us_tree_c * 1e-6), 1)},
            "note": "back-to-back calls on one stream, CUDA events over the batch, outside the timed region; "
                    "through the Python binding, and through the C ABI with its argument structs built once; "
                    "host-bound at these sizes (argument handling, planning, the launch), not device time",
        }

    # end to end through the public API with host buffers: per step, copy every
    # input from pinned host memory, run the step, read every result back.
    # The step is cut into units (the group, the softmax region, AdamW over
    # consecutive leaf slices: leaves update independently, so the slices give
    # the one-launch step's bits); each unit's inputs go up on one stream, its
    # kernels run on a second once they have landed, its results come down on
    # a third, so copies in both directions overlap each other and the kernels.
    e2e = None
    if not a.no_e2e and a.only == "all":
        host_g = [t.cpu().pin_memory() for t in g_in]
        host_gout = torch.empty(g_out.shape, dtype=g_out.dtype, pin_memory=True)
        host_sx = sx.cpu().pin_memory()
        sy2 = torch.empty_like(sy)
        host_sy = [torch.empty(sy.shape, dtype=sy.dtype, pin_memory=True) for _ in range(2)]
        # the AdamW leaves as views of four flat buffers (theta, m, v, grad) on
        # the device and in pinned host memory, each leaf starting on a 256-byte
        # boundary, so that a slice of consecutive leaves moves in one copy per
        # buffer instead of one per leaf and tensor
        numels = [leaf[0].numel() for leaf in leaves]
        offs, o = [], 0
        for n in numels:
            offs.append(o)
            o += (n + 63) // 64 * 64
        flat_d = [torch.empty(o, dtype=leaves[0][q].dtype, device="cuda") for q in range(4)]
        flat_h = [torch.empty(o, dtype=leaves[0][q].dtype, pin_memory=True) for q in range(4)]
        e_leaves = []
        for i, leaf in enumerate(leaves):
            views = tuple(flat_d[q][offs[i]:offs[i] + numels[i]] for q in range(4))
            for q in range(4):
                views[q].copy_(leaf[q])
                flat_h[q][offs[i]:offs[i] + numels[i]].copy_(leaf[q])
            e_leaves.append(views)
        torch.cuda.synchronize()
        h2d = sum(t.numel() * t.element_size() for t in host_g) + host_sx.numel() * 2 + \
            sum(t.numel() * t.element_size() for t in flat_h)
        d2h = host_gout.numel() * 2 + 2 * host_sy[0].numel() * 2 + \
            sum(t.numel() * t.element_size() for t in flat_h[:3])
        # AdamW slices of about 1/e2e_slices of the parameters each, in leaf order
        slices, cur, acc_n = [], [], 0
        per = max(1, n_adam // max(1, a.e2e_slices))
        for i, leaf in enumerate(leaves):
            cur.append(i)
            acc_n += leaf[0].numel()
            if acc_n >= per:
                slices.append(cur)
                cur, acc_n = [], 0
        if cur:
            slices.append(cur)
        units = []      # (copies in, kernels, copies out) as (device, host) pairs and a launch list
        units.append(([(d_, h_) for d_, h_ in zip(g_in, host_g)],
                      [lambda st: R.psk_group_run(wl.tokens, wl.imm, g_args, g_out, st, math=gm)],
                      [(g_out, host_gout)]))
        units.append(([(sx, host_sx)],
                      [lambda st: R.psk_softmax_region(sx, sy, ("sequential",), em, st),
                       lambda st: R.psk_softmax_region(sx, sy2, ("interleaved", 8), em, st)],
                      [(sy, host_sy[0]), (sy2, host_sy[1])]))
        for k, sl in enumerate(slices):
            lo = offs[sl[0]]
            hi = offs[slices[k + 1][0]] if k + 1 < len(slices) else o   # the slice's span, padding included
            units.append(([(flat_d[q][lo:hi], flat_h[q][lo:hi]) for q in range(4)],
                          [lambda st, sl=sl: R.psk_adamw_tree([e_leaves[i] for i in sl], tree.hp, st)],
                          [(flat_d[q][lo:hi], flat_h[q][lo:hi]) for q in range(3)]))
        n_cs = a.e2e_copy_streams
        s_ins = [torch.cuda.Stream() for _ in range(n_cs)]
        s_outs = [torch.cuda.Stream() for _ in range(n_cs)]
        s_cmp = torch.cuda.Stream()
        ev = [[torch.cuda.Event() for _ in range(3)] for _ in units]    # per unit: in, computed, out
        out_done = [None] * len(units)                                    # last step's "out" events

        def e2e_step(after):
            for u, (cin, cmp, cout) in enumerate(units):
                s_in, s_out = s_ins[u % n_cs], s_outs[u % n_cs]
                e_in, e_cmp, e_out = ev[u]
                with torch.cuda.stream(s_in):
                    s_in.wait_event(after)
                    if out_done[u] is not None:
                        s_in.wait_event(out_done[u])   # the previous step's results of this unit are read
                    for d_, h_ in cin:
                        d_.copy_(h_, non_blocking=True)
                    e_in.record(s_in)
                s_cmp.wait_event(e_in)
                for fn in cmp:
                    fn(s_cmp)
                e_cmp.record(s_cmp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(e_cmp)
                    for d_, h_ in cout:
                        h_.copy_(d_, non_blocking=True)
                    e_out.record(s_out)
                out_done[u] = e_out

        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cur_stream = torch.cuda.current_stream()
        s2.record(cur_stream)
        e2e_step(s2)
        torch.cuda.synchronize()
        barrier()
        s2.record(cur_stream)
        for _ in range(a.steps):
            e2e_step(s2)
        for u in range(len(units)):
            cur_stream.wait_event(out_done[u])
        e2.record(cur_stream)
        torch.cuda.synchronize()
        ms = max_over_ranks(s2.elapsed_time(e2))
        e2e = {"value": round(job_value(job_bytes_step, a.steps, 1, ms), 2), "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms / a.steps, 3),
               "streams": f"inputs and results on {n_cs} streams per direction, kernels on one, overlapped per unit"}

    if rank != 0:
        if ws > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
        return

    peak, peak_kind = _peaks()
    kb = dict(b_all)
    kinfo = {}
    for k in kernels:
        gbs = kb[k] / (per_kernel_ms[k] / 1e3) / 1e9
        kinfo[k] = {"ms": round(per_kernel_ms[k], 4), "algorithmic_bytes": int(kb[k]), "gbs": round(gbs, 1),
                    "frac_of_hbm_peak": round(gbs / peak, 4)}
    for k, ms in extra_ms.items():
        kbytes = b_all.get(k, b_soft)
        gbs = kbytes / (ms / 1e3) / 1e9
        kinfo[k] = {"ms": round(ms, 4), "algorithmic_bytes": int(kbytes), "gbs": round(gbs, 1),
                    "frac_of_hbm_peak": round(gbs / peak, 4), "in_value": False,
                    "rows_per_s": round((norm_rows if k.startswith(("rms", "layer")) else sx.shape[0]) / (ms / 1e3),
                                        1)}
        if k == "adamw_clip_cosine":
            del kinfo[k]["rows_per_s"]
            kinfo[k]["params_per_s"] = round(n_clip / (ms / 1e3), 1)
        if k == "group_select_log_tanh":
            del kinfo[k]["rows_per_s"]
            kinfo[k]["elems_per_s"] = round(xw.out_shape[0] * xw.out_shape[1] / (ms / 1e3), 1)
        if (k.startswith("group_") and k.endswith("_math")) or k == "group_interpreter":
            del kinfo[k]["rows_per_s"]
            kinfo[k]["elems_per_s"] = round(g_out.numel() / (ms / 1e3), 1)
    for k in extra_launches:
        if k in kernels:
            kinfo[k]["rows_per_s"] = round(norm_rows / (per_kernel_ms[k] / 1e3), 1)
    if "group" in kinfo:
        kinfo["group"]["elems_per_s"] = round(g_out.numel() / (per_kernel_ms["group"] / 1e3), 1)
        kinfo["group"]["node_evals_per_s"] = round(kinfo["group"]["elems_per_s"] * wl.n_ops, 1)
    for k in ("softmax_sequential", "softmax_interleaved8"):
        if k in kinfo:
            kinfo[k]["rows_per_s"] = round(sx.shape[0] / (per_kernel_ms[k] / 1e3), 1)
    if "adamw" in kinfo:
        kinfo["adamw"]["params_per_s"] = round(n_adam / (per_kernel_ms["adamw"] / 1e3), 1)
    dom = max(kernels, key=lambda k: per_kernel_ms[k])
    ipeak, mhz = _issue_peak()
    winst = _counter("group", f"warp_instructions_{gm}") if "group" in kernels and a.scale == 1.0 and not split \
        else None
    if winst is not None:
        ach = winst / (per_kernel_ms["group"] / 1e3) / 1e9
        kinfo["group"]["issue_rate_gwarp_instr_s"] = round(ach, 1)
        kinfo["group"]["frac_of_issue_peak"] = round(ach / ipeak, 4)
    if dom == "group" and winst is not None:
        # bound by instruction issue: executed warp-instructions per launch
        # (ncu, unchanged source) over the launch time, against the issue peak
        roofline = {"kernel": dom, "bound": "alu", "achieved": kinfo["group"]["issue_rate_gwarp_instr_s"],
                    "peak": round(ipeak, 1), "peak_source": f"152 SM x 4 issue/clk x {mhz:.0f} MHz",
                    "unit": "G warp-instr/s", "frac": kinfo["group"]["frac_of_issue_peak"], "traffic": None,
                    "hbm_gbs": kinfo["group"]["gbs"]}
    else:
        achieved = kb[dom] / (per_kernel_ms[dom] / 1e3) / 1e9
        roofline = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                    "peak_source": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                    "traffic": _counter(dom, "dram_bytes") if a.scale == 1.0 and not split else None}
    if "adamw" in kinfo:
        kinfo["adamw"]["dram_traffic"] = _counter("adamw", "dram_bytes") if a.scale == 1.0 and not split else None

    cpu = None
    if not a.no_cpu and ws == 1 and a.only == "all":
        r = cpu_sample(15.0, min_seconds=10.0)
        (nb1, dt1), (nba, dta) = r["one_core"], r["all_cores"]
        cpu = {"value": round(nba / dta / 1e9, 6), "unit": "GB/s", "cores": r["cores"], "kind": "oracle",
               "sample": (f"oracle on {r['description']}, repeated: over {r['cores']} worker processes (one per "
                          f"host core, disjoint rows and parameter ranges) {dta:.1f} s; on one core {dt1:.1f} s"),
               "one_core": {"value": round(nb1 / dt1 / 1e9, 6), "unit": "GB/s", "cores": 1},
               "all_cores_bit_identical_to_one_core": r["bit_identical"],
               "small_group_64x64_ms": round(cpu_small_group_ms(), 3),
               "gpt_tree_28_leaves_ms": round(cpu_gpt_tree_ms(), 3)}

    value = job_value(job_bytes_step, a.steps, 1, total_ms)
    line = {
        "metric": "achieved HBM GB/s (% of GB300 peak) for fused group, softmax region, AdamW params/s",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": round(total_ms / a.steps, 4), "higher_is_better": True,
        "scaling": "strong" if split else "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded device draws, shapes of the workloads)",
        "config": {"workload": "64-node group bf16 [8192,8192] + softmax region bf16 [32768,4096] "
                               "(sequential, interleaved(8)) + AdamW tree of a Llama-style 1.1B model",
                   "softmax_exp": em, "group_math": gm, "l2": "inputs larger than L2 (no flush needed)",
                   "bytes_per_step": int(job_bytes_step),
                   "parallelism": f"rows and parameters split x{ws}" if split else f"replicas x{ws}"},
        "kernels": kinfo, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
        "latency_cases": latency,
        "gpu_launches": len(kernels) * a.steps,
    }
    if a.only != "all" or a.scale != 1.0:
        line["config"]["partial"] = f"only={a.only} scale={a.scale}: a profiling run, not the benchmark"
    print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


# ------------------------------------------------------ the reference arm
def run_reference(a, ws, rank):
    """The oracle, as it stands, on this machine's host cores: each step is a bounded
    sample of the same workload, split over one worker process per host core,
    reported in the same unit."""
    if rank != 0:
        return
    for _ in range(a.warmup):
        cpu_sample(2.5)
    tot_b, tot_t = 0, 0.0
    desc, cores = "", 1
    for _ in range(a.steps):
        r = cpu_sample(2.5)
        nb, dt = r["all_cores"]
        tot_b += nb
        tot_t += dt
        desc, cores = r["description"], r["cores"]
    v = tot_b / tot_t / 1e9
    line = {
        "impl": "reference",
        "metric": "achieved HBM GB/s (% of GB300 peak) for fused group, softmax region, AdamW params/s",
        "value": round(v, 6), "unit": "GB/s", "n_gpus": ws, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": round(tot_t / a.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "64-node group bf16 [8192,8192] + softmax region bf16 [32768,4096] "
                               "(sequential, interleaved(8)) + AdamW tree of a Llama-style 1.1B model"},
        "cpu_baseline": {"value": round(v, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"oracle on {desc} per step, over {cores} worker processes (one per host core)"},
        "e2e": {"value": round(v, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    a = _args()
    ws, rank, local = _dist()
    if a.impl == "reference":
        run_reference(a, ws, rank)
    else:
        run_ours(a, ws, rank, local)


if __name__ == "__main__":
    main()
