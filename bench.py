"""Benchmark of one Medusa decode step (heads + top-k, Cartesian tree, tree
attention, verification, acceptance) on one B300 per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl medusa|reference]

Prints one JSON line (rank 0).  A "step" is one medusa_step call over the
whole batch of the workload; `value` is steps/s summed over ranks.  With N > 1
(torchrun) every rank runs an independent replica of the workload: the step
has no cross-sequence exchange at batch 1, so there is no collective on the
data path (weak scaling).  `--impl reference` times the plain CPU oracle
instead (the only reference implementation of this path), on the host cores.
"""
from __future__ import annotations

import argparse
import contextlib
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from medusa_head_tree_heads_b300 import synth  # noqa: E402

DEFAULT_WORKLOAD = "7b-bf16"
METRIC = "Medusa decode steps/s at 7B shape; achieved HBM GB/s vs B300 peak"


def algorithmic_bytes(s) -> dict:
    """Bytes each kernel must move at least once per step (weights and cache
    read once, logits never materialised)."""
    e = 2 if s.dtype == "bf16" else 4
    B, H, V, K, T = s.batch, s.hidden, s.vocab, s.n_heads, s.n_nodes
    kv = 2 * B * s.kv_len * s.n_kv_heads * s.head_dim * e
    tree_qkv = B * T * (s.n_q_heads + 2 * s.n_kv_heads) * s.head_dim * e
    return {
        "head_layer": (K * H * H + K * H + B * H) * e + B * K * H * 4,
        "head_proj_topk": K * V * H * e + B * K * H * 4,
        "tree_attn": kv + tree_qkv + B * T * H * e,
        "verify_proj": V * H * e + B * T * H * e,
        "step": (K * (H * H + H) + K * V * H + V * H + B * H) * e + kv + tree_qkv,
    }


def flops(s) -> dict:
    B, H, V, K, T = s.batch, s.hidden, s.vocab, s.n_heads, s.n_nodes
    return {"heads": 2 * B * K * (H * H + V * H), "verify": 2 * B * T * V * H,
            "attn": 4 * B * T * s.n_q_heads * s.head_dim * (s.kv_len + s.depth + 1)}


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# the dominant kernel, from an ncu capture of the full-size workload, keyed by
# the SHA-256 of the kernel's source file at capture time: a changed kernel
# reports null until it is captured again.
TRAFFIC_CAPTURES = {
    "7b-bf16": {"source": "medusa_head_tree_heads_b300/csrc/heads_tc.cu", "sha256": "03473dc9ccb0f417e3ff63ff45b937fdf3aafe10adaa423000eb5f2cbfc21394",
                "bytes": 1312627712 + 3890176},
}


def captured_traffic(workload: str):
    c = TRAFFIC_CAPTURES.get(workload)
    if c is None:
        return None
    import hashlib
    with open(os.path.join(ROOT, c["source"]), "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != c["sha256"]:
            return None
    return c["bytes"]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"], "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "source": "fallback"}


class _Nvml:
    """The few read-only NVML queries the clock sampler needs, bound with
    ctypes to the driver's libnvidia-ml (no Python NVML package required)."""

    CLOCK_SM = 1
    REASON_BITS = (("sw_power_cap", 0x4), ("hw_slowdown", 0x8), ("sw_thermal_slowdown", 0x20),
                   ("hw_thermal_slowdown", 0x40))

    def __init__(self, cuda_index: int):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        pr = torch.cuda.get_device_properties(cuda_index)
        bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(self.h)) != 0:
            if self.lib.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(self.h)) != 0:
                raise OSError("no NVML handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sm_clock(self, maximum=False) -> float:
        v = self.c.c_uint()
        fn = self.lib.nvmlDeviceGetMaxClockInfo if maximum else self.lib.nvmlDeviceGetClockInfo
        if fn(self.h, self.CLOCK_SM, self.c.byref(v)) != 0:
            raise OSError("clock query failed")
        return float(v.value)

    def reasons(self) -> set:
        v = self.c.c_ulonglong()
        if self.reasons_fn(self.h, self.c.byref(v)) != 0:
            raise OSError("reason query failed")
        return {n for n, bit in self.REASON_BITS if v.value & bit}


class Clocks:
    """SM clock and throttle-reason samples taken during a region: an NVML
    poller thread (every ~2 ms, so even a region of a few tens of ms gets
    samples), else nvidia-smi at its 100 ms period.  Reads only; no GPU
    setting is touched."""

    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.samples = []  # (sm_mhz, max_mhz, set of reasons)
        self.source = None

    def _poll(self, nv):
        mx = nv.sm_clock(maximum=True)
        while not self.stop.is_set():
            try:
                self.samples.append((nv.sm_clock(), mx, nv.reasons()))
            except OSError:
                break
            self.stop.wait(0.002)

    def __enter__(self):
        import threading
        try:
            nv = _Nvml(self.index)
            self.stop = threading.Event()
            self.thread = threading.Thread(target=self._poll, args=(nv,), daemon=True)
            self.thread.start()
            self.source = "nvml"
            return self
        except (OSError, AttributeError, RuntimeError, AssertionError):
            self.source = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.source == "nvml":
            self.stop.set()
            self.thread.join(timeout=5)
            return
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            for l in out.splitlines():
                f = [x.strip() for x in l.split(",")]
                if len(f) < 6:
                    continue
                try:
                    sm, mx = float(f[0]), float(f[1])
                except ValueError:
                    continue
                self.samples.append((sm, mx, {n for n, v in zip(self.NAMES, f[2:6]) if v.lower() == "active"}))

    def summary(self) -> dict:
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0,
                    "source": self.source}
        reasons = set()
        for _, _, r in self.samples:
            reasons |= r
        return {"sm_mhz": statistics.median(x[0] for x in self.samples),
                "sm_max_mhz": max(x[1] for x in self.samples), "reasons": sorted(reasons),
                "samples": len(self.samples), "source": self.source}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def oracle_inputs(inp):
    import numpy as np
    out = {}
    for k, v in inp.items():
        out[k] = v.view(torch.int16).numpy().view(np.uint16) if v.dtype == torch.bfloat16 else v.numpy()
    return out


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or "unknown"


def host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


@contextlib.contextmanager
def blas_one_thread():
    """Holds the BLAS library numpy calls to one thread; yields how
    ("threadpoolctl", "openblas") or None when neither way is available.
    threadpoolctl is not installed on every host, so numpy's bundled OpenBLAS
    is also reached directly through its exported thread setter."""
    try:
        from threadpoolctl import threadpool_limits
    except ImportError:
        threadpool_limits = None
    if threadpool_limits is not None:
        with threadpool_limits(limits=1):
            yield "threadpoolctl"
        return
    import ctypes
    import glob
    found = None
    import numpy as np
    for path in sorted(glob.glob(os.path.join(os.path.dirname(np.__file__), "..", "numpy.libs", "*openblas*.so*"))):
        lib = ctypes.CDLL(path)
        for name in ("scipy_openblas_{}_num_threads64_", "scipy_openblas_{}_num_threads", "openblas_{}_num_threads"):
            setn = getattr(lib, name.format("set"), None)
            getn = getattr(lib, name.format("get"), None)
            if setn is not None and getn is not None:
                found = (setn, getn)
                break
        if found:
            break
    if found is None:
        yield None
        return
    setn, getn = found
    getn.restype = ctypes.c_int
    before = getn()
    setn(ctypes.c_int(1))
    try:
        yield "openblas"
    finally:
        setn(ctypes.c_int(before))


def time_oracle(s, inp, budget_s: float = 20.0, single_thread: bool = True) -> dict:
    """The oracle as it stands, on this host's cores: whole steps until the
    time budget is used (at least one), with the BLAS library on every core;
    then one whole step with it held to one thread."""
    from oracle import medusa_oracle as O
    n = oracle_inputs(inp)
    times = []
    t_all = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        O.step(n, s)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all > budget_s:
            break
    res = {"value": len(times) / sum(times), "unit": "steps/s", "cores": host_cores(), "kind": "oracle",
           "sample": f"{len(times)} whole step(s) of {s.name} (numpy float64, BLAS on all cores)",
           "seconds": sum(times), "cpu_model": cpu_model()}
    if single_thread:
        with blas_one_thread() as how:
            if how is None:
                res["single_thread"] = {"value": None, "unavailable": "no way to hold this host's BLAS to one thread"}
            else:
                t0 = time.perf_counter()
                O.step(n, s)
                dt = time.perf_counter() - t0
                res["single_thread"] = {"value": 1.0 / dt, "unit": "steps/s", "cores": 1,
                                        "sample": f"1 whole step of {s.name} (BLAS held to one thread by {how})"}
    return res


def workload_config(s, parallelism: str) -> dict:
    """The workload's sizes, shared by both arms' JSON lines."""
    return {"workload": s.name, "batch": s.batch, "hidden": s.hidden, "vocab": s.vocab, "heads": s.n_heads,
            "topk": list(s.topk), "tree_nodes": s.n_nodes, "kv_len": s.kv_len, "q_heads": s.n_q_heads,
            "kv_heads": s.n_kv_heads, "head_dim": s.head_dim, "accept": s.accept, "parallelism": parallelism}


def run_reference(args, world, rank):
    if rank != 0:
        return
    s = synth.SHAPES[args.workload]
    plan = synth.load_plans()[s.name]
    inp = synth.make_inputs(s, plan)
    # each timed "step" is one whole oracle step (bounded: a few minutes for K + W)
    from oracle import medusa_oracle as O
    n = oracle_inputs(inp)
    for _ in range(args.warmup):
        O.step(n, s)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        O.step(n, s)
    dt = time.perf_counter() - t0
    v = args.steps / dt
    cores = host_cores()
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "steps/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(s, "oracle on the host cores"),
            "cpu_baseline": {"value": v, "unit": "steps/s", "cores": cores, "kind": "oracle",
                             "sample": f"{args.steps} whole step(s) of {s.name} after {args.warmup} warm-up",
                             "cpu_model": cpu_model()},
            "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_medusa(args, world, rank, local):
    from medusa_head_tree_heads_b300 import medusa as M
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    s = synth.SHAPES[args.workload]
    plan = synth.load_plans()[s.name]
    inp = synth.make_inputs(s, plan)
    dinp = {k: v.cuda() for k, v in inp.items()}
    cfg = M.make_config(s)
    ws = M.alloc_workspace(cfg)
    out = M.alloc_outputs(cfg)
    io = M.step_io(dinp, out)
    stream = torch.cuda.current_stream()

    def step():
        M.medusa_step(cfg, io, ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if not args.no_graph:  # one CUDA graph per step: no host launch gaps between the kernels
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            M.medusa_step(cfg, io, ws)
        step = graph.replay
        for _ in range(3):
            step()
        torch.cuda.synchronize()
    assert M.medusa_get_device_error(ws) == 0
    # sanity: the planted acceptance
    acc = out["accept_len"].cpu().tolist()
    planted = [q["depth"] for q in plan["seqs"]]

    # ---- timed region: K steps, inputs resident in HBM (1.7+ GB > L2)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = ev0.elapsed_time(ev1) / args.steps
    ms = reduce_max(ms, world)
    value = world * 1e3 / ms

    # ---- per-kernel durations (same step with events around each kernel)
    nk = len(M.STEP_KERNELS)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * nk)] for _ in range(args.steps)]
    for row in evs:  # torch creates the CUDA event lazily, at its first record
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    if args.no_graph:
        for i in range(args.steps):
            M.medusa_step_profiled(cfg, io, ws, evs[i])
    else:  # one capture per event set, replayed like the timed steps
        graphs = []
        for i in range(args.steps):
            gp = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gp):
                M.medusa_step_profiled(cfg, io, ws, evs[i])
            graphs.append(gp)
        torch.cuda.synchronize()
        for gp in graphs:
            gp.replay()
    torch.cuda.synchronize()
    per_kernel = {}
    for k, name in enumerate(M.STEP_KERNELS):
        per_kernel[name] = statistics.mean(evs[i][2 * k].elapsed_time(evs[i][2 * k + 1]) for i in range(args.steps))
    byts = algorithmic_bytes(s)
    peaks = measured_peaks()
    dom = "head_proj_topk"
    achieved = byts[dom] / (per_kernel[dom] * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": captured_traffic(s.name) if dom == "head_proj_topk" else None,
                "peak_source": peaks["source"], "algorithmic_bytes": byts[dom],
                "kernel_ms": {k: round(v, 4) for k, v in per_kernel.items()},
                "step_achieved_gbs": round(byts["step"] / (ms * 1e-3) / 1e9, 1),
                "step_frac": round(byts["step"] / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}

    # ---- end to end through the public API: every step's inputs are copied
    # from pinned host memory and its result is read back to the host.  Two
    # buffer sets pipeline the copies with the steps: step n+1's inputs upload
    # on an upload stream while step n computes, and the host waits for step n's
    # result while step n+1 runs (each step still copies in and reads out).
    # A step's inputs travel as one packed buffer (each tensor at a 256-byte
    # aligned offset): one host-to-device copy per step.
    step_in = ["h", "root_token", "q", "k_tree", "v_tree"]
    offs, nbytes = {}, 0
    for k in step_in:
        offs[k] = nbytes
        nbytes = (nbytes + inp[k].numel() * inp[k].element_size() + 255) // 256 * 256
    host_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    for k in step_in:
        n_k = inp[k].numel() * inp[k].element_size()
        host_in[offs[k]:offs[k] + n_k].copy_(inp[k].contiguous().view(-1).view(torch.uint8))

    def views(buf):
        return {k: buf[offs[k]:offs[k] + inp[k].numel() * inp[k].element_size()].view(inp[k].dtype).view(inp[k].shape)
                for k in step_in}

    step_out = ["accept_len", "acc_tokens", "bonus"]
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()  # one stream each way: an upload never queues behind a readback
    sets = []
    for j in range(2):
        packed = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        d_j = dict(dinp)
        d_j.update(views(packed))
        o_j = M.alloc_outputs(cfg)
        sets.append({"packed": packed, "out": o_j, "io": M.step_io(d_j, o_j), "ws": M.alloc_workspace(cfg),
                     "host_out": {k: torch.empty(o_j[k].shape, dtype=o_j[k].dtype).pin_memory() for k in step_out},
                     "ev_in": torch.cuda.Event(), "ev_done": torch.cuda.Event(), "ev_out": torch.cuda.Event()})
    h2d = nbytes
    d2h = sum(v.numel() * v.element_size() for v in sets[0]["host_out"].values())

    def e2e_run(n_steps):
        last = None
        for n in range(n_steps):
            b = sets[n % 2]
            with torch.cuda.stream(up):
                up.wait_event(b["ev_done"])  # the set's previous step has finished with its inputs
                b["packed"].copy_(host_in, non_blocking=True)
                b["ev_in"].record(up)
            comp.wait_event(b["ev_in"])
            M.medusa_step(cfg, b["io"], b["ws"], comp)
            b["ev_done"].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(b["ev_done"])
                for k in step_out:
                    b["host_out"][k].copy_(b["out"][k], non_blocking=True)
                b["ev_out"].record(down)
            if last is not None:
                last["ev_out"].synchronize()  # step n-1's result is on the host
            last = b
        last["ev_out"].synchronize()
        return last["host_out"]

    e2e_run(4)
    barrier(world)
    t0 = time.perf_counter()
    res_host = e2e_run(args.steps)
    e2e_dt = reduce_max((time.perf_counter() - t0) / args.steps, world)
    assert res_host["accept_len"].tolist() == planted

    loop = None
    if s.name == DEFAULT_WORKLOAD and not args.no_loop:
        loop = decode_loop_figures(args)

    line = {"metric": METRIC, "value": round(value, 2), "unit": "steps/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": s.dtype, "data": "synthetic",
            "config": dict(workload_config(s, f"replicas{world}"), l2="inputs larger than L2 (no flush)",
                           accept_len=acc, launch="eager" if args.no_graph else "cuda_graph"),
            "roofline": roofline,
            "e2e": {"value": round(world / e2e_dt, 2), "unit": "steps/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps * M.step_launches(cfg), "clocks": clk.summary()}
    if loop is not None:
        line["decode_loop"] = loop
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = time_oracle(s, inp, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)


def decode_loop_figures(args, name: str = "toy-7b") -> dict:
    """Rounds of decoding over the 7B-shaped table backbone (the stage calls
    of the library, the commit of the kept branch and the next inputs, with
    the backbone's table lookups between tree and attention), captured as one
    CUDA graph of all rounds that starts by restoring the initial caches:
    tokens per round and tokens per second."""
    from medusa_head_tree_heads_b300 import decode_loop
    t = synth.TOYS[name]
    loop = decode_loop.DecodeLoop(t, synth.make_toy(t))
    loop.run()  # warm-up (and the kernels' first-launch set-up)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        loop.reset()
        loop.run()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    reps = 5
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    sec = e0.elapsed_time(e1) / 1e3 / reps
    tokens = loop.tokens()
    return {"workload": name, "rounds": t.rounds, "batch": t.batch, "tokens": tokens,
            "tokens_per_round": round(tokens / (t.rounds * t.batch), 3),
            "ms_per_round": round(sec / t.rounds * 1e3, 4), "tokens_per_s": round(tokens / sec, 1),
            "launch": "one CUDA graph of all rounds (eager stage calls, no fused step)",
            "heads": "synthetic, right per (head, token) with probability " + str(list(t.head_acc))}


def run_vocab_shards(args, world, rank, local):
    """The vocabulary-sharded step: rank r holds rows of W2 and lm_head for
    shard r of `world`; every step is medusa_shard_partial, one all-gather of
    the records (NCCL), medusa_shard_finish.  One step runs on all ranks at
    once, so value = steps/s of the job (strong scaling: the work per step is
    fixed as the rank count grows)."""
    from medusa_head_tree_heads_b300 import medusa as M
    from medusa_head_tree_heads_b300 import shards as SH
    torch.cuda.set_device(local)
    s = synth.SHAPES[args.workload]
    plan = synth.load_plans()[s.name]
    inp = synth.make_inputs(s, plan)
    v0, v1 = SH.bounds(s.vocab, world)[rank]
    W2s, lms = SH.shard_weights(inp.pop("W2"), inp.pop("lm_head"), v0, v1)
    dinp = {k: v.cuda() for k, v in inp.items()}
    dinp["W2"], dinp["lm_head"] = W2s.cuda(), lms.cuda()
    del W2s, lms
    st = SH.ShardedStep(s, world, rank)
    out = M.alloc_outputs(st.cfg)
    io = M.step_io(dinp, out)

    def step():
        st.partial(io)
        if world > 1:
            SH.exchange(st.record, st.records)
        else:
            st.records[0].copy_(st.record)
        st.finish(io)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert M.medusa_get_device_error(st.ws) == 0
    acc = out["accept_len"].cpu().tolist()
    assert acc == [q["depth"] for q in plan["seqs"]], acc
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        ev0.record()
        for _ in range(args.steps):
            step()
        ev1.record()
        torch.cuda.synchronize()
    barrier(world)
    ms = reduce_max(ev0.elapsed_time(ev1) / args.steps, world)
    byts = algorithmic_bytes(s)
    shard_bytes = byts["step"] - (s.n_heads + 1) * (s.vocab - (v1 - v0)) * s.hidden * (2 if s.dtype == "bf16" else 4)
    peaks = measured_peaks()
    line = {"metric": METRIC, "value": round(1e3 / ms, 2), "unit": "steps/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "strong",
            "vs_baseline": None, "dtype": s.dtype, "data": "synthetic",
            "config": dict(workload_config(s, f"vocab-sharded x{world}"), l2="inputs larger than L2 (no flush)",
                           accept_len=acc, launch="eager, one all-gather per step"),
            "roofline": {"bound": "hbm", "kernel": "whole sharded step (rank 0)", "unit": "GB/s",
                         "achieved": round(shard_bytes / (ms * 1e-3) / 1e9, 1), "peak": peaks["hbm_gbs"],
                         "frac": round(shard_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4), "traffic": None,
                         "peak_source": peaks["source"], "algorithmic_bytes": shard_bytes},
            "gpu_launches": None, "clocks": clk.summary()}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.SHAPES))
    ap.add_argument("--impl", default="medusa", choices=["medusa", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch each step eagerly instead of replaying a CUDA graph")
    ap.add_argument("--no-loop", action="store_true", help="skip the multi-round decoding figures")
    ap.add_argument("--vocab-shards", action="store_true",
                    help="split W2 / lm_head rows over the ranks (one all-gather per step) instead of replicas")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    args.warmup = max(args.warmup, 3)  # at least 3 warm-up steps, reported as run
    if args.impl == "reference":
        # each oracle step takes seconds: keep the whole run within a few minutes
        # (at most 20 timed steps, reported as run)
        args.steps = min(args.steps, 20)
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.vocab_shards:
        run_vocab_shards(args, world, rank, local)
    else:
        run_medusa(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
