"""Benchmark of the tree-verify step on GB300.

One step = the whole hot path on one batch: tsd_tree_build (top-k + best-first
tree) -> tsd_tree_verify_attn (branch-aware attention) -> tsd_accept_walk
(argmax + greedy walk) -> tsd_commit_path (accepted-path KV commit), chained
on one stream.  Metric: verified tree nodes per second (B * D per step).

Default workload: the long-context GQA verify (B=8, 32 q / 8 KV heads, head
dim 128, bf16 KV, prefix 32768, vocab 151936, depth 8, top-10, budget 64), the
largest single-GPU configuration and one of the two the HBM-roofline target is
stated on; the same line also carries the other one, the batched serving
workload (B=32, prefixes U{1024..4096}, budget 32), measured the same way
(--also, "" to skip).  Other workloads: --config toy|qwen|batched|long|mla.

Timing: W untimed warm-up steps, then K steps, each replayed from a CUDA
graph of the four calls and bracketed by CUDA events on the launching
stream; before every timed step the L2 is flushed (a memset of twice its
size) and the prefix lengths the previous commit advanced are restored, both
outside the events.  A barrier and a device synchronise bracket the timed
region; the per-step time is the max over ranks.  A second, eager pass times
each call separately for the per-kernel roofline.  The end-to-end leg times
the same step through the Python API with host (pinned) inputs copied in and
the step's results copied out inside the timed region.

--impl reference times the CPU oracle (the plain fp64 restatement the tests
compare against) on a bounded sample of the same workload on the host cores.
Under torchrun each rank runs its own batch (requests are independent: weak
scaling, no collective on the data path); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from tree_speculative_decoding_tsd_gb300 import workloads as W  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
METRIC = "tree-verify nodes/s"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--config", default="long", choices=list(W.WORKLOADS))
    p.add_argument("--also", default="batched",
                   help="comma-separated workloads measured in the same run (step and "
                        "per-call times, roofline), reported under 'also'")
    p.add_argument("--no-graph", action="store_true", help="time eager calls, not graph replay")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="budget of the CPU-oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


# ------------------------------------------------------------ distributed --

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = False
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend=backend)
            self.pg = True

    def barrier(self):
        if self.pg:
            import torch.distributed as dist
            dist.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch.distributed as dist
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            import torch.distributed as dist
            dist.destroy_process_group()


# ------------------------------------------------------------ the workload --

def workload_desc(w):
    plen = "U{%d..%d}" % (w.P_min, w.P) if w.P_min != w.P else str(w.P)
    return (f"{w.name}: B={w.B} S={w.S} k={w.k} D={w.D} V={w.V} P={plen} Hq={w.Hq} "
            f"Hkv={w.Hkv} dk={w.dk} dv={w.dv}{' (V=K[:dv])' if w.v_aliases_k else ''} {w.dtype}")


def algorithmic_bytes(w, plen):
    """Bytes each call must move at minimum (reads + writes), per step."""
    es = 4 if w.dtype == "f32" else 2
    P = int(np.asarray(plen, dtype=np.int64).sum())
    R = w.R
    kv_row = w.dk * es + (0 if w.v_aliases_k else w.dv * es)
    build = w.B * w.S * w.V * 4 + w.B * R * (4 * 4 + 8 + 1)
    verify = (P * w.Hkv * kv_row                       # prefix K/V, once
              + w.B * R * w.Hq * w.dk * es                # q
              + w.B * R * w.Hkv * kv_row                  # scratch-pad tree K/V
              + w.B * R * 8                               # masks
              + w.B * R * w.Hq * (w.dv * es + 4))         # out + lse
    accept = w.B * R * w.V * 4 + w.B * R * (4 * 3 + 8 + 1) + w.B * (w.S + 4) * 4
    return dict(build=build, verify=verify, accept=accept), P * w.Hkv * kv_row


def make_inputs(w, dev, rank):
    """Seeded synthetic inputs on the device (rank-offset seed per replica)."""
    if rank:
        w = w.scaled(index=w.index + 1000 * rank)
    lg = W.draft_logits(w)
    probs = W.draft_probs(w, lg)
    root = W.root_tokens(w)
    plen = W.prefix_lens(w)
    q = W.queries(w)
    kc, vc = W.kv_cache(w)
    kt, vt = W.tree_kv(w)
    host = dict(logits=lg, probs=probs, root=root, plen=plen, q=q, kc=kc, vc=vc, kt=kt, vt=vt)
    d = {k: (None if v is None else v.to(dev)) for k, v in host.items() if k != "logits"}
    return w, host, d


class Clocks:
    """SM clock and clock-event reasons sampled during the timed region.

    Reads NVML through ctypes from a background thread every 0.2 ms (the timed
    regions of the small workloads last a few milliseconds, shorter than one
    nvidia-smi sampling period).  Falls back to `nvidia-smi -lms 100` when NVML
    cannot be loaded.  Only reads: no clock or other GPU setting is changed."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, dev):
        self.samples = []
        self.t0 = self.t1 = None
        self.max_mhz = None
        self.proc = None
        self.thread = None
        self.stop_flag = threading.Event()
        try:
            self._open_nvml(dev)
        except (OSError, AttributeError, RuntimeError):
            self.nvml = None
            self._start_smi(dev.index if dev.index is not None else 0)
            return
        self.thread = threading.Thread(target=self._poll, daemon=True)
        self.thread.start()
        deadline = time.perf_counter() + 2.0
        while not self.samples and time.perf_counter() < deadline:
            time.sleep(0.001)

    def _open_nvml(self, dev):
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        h = ctypes.c_void_p()
        ok = False
        try:
            uuid = str(torch.cuda.get_device_properties(dev).uuid)
            for u in (uuid, "GPU-" + uuid):
                if nv.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) == 0:
                    ok = True
                    break
        except (AttributeError, RuntimeError):
            pass
        if not ok and nv.nvmlDeviceGetHandleByIndex_v2(dev.index or 0, ctypes.byref(h)) != 0:
            raise RuntimeError("no NVML handle")
        self.nvml, self.h = nv, h
        self.get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = int(mx.value)

    def _poll(self):
        mhz = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self.stop_flag.is_set():
            t = time.perf_counter()
            if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0 and \
                    self.get_reasons(self.h, ctypes.byref(rs)) == 0:
                self.samples.append((t, int(mhz.value), int(rs.value)))
            time.sleep(0.0002)

    def _start_smi(self, index):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index),
                 "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def begin(self):
        self.t0 = time.perf_counter()

    def end(self):
        self.t1 = time.perf_counter()

    def stop(self):
        if self.thread is not None:
            self.stop_flag.set()
            self.thread.join(timeout=2)
            win = [s for s in self.samples if self.t0 <= s[0] <= self.t1]
            if not win:
                return None
            reasons = sorted({n for _, _, r in win for b, n in self.REASONS.items() if r & b})
            return {"sm_mhz": statistics.median(s[1] for s in win), "sm_max_mhz": self.max_mhz,
                    "samples": len(win), "source": "nvml, 0.2 ms period", "reasons": reasons}
        return self._stop_smi()

    def _stop_smi(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 7 and parts[0].isdigit():
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [int(r[0]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": int(rows[0][1]),
                "samples": len(rows), "source": "nvidia-smi, 100 ms period", "reasons": reasons}


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def load_tensor_peak():
    """Dense bf16 TF/s for a kernel timed alone (the burst figure)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def verify_flops(w, plen):
    """Tensor-core work of the verify call: every packed row against every
    prefix key, q.k over dk and p.v over dv (2 flops per multiply-add)."""
    P = int(np.asarray(plen, dtype=np.int64).sum())
    return 2.0 * w.R * w.Hq * P * (w.dk + w.dv)


def load_traffic():
    """ncu DRAM bytes per launch, keyed by kernel, with the source digest they were taken at."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def source_digest(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "tree_speculative_decoding_tsd_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


CALL_SOURCES = {
    "build": ["tsd_tree_build.cu", "tsd_scan.cuh", "tsd_common.cuh"],
    "build_conditioned": ["tsd_tree_cond.cu", "tsd_common.cuh"],
    "verify": ["tsd_verify.cu", "tsd_verify_tc.cu", "tsd_verify_mla.cu", "tsd_verify_mma.cu",
               "tsd_verify.cuh", "tsd_tcgen05.cuh", "tsd_common.cuh"],
    "accept": ["tsd_accept.cu", "tsd_scan.cuh", "tsd_commit.cuh", "tsd_common.cuh"],
    "commit": ["tsd_commit.cu", "tsd_commit.cuh", "tsd_common.cuh"],
    "accept_commit": ["tsd_accept.cu", "tsd_scan.cuh", "tsd_commit.cuh", "tsd_common.cuh"],
}


# ---------------------------------------------------------------- ours ----

def run_ours(args, dist, config=None, lite=False):
    """Measure one workload.  lite: the whole step and the per-call times only
    (no end-to-end, adaptive or paged legs)."""
    import tree_speculative_decoding_tsd_gb300 as T
    from tree_speculative_decoding_tsd_gb300.step import TreeVerifyStep

    config = config or args.config
    dev = torch.device("cuda", dist.local)
    torch.cuda.set_device(dev)
    w0 = W.WORKLOADS[config]
    w, host, d = make_inputs(w0, dev, dist.rank)
    step = TreeVerifyStep.for_workload(w, dev)
    stream = torch.cuda.Stream(device=dev)

    # target logits follow the tree's depths: build the tree once, untimed
    with torch.cuda.stream(stream):
        step.build(d["probs"], d["root"], stream)
    stream.synchronize()
    depth = step.tree.depth.cpu()
    host["tl"] = W.target_logits(w, depth, host["logits"])
    d["tl"] = host["tl"].to(dev)
    plen0 = d["plen"].clone()
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)

    args_step = (d["probs"], d["root"], d["q"], d["kc"], d["vc"], d["plen"], d["kt"], d["vt"],
                 d["tl"])

    def one_step():
        step.run(*args_step, stream=stream)

    def prep():
        d["plen"].copy_(plen0)
        flush.zero_()

    # warm-up (eager), then capture the step as a graph
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            prep()
            one_step()
    stream.synchronize()
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            one_step()
        with torch.cuda.stream(stream):
            for _ in range(max(3, args.warmup)):
                prep()
                graph.replay()
        stream.synchronize()

    # ---- timed region A: the whole step ----
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = Clocks(dev)
    dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter()
    clocks.begin()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            prep()
            ev[i][0].record(stream)
            if graph is not None:
                graph.replay()
            else:
                one_step()
            ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    clocks.end()
    dist.barrier()
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = dist.max(statistics.mean(step_ms))
    median_ms = statistics.median(step_ms)

    # ---- timed region B: per-call durations (eager) ----
    calls = ["build", "verify", "accept", "commit", None, "accept_commit"]
    evc = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            prep()
            e = evc[i]
            e[0].record(stream)
            step.build(d["probs"], d["root"], stream)
            e[1].record(stream)
            step.verify(d["q"], d["kc"], d["vc"], d["plen"], d["kt"], d["vt"], stream)
            e[2].record(stream)
            step.accept(d["tl"], stream)
            e[3].record(stream)
            step.commit(d["kt"], d["vt"], d["kc"], d["vc"], d["plen"], stream)
            e[4].record(stream)
            # the same walk and commit as one call (tsd_accept_commit), from
            # the same state
            prep()
            e[5].record(stream)
            step.accept_commit(d["tl"], d["kt"], d["vt"], d["kc"], d["vc"], d["plen"], stream)
            e[6].record(stream)
    torch.cuda.synchronize(dev)
    per_call = {c: statistics.mean(evc[i][j].elapsed_time(evc[i][j + 1]) for i in range(args.steps))
                for j, c in enumerate(calls) if c is not None}
    err_word = int(step.err[0].item())

    e2e = adaptive = paged = None
    if not lite:
        # ---- e2e: host buffers through the Python API ----
        e2e = run_e2e(args, step, host, d, dev, stream, plen0)
        # ---- cost-aware adaptive budget (tsd_tree_build_adaptive) ----
        adaptive = run_adaptive(args, w, step, d, dev, stream)
        # ---- the same verify through a shuffled page pool ----
        paged = run_paged(args, w, step, d, dev, stream, plen0)

    nodes = w.B * w.D
    value = nodes * dist.world / (ms / 1e3)
    algo, kv_bytes = algorithmic_bytes(w, host["plen"].numpy())
    hbm_peak, peak_kind = load_peaks()
    dominant = max(("build", "verify", "accept"), key=lambda c: per_call[c])
    achieved = algo[dominant] / (per_call[dominant] / 1e3) / 1e9
    # latent heads: the verify call is a dense contraction (about 2200 flop per
    # byte of KV), so its roofline is the tensor pipe
    tensor_bound = w.v_aliases_k and dominant == "verify"
    traffic = load_traffic().get(f"{config}:{dominant}")
    traffic_val = None
    if traffic and traffic.get("digest") == source_digest(CALL_SOURCES[dominant]):
        traffic_val = traffic.get("bytes_per_launch")
    n_verify_kernels = 2 if step.ws_verify.numel() > 16 else 1
    # build: top-k scan + tree; verify; accept + commit: argmax scan + walk (which commits)
    launches_per_step = 2 + n_verify_kernels + 2

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "nodes/s",
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded, shapes and distributions of the workload)",
        "config": {"workload": workload_desc(w), "nodes_per_step": nodes,
                   "launch": "cuda_graph" if graph is not None else "eager",
                   "streams": ("2 (target argmax beside the attention)"
                               if step.overlap_argmax else "1"),
                   "l2": "flushed before every timed step (memset of 2x L2, outside the events)",
                   "parallelism": f"replicas x{dist.world} (independent requests)"},
        "step_latency_us": {"mean": round(ms * 1e3, 2), "median": round(median_ms * 1e3, 2)},
        "per_call_us": {c: round(v * 1e3, 2) for c, v in per_call.items()},
        "attn_kv_gbs": round(kv_bytes / (per_call["verify"] / 1e3) / 1e9, 1),
        "attn_kv_frac_of_hbm": round(kv_bytes / (per_call["verify"] / 1e3) / 1e9 / hbm_peak, 4),
        "roofline": {"kernel": dominant, "bound": "hbm", "achieved": round(achieved, 1),
                     "peak": hbm_peak, "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": algo[dominant], "traffic": traffic_val},
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "launches_per_step": launches_per_step,
        "clocks": clk,
        "wall_s_timed_region": round(t_wall, 4),
        "device_err_word": err_word,
        "mean_accept_len": float(step.walk.accept_len.float().mean().item()),
        "adaptive": adaptive,
        "paged": paged,
    }
    if tensor_bound:
        tpeak, tkind = load_tensor_peak()
        fl = verify_flops(w, host["plen"].numpy())
        tf = fl / (per_call["verify"] / 1e3) / 1e12
        line["roofline"] = {"kernel": "verify", "bound": "tensor", "achieved": round(tf, 1),
                            "peak": tpeak, "unit": "TFLOP/s", "frac": round(tf / tpeak, 4),
                            "peak_source": f"{tkind} (MEASURED_PEAKS.json bf16_tflops, burst)"
                            if tkind == "measured" else "fallback 1.9 PF/s",
                            "algorithmic_flops_per_launch": fl, "traffic": traffic_val,
                            "algorithmic_bytes_per_launch": algo["verify"]}
    if lite:
        for key in ("e2e", "adaptive", "paged", "gpu_launches", "wall_s_timed_region"):
            line.pop(key, None)
    del step, d
    torch.cuda.empty_cache()
    return line, w, host


def run_paged(args, w, step, d, dev, stream, plen0, page_size=128):
    """tsd_tree_verify_attn_paged on the workload's cache scattered over a
    shuffled pool of 128-token pages (per-call CUDA events, eager), next to the
    contiguous verify of the same step."""
    import tree_speculative_decoding_tsd_gb300 as T
    cap = -(-w.cap // page_size) * page_size
    mp = cap // page_size
    g = torch.Generator(device="cpu").manual_seed(1234)
    perm = torch.randperm(w.B * mp, generator=g).to(dev)

    def to_pool(c):
        if c is None:
            return None
        c = torch.nn.functional.pad(c, (0, 0, 0, cap - c.shape[2]))
        pages = c.view(w.B, w.Hkv, mp, page_size, c.shape[3]).permute(0, 2, 1, 3, 4)
        pool = torch.empty((w.B * mp, w.Hkv, page_size, c.shape[3]), dtype=c.dtype, device=dev)
        pool[perm] = pages.reshape(w.B * mp, w.Hkv, page_size, c.shape[3])
        return pool

    kpool, vpool = to_pool(d["kc"]), to_pool(d["vc"])
    table = perm.view(w.B, mp).to(torch.int32).contiguous()
    desc = T.make_desc(w.B, w.R, w.Hq, w.Hkv, w.dk, w.dv, cap, w.torch_dtype, w.v_aliases_k,
                       w.scale)
    ws = T.workspace(T.tsd_verify_workspace_size(desc), dev)
    t = step.tree
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        d["plen"].copy_(plen0)
        for i in range(3 + args.steps):
            if i >= 3:
                ev[i - 3][0].record(stream)
            T.tsd_tree_verify_attn_paged(desc, d["q"], kpool, vpool, table, page_size, d["plen"],
                                         d["kt"], d["vt"], t.mask, step.out, step.lse, ws,
                                         step.err, stream)
            if i >= 3:
                ev[i - 3][1].record(stream)
    torch.cuda.synchronize(dev)
    us = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3
    del kpool, vpool
    return {"verify_us": round(us, 2), "page_size": page_size, "pages": w.B * mp}


def run_adaptive(args, w, step, d, dev, stream):
    """Cost model fitted to this GPU's own step latencies at budgets D/4, D/2, D
    (convex, non-decreasing in n), then tsd_tree_build_adaptive timed per call
    with CUDA events; reports the per-call time and the kept node counts."""
    size = w.B * w.cap * w.Hkv * (w.dk + (0 if w.v_aliases_k else w.dv))
    if size > 2e8:
        return {"skipped": "synthetic inputs for the calibration sweep too large to generate "
                           "in the default run"}
    try:
        from tree_speculative_decoding_tsd_gb300 import costmodel
        ell = int(np.mean(W.prefix_lens(w).numpy()))
        budgets = sorted({max(1, w.D // 4), max(1, w.D // 2), w.D})
        cost_d, samples = costmodel.measure(w, budgets, [ell], steps=5, warmup=2, device=dev)
        model = costmodel.CostModel.from_samples(cost_d, samples)
    except ImportError as e:
        return {"skipped": f"cost fit unavailable: {e}"}
    cd, cv = model.tables([ell] * w.B, w.D)
    cd, cv = torch.from_numpy(cd).to(dev), torch.from_numpy(cv).to(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            step.build_adaptive(d["probs"], d["root"], cd, cv, stream)
        for a, b in ev:
            a.record(stream)
            step.build_adaptive(d["probs"], d["root"], cd, cv, stream)
            b.record(stream)
    torch.cuda.synchronize(dev)
    n = step.n_nodes.cpu().numpy()
    return {"build_adaptive_us": round(statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3, 2),
            "mean_nodes": float(n.mean()), "min_nodes": int(n.min()), "max_nodes": int(n.max()),
            "D_max": w.D, "cost_model": {"cost_d_us": round(cost_d, 2), "prefix_len": ell,
                                         "budgets": budgets,
                                         "verify_side_us": [round(x, 2) for x in samples[ell][1]]}}


def run_e2e(args, step, host, d, dev, stream, plen0):
    """Same step through the Python API with host (pinned) inputs: H2D of the
    step's inputs, the four calls, D2H of the results, all inside the events.
    Up to 64 MiB of inputs per step the copies go in order on the compute
    stream into the buffers of a captured step, which is then replayed (the
    documented TreeVerifyStep.capture flow: no per-call host work, which
    otherwise bounds a step this small); above it they run on two copy
    streams (the drafter's outputs, then the attention inputs on one; the
    target logits on the other) and each call waits only for its own inputs,
    so the copies overlap the build and the attention.  The persistent KV
    cache stays resident."""
    names = ["probs", "root", "q", "kt", "vt", "tl", "plen"]
    pinned = {n: host[n].pin_memory() for n in names if host.get(n) is not None}
    dbuf = {n: torch.empty_like(pinned[n], device=dev) for n in pinned}
    res = [step.walk.accept_len, step.walk.accept_rows, step.walk.bonus, step.walk.chain_id,
           step.tree.token]
    outs = [torch.empty(r.shape, dtype=r.dtype, pin_memory=True) for r in res]
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = sum(t.numel() * t.element_size() for t in outs)
    overlap = h2d > (64 << 20)
    copy1 = torch.cuda.Stream(device=dev)
    copy2 = torch.cuda.Stream(device=dev)
    groups = [(copy1, "build", ["probs", "root", "plen"]), (copy1, "verify", ["q", "kt", "vt"]),
              (copy2, "accept", ["tl"])]
    graph = None
    if not overlap and not args.no_graph:
        # the documented replay flow: the step captured once on these device
        # buffers, then per step refill them in place and replay
        for k in pinned:
            dbuf[k].copy_(pinned[k])
        graph = step.capture(dbuf["probs"], dbuf["root"], dbuf["q"], d["kc"], d["vc"],
                             dbuf["plen"], dbuf["kt"], dbuf.get("vt"), dbuf["tl"], stream=stream)
        stream.synchronize()
    evs = []
    n = max(3, args.steps // 2)
    for i in range(n + 2):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        if graph is not None:
            with torch.cuda.stream(stream):
                for k in pinned:
                    dbuf[k].copy_(pinned[k], non_blocking=True)
                graph.replay()
                for o, r in zip(outs, res):
                    o.copy_(r, non_blocking=True)
                b.record(stream)
            b.synchronize()
            if i >= 2:
                evs.append(a.elapsed_time(b))
            continue
        ready = {}
        for cs, call, group in groups:
            cs = cs if overlap else stream
            if overlap:
                cs.wait_event(a)
            with torch.cuda.stream(cs):
                for k in group:
                    if k in pinned:
                        dbuf[k].copy_(pinned[k], non_blocking=True)
                if overlap:
                    ready[call] = torch.cuda.Event()
                    ready[call].record(cs)
        with torch.cuda.stream(stream):

            def need(call):
                if call in ready:
                    stream.wait_event(ready[call])

            need("build")
            step.build(dbuf["probs"], dbuf["root"], stream)
            need("verify")
            step.verify(dbuf["q"], d["kc"], d["vc"], dbuf["plen"], dbuf["kt"], dbuf.get("vt"),
                        stream)
            need("accept")
            step.accept_commit(dbuf["tl"], dbuf["kt"], dbuf.get("vt"), d["kc"], d["vc"],
                               dbuf["plen"], stream)
            for o, r in zip(outs, res):
                o.copy_(r, non_blocking=True)
            b.record(stream)
        b.synchronize()
        if i >= 2:
            evs.append(a.elapsed_time(b))
    ms = statistics.mean(evs)
    w_nodes = step.B * step.D
    return {"value": round(w_nodes / (ms / 1e3), 1), "unit": "nodes/s",
            "ms_per_step": round(ms, 5), "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h),
            "copies": "two copy streams, each call waits for its inputs" if overlap
                      else "in order on the compute stream, then one graph replay of the step"
                      if graph is not None else "in order on the compute stream",
            "note": "inputs copied from pinned host memory and results read back every step; "
                    "the persistent KV cache stays resident"}


# ------------------------------------------------------------ CPU oracle --

def oracle_step(w, host, b_sel, nthreads=0):
    """The whole step in the CPU oracle for requests b_sel (the same inputs)."""
    import oracle
    sl = slice(b_sel[0], b_sel[-1] + 1)
    probs = host["probs"][sl].numpy()
    tp, ti = oracle.topk(probs, w.k, nthreads)
    enum_paths = sum(w.k ** s for s in range(1, w.S + 1))
    tree = oracle.tree(tp, ti, w.D, host["root"][sl].numpy(),
                       method="enum" if enum_paths <= 4_000_000 else "beam")
    kv = lambda t: None if t is None else W.bits(t[sl])  # noqa: E731
    oracle.verify_attn(kv(host["q"]), kv(host["kc"]), kv(host["vc"]), host["plen"][sl].numpy(),
                       kv(host["kt"]), kv(host["vt"]), tree["mask"], w.scale,
                       v_aliases_k=w.v_aliases_k, dv=w.dv, nthreads=nthreads)
    tgt = oracle.argmax(host["tl"][sl].numpy(), nthreads)
    walk = oracle.accept_walk(tgt, tree, w.S)
    kc = W.bits(host["kc"][sl]).copy()
    vc = None if host["vc"] is None else W.bits(host["vc"][sl]).copy()
    oracle.commit(W.bits(host["kt"][sl]), None if host["vt"] is None else W.bits(host["vt"][sl]),
                  walk["accept_rows"], walk["accept_len"], kc, vc, host["plen"][sl].numpy().copy(),
                  w.S, v_aliases_k=w.v_aliases_k)


def cpu_baseline(w, host, seconds, min_steps=1):
    import oracle
    oracle.build()
    cores = oracle.hardware_threads()
    n_req = 1
    t0 = time.perf_counter()
    steps = 0
    while True:
        oracle_step(w, host, [0], nthreads=cores)
        steps += 1
        if time.perf_counter() - t0 >= seconds or steps >= 1000:
            if steps >= min_steps:
                break
    t = (time.perf_counter() - t0) / steps
    # the same step on one thread (one step at least, about a third of the budget)
    t1_0 = time.perf_counter()
    steps1 = 0
    while True:
        oracle_step(w, host, [0], nthreads=1)
        steps1 += 1
        if time.perf_counter() - t1_0 >= seconds / 3 or steps1 >= 1000:
            break
    t1 = (time.perf_counter() - t1_0) / steps1
    return {"value": round(n_req * w.D / t, 3), "unit": "nodes/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{steps} full oracle step(s) of request 0 of the {w.name} workload "
                      f"({w.D} nodes each; all {w.R * w.Hq} attention rows in fp64), "
                      f"{t:.3f} s per step",
            "s_per_step_all_cores": round(t, 4),
            "s_per_step_one_thread": round(t1, 4)}


def run_reference(args, dist):
    if dist.rank != 0:
        return None
    w = W.WORKLOADS[args.config]
    host = {"probs": W.draft_probs(w), "root": W.root_tokens(w), "plen": W.prefix_lens(w),
            "q": W.queries(w)}
    host["kc"], host["vc"] = W.kv_cache(w)
    host["kt"], host["vt"] = W.tree_kv(w)
    import oracle
    tp, ti = oracle.topk(host["probs"][:1].numpy(), w.k)
    depth = np.zeros((w.B, w.R), np.int32)
    depth[:1] = oracle.tree(tp, ti, w.D, host["root"][:1].numpy(), method="beam")["depth"]
    host["tl"] = W.target_logits(w, torch.from_numpy(depth))
    cores = oracle.hardware_threads()
    for _ in range(args.warmup):
        oracle_step(w, host, [0], nthreads=cores)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(w, host, [0], nthreads=cores)
        times.append(time.perf_counter() - t0)
    t = statistics.mean(times)
    v = round(w.D / t, 3)
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "nodes/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": workload_desc(w)},
            "cpu_baseline": {"value": v, "unit": "nodes/s", "cores": cores, "kind": "oracle",
                             "sample": f"request 0 of the {w.name} workload per step "
                                       f"({w.D} nodes; full oracle step)"},
            "e2e": {"value": v, "unit": "nodes/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    dist = Dist()
    try:
        if args.impl == "reference":
            line = run_reference(args, dist)
            if line is not None:
                print(json.dumps(line), flush=True)
            return
        line, w, host = run_ours(args, dist)
        also = [c for c in args.also.split(",") if c and c != args.config]
        if also:
            line["also"] = {}
            for c in also:
                sub, _, _ = run_ours(args, dist, config=c, lite=True)
                line["also"][c] = {k: sub[k] for k in (
                    "value", "unit", "ms_per_step", "config", "step_latency_us", "per_call_us",
                    "attn_kv_gbs", "attn_kv_frac_of_hbm", "roofline", "clocks",
                    "device_err_word", "launches_per_step")}
        if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, host, args.cpu_seconds)
        elif dist.rank == 0:
            line["cpu_baseline"] = None
        if dist.rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
