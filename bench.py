#!/usr/bin/env python
"""Throughput of token-tree verification on GB300: tree nodes verified per second.

One step = one pass of the whole hot path over one batch of synthetic input:
one layer of tree attention (the kernel builds the topology-aware mask from
parent[] itself) and the verification of the workload (greedy and/or
multi-step speculative sampling).  Verification reads only the step's logits
and proposals, not the attention output, so it runs on a second stream
concurrently with the attention launch (--serial: after it).  `value` = tree
nodes verified / s over the whole job with inputs resident in HBM; `e2e` = the
same metric when every step also copies its inputs from pinned host memory and
reads its results back.

Timing: W untimed warm-up steps (every CUDA graph has been replayed once before
them), then exactly K steps between CUDA events on the launching stream,
bracketed by barrier + synchronize; each step replays a CUDA graph of the step
on one of R input copies whose total size is at least 4x the L2 cache (or one
copy that alone is), so every step reads its inputs from HBM.  Clocks are
sampled through NVML every few milliseconds during the timed region.  After
it, outside the timed region: the median of per-step times, the same steps as
plain launches (no graph), the serial composition, and each launch alone.  The
default run also measures every other workload the same way (`per_workload`).
Under torchrun each rank runs an independent replica (replicas only: no data
exchange) and the maximum time over ranks is reported.

`--impl reference` times the CPU oracle (the only reference implementation:
the pages ship no code) on the host cores over a bounded sample of the same
workload.
"""
import argparse
import hashlib
import json
import math
import os
import platform
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tree nodes verified/sec (attn+verify)"
UNIT = "nodes/s"
DEFAULT_WORKLOAD = "batch32-P2048-n16"  # the largest configuration that fits one GPU
# Every workload the bench line also reports in its per_workload record.
PER_WORKLOAD = ["llama7b-layer-P1024-n20", "batch8-ragged-merge64-mss", "gqa64x8-P32768-n128",
                "batch32-P2048-n16", "tiny-f32-P128-n16"]


def parse_args():
    p = argparse.ArgumentParser(description=__doc__)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-per-workload", action="store_true", help="skip the per_workload record")
    p.add_argument("--serial", action="store_true",
                   help="verification after attention on one stream (default: concurrent on a second stream)")
    p.add_argument("--no-e2e", action="store_true", help="profiling runs: skip e2e, baselines, JSON line")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU oracle sample budget")
    p.add_argument("--top-k", type=int, default=0, help="stochastic verification against the top-k warped LLM law")
    p.add_argument("--top-p", type=float, default=1.0, help="... and top-p (needs --top-k)")
    p.add_argument("--row", choices=["step", "kv_commit", "sequence_baseline", "tree_build"], default="step",
                   help="step: the hot path (attention + verification); kv_commit: the commit of the "
                        "accepted path that follows verification, timed alone; sequence_baseline: tree "
                        "attention against the same work done per root-to-leaf sequence; tree_build: "
                        "expansion (top-k children) and merge of token trees on the GPU")
    return p.parse_args()


# --------------------------------------------------------------------------- common


def whole_job_ms(ms_total, world, device):
    """Length of the timed region for the whole job: the largest over ranks
    (the job ends when its slowest replica does).  Every rank calls it."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms_total], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_total = float(t.item())
    return ms_total


def whole_job_value(ms_total, steps, nodes_per_step, world):
    """Tree nodes verified per second by the whole job: each of the `world`
    replicas verifies `nodes_per_step` nodes per step."""
    return world * nodes_per_step / (ms_total / steps * 1e-3)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def workload_inputs(spec):
    import workloads as W
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    gi = W.make_greedy_inputs(spec, trees) if spec.greedy else None
    si = W.make_stochastic_inputs(spec, trees) if spec.stochastic else None
    return trees, att, gi, si


WARP = {}  # top_k / top_p of the stochastic verification, when warped
MIN_GRAPH_LAUNCHES = 4  # steps (or launches of one kind) per captured timing graph, at least


def config_of(spec, extra=None):
    cfg = {"workload": spec.name, "B": spec.B, "Hq": spec.Hq, "Hkv": spec.Hkv, "D": spec.D,
           "prefix": list(spec.prefix) if isinstance(spec.prefix, tuple) else spec.prefix,
           "nodes_per_request": spec.nodes, "vocab": spec.V,
           "verify": "+".join(v for v, on in (("greedy", spec.greedy), ("stochastic", spec.stochastic)) if on),
           "tree": spec.tree,
           # The same statement in both arms, so that their configs compare equal.
           "l2": "inputs read from HBM every step: rotating input copies totalling >= 4x L2 "
                 "(one copy when it alone is that large)",
           "parallelism": "replicas"}
    if WARP:
        cfg["warp"] = dict(WARP)
    if extra:
        cfg.update(extra)
    return cfg


def attention_bytes(spec, trees):
    """Algorithmic bytes of one tree-attention launch: every (request, KV head)
    reads its K and V rows 0 .. P_b+n_b-1 once, Q is read once, O written once."""
    esz = 2 if spec.dtype == "bf16" else 4
    sizes = np.diff(trees.node_offsets)
    keys = int((trees.prefix_len + sizes).sum())
    N = int(trees.node_offsets[-1])
    return 2 * keys * spec.Hkv * spec.D * esz + 2 * N * spec.Hq * spec.D * esz


def attention_flops(spec, trees):
    """Algorithmic FLOPs of one tree-attention launch: per query row and per
    key it sees (the prefix, then the node and its ancestors), one D-long dot
    product for the score and one for the value update, 2 FLOPs per MAC."""
    import workloads as W
    offs = trees.node_offsets
    keys_seen = 0.0
    for b in range(len(offs) - 1):
        depth = W.tree_depths(np.asarray(trees.parent[offs[b]:offs[b + 1]]))
        keys_seen += float(len(depth) * int(trees.prefix_len[b]) + (depth.astype(np.int64) + 1).sum())
    return 4.0 * spec.D * spec.Hq * keys_seen


def verify_bytes(spec, trees, visited_rows=None, rejected_rows=0):
    """Greedy: every logits row once (the one-pass verifier takes every row's
    argmax in parallel instead of walking the rows one after another).
    Stochastic: the LLM row of every node the walk visits, plus the full
    proposal row of each rejected child (an accepted child needs one entry);
    without a visit count, every LLM row."""
    N = int(trees.node_offsets[-1])
    b = 0
    if spec.greedy:
        b += N * spec.V * 4
    if spec.stochastic:
        b += ((N if visited_rows is None else visited_rows) + rejected_rows) * spec.V * 4
    return b


class ClockSampler:
    """nvidia-smi samples (200 ms) while the benchmark runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                self.samples.append((time.time(), f))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        win = [f for (t, f) in self.samples if t0 - 0.25 <= t <= t1 + 0.25]
        if not win:
            win = [f for (_, f) in self.samples]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"],
                    "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(f[1]) for f in win if num(f[1]) is not None]
        smax = [num(f[2]) for f in win if num(f[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for f in win for i in range(4) if f[5 + i].lower().startswith("active")})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons, "samples": len(win),
                "power_w_max": max((num(f[3]) or 0.0) for f in win)}


def _peaks_file():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f)
    return None


def measured_peaks(sustained=False):
    """(HBM GB/s, dense bf16 TFLOP/s, which): the burst tensor figure for a
    kernel timed alone, the sustained one for a kernel inside a long run."""
    j = _peaks_file()
    if j is not None:
        tf = j.get("bf16_tflops_sustained", j["bf16_tflops"]) if sustained else j["bf16_tflops"]
        return float(j["hbm_gbs"]), float(tf), "measured"
    return 6800.0, (1700.0 if sustained else 1900.0), "fallback"


def measured_sm_max_mhz():
    j = _peaks_file()
    return float(j.get("sm_max_mhz", 2070.0)) if j is not None else 2070.0


class NvmlClockSampler:
    """SM clock, maximum SM clock, power and clock-event reasons of the bench's
    GPU, read through NVML's C library every few milliseconds by a thread, so
    that even a timed region of a few milliseconds has samples.  Queries only:
    nothing here changes a setting of the GPU."""

    REASON_BITS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
                   0x4: "sw_power_cap"}

    def __init__(self, ids, period_s=0.002):
        import ctypes
        self.samples = []
        self.period = period_s
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        ok = False
        for kind, key in ids:
            if kind == "uuid":
                ok = self.lib.nvmlDeviceGetHandleByUUID(key.encode(), ctypes.byref(self.h)) == 0
            elif kind == "pci":
                ok = self.lib.nvmlDeviceGetHandleByPciBusId_v2(key.encode(), ctypes.byref(self.h)) == 0
            elif kind == "index":
                ok = self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(int(key)), ctypes.byref(self.h)) == 0
            if ok:
                self.which = "%s %s" % (kind, key)
                break
        if not ok:
            raise OSError("no NVML handle for the device")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        self.stop_flag = False
        self.thread = None

    def mark(self):
        """One sample taken now by the calling thread (kept with the others)."""
        s = self.sample()
        if s is not None:
            self.samples.append(s)

    def sample(self):
        import ctypes
        t = time.time()
        sm, smax, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(sm)) != 0:  # NVML_CLOCK_SM
            return None
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(smax))
        power = float(mw.value) / 1e3 if self.lib.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(mw)) == 0 else None
        reasons = int(rs.value) if self.reasons_fn(self.h, ctypes.byref(rs)) == 0 else 0
        return (t, float(sm.value), float(smax.value), power, reasons)

    def _run(self):
        while not self.stop_flag:
            # (NVML's queries take milliseconds each on this part, so the
            # period is a lower bound.)
            s = self.sample()
            if s is not None:
                self.samples.append(s)
            time.sleep(self.period)

    def start(self):
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def stop(self):
        self.stop_flag = True
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        note = None
        if not win:  # nothing inside: the samples nearest to either end (within 50 ms)
            win = [s for s in self.samples if t0 - 0.05 <= s[0] <= t1 + 0.05]
            note = "nearest samples within 50 ms of the region (taken right at its edges when it is short)"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no NVML samples"], "samples": 0,
                    "source": "nvml"}
        reasons = sorted({name for s in win for bit, name in self.REASON_BITS.items() if s[4] & bit})
        out = {"sm_mhz": float(np.median([s[1] for s in win])), "sm_max_mhz": max(s[2] for s in win),
               "sm_mhz_min": min(s[1] for s in win), "reasons": reasons, "samples": len(win),
               "power_w_max": max((s[3] or 0.0) for s in win), "source": "nvml (%s), every %g ms"
               % (self.which, self.period * 1e3)}
        if note:
            out["note"] = note
        return out


class ClockRecord:
    """Clock samples during the bench: NVML (a few ms apart) when its library
    loads, else nvidia-smi (200 ms apart)."""

    def __init__(self, dev):
        import torch
        props = torch.cuda.get_device_properties(dev)
        ids = []
        uuid = getattr(props, "uuid", None)
        if uuid is not None:
            u = str(uuid)
            ids += [("uuid", u if u.startswith("GPU-") else "GPU-" + u)]
        if hasattr(props, "pci_bus_id") and hasattr(props, "pci_device_id"):
            ids.append(("pci", "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                                     props.pci_device_id)))
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        parts = [x.strip() for x in vis.split(",") if x.strip()]
        if parts and all(x.isdigit() for x in parts) and dev.index < len(parts):
            ids.append(("index", parts[dev.index]))
        elif not parts:
            ids.append(("index", dev.index))
        try:
            self.impl = NvmlClockSampler(ids)
        except (OSError, AttributeError):
            self.impl = ClockSampler(int(ids[-1][1]) if ids and ids[-1][0] == "index" else dev.index)

    def start(self):
        self.impl.start()

    def mark(self):
        """A synchronous sample (NVML only): taken right before and right after
        a timed region too short for the sampling thread to see."""
        if hasattr(self.impl, "mark"):
            self.impl.mark()

    def stop(self):
        self.impl.stop()

    def summary(self, t0, t1):
        return self.impl.summary(t0, t1)


KERNEL_SOURCES = {
    # What decides one attention launch's DRAM traffic: the kernel, the device
    # headers it includes and the host planner that cuts the work.
    "tree_attn_keys_kernel": ["tsv_attention_keys.cu"],
    "tree_attn_tc_kernel": ["tsv_attention_tc.cu"],
    "tree_attn_tc1_kernel": ["tsv_attention_tc1.cu"],
    "tree_attn_simt_kernel": ["tsv_attention_simt.cu"],
}
KERNEL_COMMON = ["tsv_attention_common.cuh", "tsv_device.cuh", "tsv_internal.h", "tsv_api.cu"]


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tree_speculative_verification_attention_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel] + KERNEL_COMMON:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload, kernel):
    """DRAM bytes per attention launch from the committed ncu summary, if it
    was taken on the current sources of that kernel; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        j = json.load(f)
    e = j.get(workload)
    if not e or e.get("kernel") != kernel or e.get("source_hash") != kernel_source_hash(kernel):
        return None
    return float(e["dram_bytes_per_launch"])


# --------------------------------------------------------------------------- CPU oracle


def oracle_step_time(spec, trees, att, gi, si, budget_s, heads_sample=None):
    """Times the oracle on a bounded sample of one step and extrapolates to the
    whole step.  Returns (seconds per full step, cores, sample description)."""
    import oracle
    Hkv = spec.Hkv
    G = spec.Hq // Hkv
    kv_heads = list(range(Hkv)) if heads_sample is None else list(range(min(Hkv, heads_sample)))
    qh = [g * G + r for g in kv_heads for r in range(G)]
    q = att.q[:, qh].float().numpy()
    k = att.k_cache[:, :, kv_heads].float().numpy()
    v = att.v_cache[:, :, kv_heads].float().numpy()
    reps, t_att, t_ver = 0, 0.0, 0.0
    t_begin = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        oracle.tree_attention(q, k, v, trees.prefix_len, trees.node_offsets, trees.parent)
        t1 = time.perf_counter()
        if gi is not None:
            oracle.verify_greedy(gi.logits, gi.tokens, trees.parent, trees.node_offsets)
        if si is not None:
            oracle.verify_stochastic(si.llm_logits, si.ssm_probs, si.tokens, trees.parent,
                                     trees.node_offsets, si.u_accept, si.u_sample, **WARP)
        t2 = time.perf_counter()
        t_att += t1 - t0
        t_ver += t2 - t1
        reps += 1
        if time.perf_counter() - t_begin >= budget_s:
            break
    scale = Hkv / len(kv_heads)
    per_step = (t_att * scale + t_ver) / reps
    sample = ("%d repetition(s) of: tree attention over %d of %d KV heads (x%.0f to the full layer) + "
              "the full verification" % (reps, len(kv_heads), Hkv, scale))
    return per_step, oracle.num_threads(), sample


def host_cpu_model(cpuinfo="/proc/cpuinfo"):
    """The host CPU as the OS describes it (x86: the model name; Arm: the
    implementer and part codes), else the machine type."""
    fields = {}
    try:
        with open(cpuinfo) as f:
            for line in f:
                key, sep, val = line.partition(":")
                if sep and key.strip() not in fields:
                    fields[key.strip()] = val.strip()
    except OSError:
        pass
    if fields.get("model name"):
        return fields["model name"]
    if "CPU part" in fields:
        return "%s (CPU implementer %s, part %s)" % (platform.machine(), fields.get("CPU implementer", "?"),
                                                     fields["CPU part"])
    return platform.machine() or None


def oracle_baseline(spec, trees, att, gi, si, budget_s, heads, n_nodes):
    """The cpu_baseline entry: the oracle on all host cores over a sample of
    about budget_s seconds, then once more on one core (one repetition)."""
    import oracle
    per_step, cores, sample = oracle_step_time(spec, trees, att, gi, si, budget_s, heads)
    oracle.set_num_threads(1)
    try:
        one_core, _, _ = oracle_step_time(spec, trees, att, gi, si, 0.0, heads)
    finally:
        oracle.set_num_threads(cores)
    return {"value": n_nodes / per_step, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
            "single_core": {"value": n_nodes / one_core, "unit": UNIT, "cores": 1,
                            "sample": "one repetition of the same sample"},
            "nproc": os.cpu_count(), "cpu_model": host_cpu_model()}


def choose_heads_sample(spec, trees):
    """KV heads whose oracle attention takes about 0.5 s at ~1 GFLOP/s per core."""
    sizes = np.diff(trees.node_offsets)
    flops_per_head = 4.0 * spec.D * float(((trees.prefix_len + sizes) * sizes).sum()) * (spec.Hq // spec.Hkv)
    import oracle
    budget = 0.5 * 1e9 * max(1, oracle.num_threads())
    return max(1, min(spec.Hkv, int(budget // max(flops_per_head, 1.0))))


def run_reference(args, spec):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    trees, att, gi, si = workload_inputs(spec)
    n_nodes = int(trees.node_offsets[-1])
    heads = choose_heads_sample(spec, trees)
    per_step, cores, sample = oracle_step_time(spec, trees, att, gi, si, 0.0, heads)  # warm
    for _ in range(max(0, args.warmup - 1)):
        oracle_step_time(spec, trees, att, gi, si, 0.0, heads)
    total = 0.0
    for _ in range(args.steps):
        s, cores, sample = oracle_step_time(spec, trees, att, gi, si, 0.0, heads)
        total += s
    ms = 1e3 * total / args.steps
    value = n_nodes / (total / args.steps)
    base = oracle_baseline(spec, trees, att, gi, si, 0.0, heads, n_nodes)  # adds the one-core figure
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(spec), "reference_impl": "CPU fp64 oracle (the pages ship no code)",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "per step: " + sample, "single_core": base["single_core"],
                             "nproc": base["nproc"], "cpu_model": base["cpu_model"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU


class DeviceWorkload:
    """One workload on the device: R rotating copies of the step's inputs (their
    total is at least 4x the L2 cache, or one copy is already larger, so each
    step reads its inputs from HBM), each with its own outputs and workspaces,
    and the calls of one step.

    Within a step, verification reads only the given logits and proposals, so
    it does not wait for the attention launch: with ``overlap`` the
    verification launches follow attention on the same stream in the
    library's overlap mode (tsv_set_verify_overlap): they are launched once
    every CTA of the launch before them is resident, run in the SM room it
    leaves, and complete after it.  The stochastic walk starts beside
    attention at full size on the SMs attention leaves idle (a tensor-bound
    launch's spare SMs, a persistent launch's SMs as its tail frees them), and
    greedy verification beside both."""

    def __init__(self, spec, tsv, dev, stream, overlap=True):
        import torch
        self.spec, self.tsv, self.dev, self.stream, self.overlap = spec, tsv, dev, stream, overlap
        trees, att, gi, si = workload_inputs(spec)
        self.trees, self.att, self.gi, self.si = trees, att, gi, si
        self.B, self.N = spec.B, int(trees.node_offsets[-1])

        def to_dev(x):
            t = x if isinstance(x, torch.Tensor) else torch.as_tensor(np.ascontiguousarray(x))
            return t.to(dev)

        base = {"q": to_dev(att.q), "k": to_dev(att.k_cache), "v": to_dev(att.v_cache),
                "parent": to_dev(trees.parent), "offs": to_dev(trees.node_offsets),
                "plen": to_dev(trees.prefix_len)}
        if gi is not None:
            base.update(logits=to_dev(gi.logits), gtok=to_dev(gi.tokens))
        if si is not None:
            base.update(llm=to_dev(si.llm_logits), ssm=to_dev(si.ssm_probs), stok=to_dev(si.tokens),
                        ua=to_dev(si.u_accept), us=to_dev(si.u_sample))
        self.per_copy = sum(t.numel() * t.element_size() for t in base.values())
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.R = int(min(64, max(1, math.ceil(4 * l2 / self.per_copy))))
        self.copies = [base] + [{k: t.clone() for k, t in base.items()} for _ in range(self.R - 1)]
        # Steps (and attention launches) per captured graph: at least
        # MIN_GRAPH_LAUNCHES, cycling over the R copies, so a graph replay's own
        # launch gap is not charged to every step.  One copy streams at least
        # 4 x L2 when R is 1, so consecutive steps on it still start cold.
        self.L = max(self.R, MIN_GRAPH_LAUNCHES)
        # Verification alone reads only the logits and proposals: its graphs
        # cycle over Rv copies of those inputs, together at least 4 x L2 (the
        # full copies first, then clones of the verification inputs).
        vkeys = [k for k in ("logits", "gtok", "llm", "ssm", "stok", "ua", "us", "parent", "offs") if k in base]
        vbytes = sum(base[k].numel() * base[k].element_size() for k in vkeys)
        self.Rv = int(min(64, max(self.R, math.ceil(4 * l2 / vbytes))))
        self.vcopies = self.copies + [{k: base[k].clone() for k in vkeys} for _ in range(self.Rv - self.R)]
        self.Lv = max(self.Rv, MIN_GRAPH_LAUNCHES)
        h = tsv.handle(dev.index)
        B, N = self.B, self.N
        code = tsv.TSV_BF16 if spec.dtype == "bf16" else tsv.TSV_F32
        ws_attn = tsv.tsv_tree_attention_workspace_size(h, code, B, trees.prefix_len, trees.node_offsets, spec.Hq,
                                                        spec.Hkv, spec.D, False)
        ws_g = tsv.tsv_tree_verify_greedy_workspace_size(h, B, N, spec.V)
        ws_s = tsv.tsv_tree_verify_stochastic_workspace_size(h, B, N, spec.V)
        self.ws_sizes = (ws_attn, ws_g, ws_s)

        def make_state(c):
            st = {"status": torch.zeros(B, dtype=torch.int32, device=dev), "out": torch.empty_like(c["q"]),
                  "ws_attn": torch.zeros(max(ws_attn, 1), dtype=torch.uint8, device=dev),
                  "ws_g": torch.zeros(max(ws_g, 1), dtype=torch.uint8, device=dev),
                  "ws_s": torch.zeros(max(ws_s, 1), dtype=torch.uint8, device=dev)}
            mk = lambda: {k: torch.empty(n, dtype=torch.int32, device=dev) for k, n in
                          (("path", N), ("accept_len", B), ("bonus", B), ("n_tried", B), ("status", B))}
            st["g"], st["s"] = mk(), mk()
            return st

        self.states = [make_state(c) for c in self.copies]

        def make_vstate():  # verification workspaces and outputs of a verification-only copy
            st = {"ws_g": torch.zeros(max(ws_g, 1), dtype=torch.uint8, device=dev),
                  "ws_s": torch.zeros(max(ws_s, 1), dtype=torch.uint8, device=dev)}
            mk = lambda: {k: torch.empty(n, dtype=torch.int32, device=dev) for k, n in
                          (("path", N), ("accept_len", B), ("bonus", B), ("n_tried", B), ("status", B))}
            st["g"], st["s"] = mk(), mk()
            return st

        self.vstates = self.states + [make_vstate() for _ in range(self.Rv - self.R)]
        # Kernels per step: one attention launch (masks built and splits merged
        # inside; the fp32 CUDA-core path first prepares the ancestor bitsets in
        # a launch of its own), one per verification kind.
        self.kernels_per_step = (1 if spec.dtype == "bf16" else 2) + (gi is not None) + (si is not None)

    # ------------------------------------------------------------------ calls
    def attention(self, c, st):
        # The kernel builds the ancestor masks from parent[] itself (and
        # validates the tree), so tree preparation runs inside this launch.
        t = self.trees
        self.tsv.tree_attention(c["q"], c["k"], c["v"], t.prefix_len, t.node_offsets, c["plen"], c["offs"],
                                parent=c["parent"], anc=None, out=st["out"], workspace=st["ws_attn"],
                                status=st["status"])

    def greedy(self, c, st):
        self.tsv.tree_verify_greedy(c["logits"], c["gtok"], c["parent"], c["offs"], workspace=st["ws_g"],
                                    out=st["g"])

    def stochastic(self, c, st):
        self.tsv.tree_verify_stochastic(c["llm"], c["ssm"], c["stok"], c["parent"], c["offs"], c["ua"], c["us"],
                                        workspace=st["ws_s"], out=st["s"], **WARP)

    def verify(self, c, st):
        if self.gi is not None:
            self.greedy(c, st)
        if self.si is not None:
            self.stochastic(c, st)

    def step(self, c, st, overlap=None):
        overlap = self.overlap if overlap is None else overlap
        self.attention(c, st)
        if not overlap:
            self.verify(c, st)
            return
        with self.tsv.verify_overlap(overlap_kinds(self.tsv, self.gi is not None),
                                     device=self.dev.index):
            if self.si is not None:
                self.stochastic(c, st)  # leaves room beside its CTAs for greedy's
            if self.gi is not None:
                self.greedy(c, st)

    # ------------------------------------------------------------------ graphs
    def _graph(self, fn):
        import torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            fn()
        return g

    def capture(self):
        """CUDA graphs: L steps cycling over the R copies in one graph (so the
        host replays one graph per L steps and stays ahead of the GPU), one
        graph per copy, and graphs of L attention launches and of Lv launches
        of each verification alone (cycling over the Rv verification copies)."""
        import torch
        cs = list(zip(self.copies, self.states))
        vs = list(zip(self.vcopies, self.vstates))
        for c, st in cs:  # eager run once; checks the statuses
            self.step(c, st)
        for c, st in vs[self.R:]:
            self.verify(c, st)
        torch.cuda.synchronize()
        assert (self.states[0]["status"].cpu() == 0).all()
        cyc = [cs[i % self.R] for i in range(self.L)]
        vcyc = [vs[i % self.Rv] for i in range(self.Lv)]
        self.g_steps = self._graph(lambda: [self.step(c, st) for c, st in cyc])
        self.g_one = [self._graph(lambda c=c, st=st: self.step(c, st)) for c, st in cs]
        self.g_serial = self._graph(lambda: [self.step(c, st, overlap=False) for c, st in cyc])
        self.g_attn = self._graph(lambda: [self.attention(c, st) for c, st in cyc])
        self.g_greedy = self._graph(lambda: [self.greedy(c, st) for c, st in vcyc]) if self.gi is not None else None
        self.g_mss = self._graph(lambda: [self.stochastic(c, st) for c, st in vcyc]) if self.si is not None else None
        # Every graph is replayed once here, so none launches for the first time
        # inside a timed region.
        for g in [self.g_steps, self.g_serial, self.g_attn, self.g_greedy, self.g_mss] + self.g_one:
            if g is not None:
                g.replay()
        torch.cuda.synchronize()
        counted = graph_kernel_count(self.g_one[0])
        if counted is not None:
            assert counted == self.kernels_per_step, (counted, self.kernels_per_step)

    def run_steps(self, k):
        for _ in range(k // self.L):
            self.g_steps.replay()
        for i in range(k % self.L):
            self.g_one[i % self.R].replay()

    # ------------------------------------------------------------------ timing forms
    def _events(self, n):
        import torch
        return [torch.cuda.Event(enable_timing=True) for _ in range(n)]

    def graph_ms(self, g, launches_per_replay, reps):
        """Mean device time per launch of a pre-replayed graph, replayed reps times."""
        import torch
        e0, e1 = self._events(2)
        torch.cuda.synchronize()
        e0.record(self.stream)
        for _ in range(reps):
            g.replay()
        e1.record(self.stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (reps * launches_per_replay)

    def per_step_graph_ms(self, n):
        """Device time of each of n steps replayed one graph per step (events between steps)."""
        import torch
        ev = self._events(n + 1)
        torch.cuda.synchronize()
        ev[0].record(self.stream)
        for i in range(n):
            self.g_one[i % self.R].replay()
            ev[i + 1].record(self.stream)
        torch.cuda.synchronize()
        return [ev[i].elapsed_time(ev[i + 1]) for i in range(n)]

    def per_step_plain_ms(self, n):
        """Device time of each of n steps issued as plain launches from the host
        (no graph; the calls go through the C ABI every step)."""
        import torch
        cs = list(zip(self.copies, self.states))
        for c, st in cs[:3]:
            self.step(c, st)
        ev = self._events(n + 1)
        torch.cuda.synchronize()
        ev[0].record(self.stream)
        for i in range(n):
            c, st = cs[i % self.R]
            self.step(c, st)
            ev[i + 1].record(self.stream)
        torch.cuda.synchronize()
        return [ev[i].elapsed_time(ev[i + 1]) for i in range(n)]

    def walk_rows(self):
        """(visited, rejected) rows of copy 0's last stochastic walk, as the
        kernel reports them: accept_len + 1 visited nodes per request, and every
        child tried but not accepted (each needs its full proposal row)."""
        if self.si is None:
            return None, 0
        s = self.states[0]["s"]
        visited = int((s["accept_len"] + 1).sum().item())
        return visited, int((s["n_tried"] - s["accept_len"]).sum().item())

    def measure(self, n_steps):
        """The step and each of its launches alone, outside any timed region of the bench line."""
        reps = max(1, n_steps // self.L)
        vreps = max(1, n_steps // self.Lv)
        steps = self.per_step_graph_ms(n_steps)
        out = {"graph_mean_ms": self.graph_ms(self.g_steps, self.L, reps),
               "graph_median_ms": float(np.median(steps)),
               "serial_graph_mean_ms": self.graph_ms(self.g_serial, self.L, reps),
               "attention_ms": self.graph_ms(self.g_attn, self.L, reps)}
        if self.g_greedy is not None:
            out["greedy_ms"] = self.graph_ms(self.g_greedy, self.Lv, vreps)
        if self.g_mss is not None:
            out["stochastic_ms"] = self.graph_ms(self.g_mss, self.Lv, vreps)
        plain = self.per_step_plain_ms(n_steps)
        out["plain_median_ms"] = float(np.median(plain))
        out["plain_mean_ms"] = float(np.mean(plain))
        return out


def attention_kernel_name(spec, trees):
    G = spec.Hq // spec.Hkv
    sizes = np.diff(trees.node_offsets)
    keys_kernel = all(int(n) * G <= 64 for n in sizes) and 64 % G == 0
    tile_pairs = any(int(n) * G > 128 for n in sizes)  # some request has 2+ row tiles
    return ("tree_attn_simt_kernel" if spec.dtype != "bf16" else
            "tree_attn_keys_kernel" if keys_kernel else
            "tree_attn_tc_kernel" if tile_pairs else "tree_attn_tc1_kernel")


def overlap_kinds(tsv, greedy):
    """Overlap flags of a step's verification calls (stochastic first, then
    greedy): the stochastic walk beside attention at full size, on the SMs the
    launch leaves idle (a tensor-bound launch's spare SMs, a persistent
    launch's SMs as its tail frees them), and greedy beside the walk."""
    return (tsv.TSV_OVERLAP_GREEDY if greedy else 0) | tsv.TSV_OVERLAP_STOCHASTIC_FULL


def attention_exps(spec, trees):
    """Exponentials of one tree-attention launch: one per query row per key it sees."""
    return attention_flops(spec, trees) / (4.0 * spec.D)


def sfu_exp_rate(num_sms):
    """Exponentials per second: 32 ex2 per clock per SM (measured on this GPU by a
    throughput loop of ex2.approx.f32) at the maximum SM clock."""
    return 32.0 * num_sms * measured_sm_max_mhz() * 1e6


def rooflines(spec, trees, attn_ms, step_ms, walk_rows, num_sms):
    """(attention-launch roofline, step roofline).  The attention launch is
    timed alone (burst tensor peak); the step is a long run (sustained peak)."""
    peak, peak_tf, peak_kind = measured_peaks()
    peak_tf_sus = measured_peaks(sustained=True)[1]
    abytes, aflops, aexps = attention_bytes(spec, trees), attention_flops(spec, trees), attention_exps(spec, trees)
    kernel = attention_kernel_name(spec, trees)
    gbs = abytes / (attn_ms * 1e-3) / 1e9
    t_bytes, t_flops, t_exps = abytes / (peak * 1e9), aflops / (peak_tf * 1e12), aexps / sfu_exp_rate(num_sms)
    if spec.dtype == "bf16" and t_flops > t_bytes:
        tf = aflops / (attn_ms * 1e-3) / 1e12
        att = {"bound": "tensor", "achieved": tf, "peak": peak_tf, "unit": "TFLOP/s", "frac": tf / peak_tf,
               "peak_kind": peak_kind + " bf16_tflops (burst)"}
    else:
        att = {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
               "peak_kind": peak_kind + " hbm_gbs"}
    att.update({"traffic": recorded_traffic(spec.name, kernel), "kernel": kernel, "launch_ms": attn_ms,
                "algorithmic_bytes": abytes, "algorithmic_flops": aflops, "exponentials": aexps,
                "hbm_gbs": gbs, "hbm_frac": gbs / peak,
                "combined_frac": max(t_bytes, t_flops if spec.dtype == "bf16" else 0.0, t_exps) / (attn_ms * 1e-3)})
    vbytes = verify_bytes(spec, trees, *walk_rows)
    sbytes = abytes + vbytes
    sgbs = sbytes / (step_ms * 1e-3) / 1e9
    s_flops = aflops / (peak_tf_sus * 1e12) if spec.dtype == "bf16" else 0.0
    step = {"bound": "hbm", "achieved": sgbs, "peak": peak, "unit": "GB/s", "frac": sgbs / peak,
            "peak_kind": peak_kind + " hbm_gbs",
            "algorithmic_bytes": sbytes, "attention_bytes": abytes, "verify_bytes": vbytes,
            "stochastic_rows": {"visited_llm": walk_rows[0], "rejected_proposals": walk_rows[1]},
            "combined_frac": max(sbytes / (peak * 1e9), s_flops, t_exps) / (step_ms * 1e-3),
            "what": "KV + Q + O of the attention launch, every greedy logits row, the visited LLM rows and "
                    "rejected proposal rows of the stochastic walk; one step / step time"}
    return att, step


def workload_summary(spec, w, forms, step_ms, num_sms):
    """A compact record of one workload measured in the same run."""
    att, step = rooflines(spec, w.trees, forms["attention_ms"], step_ms, w.walk_rows(), num_sms)
    out = {"nodes": w.N, "step_ms": step_ms, "nodes_per_s": w.N / (step_ms * 1e-3),
           "attention": {k: att[k] for k in ("kernel", "launch_ms", "bound", "frac", "hbm_frac", "combined_frac")},
           "step_roofline": {k: step[k] for k in ("frac", "combined_frac", "algorithmic_bytes")},
           "rotating_copies": w.R, "steps_per_graph": w.L, "verification_copies": w.Rv}
    out["timing"] = {k: v for k, v in forms.items() if k != "attention_ms"}
    return out


def run_ours(args, spec):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import tree_speculative_verification_attention_gb300 as tsv

    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    w = DeviceWorkload(spec, tsv, dev, stream, overlap=not args.serial)
    w.capture()
    N, R, L, Rv, Lv, kernels_per_step = w.N, w.R, w.L, w.Rv, w.Lv, w.kernels_per_step

    clocks = ClockRecord(dev)
    clocks.start()
    w.run_steps(max(3, args.warmup))
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    # ---------------------------------------------------------------- timed region
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark()
    t_wall0 = time.time()
    e0.record(stream)
    w.run_steps(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    clocks.mark()
    if world > 1:
        dist.barrier()
    ms_total = whole_job_ms(e0.elapsed_time(e1), world, dev)
    ms_step = ms_total / args.steps
    value = whole_job_value(ms_total, args.steps, N, world)
    timed_clocks = clocks.summary(t_wall0, t_wall1)

    # ---------------------------------------------------------------- the other timing forms
    forms = w.measure(int(min(max(args.steps, 20), 200)))
    attn_ms = forms["attention_ms"]
    if args.no_e2e:
        clocks.stop()
        print(json.dumps({"ms_per_step": ms_step, "attn_launch_ms": attn_ms, "timing": forms}), flush=True)
        return

    roofline, roofline_step = rooflines(spec, w.trees, attn_ms, ms_step, w.walk_rows(), num_sms)
    e2e = measure_e2e(args, spec, w.trees, w.att, w.gi, w.si, tsv.handle(local), tsv, dev, stream, *w.ws_sizes)

    per_workload = None
    if rank == 0 and world == 1 and not args.no_per_workload:
        import workloads as W
        per_workload = {spec.name: workload_summary(spec, w, forms, ms_step, num_sms)}
        per_workload[spec.name]["clocks"] = timed_clocks
        del w
        torch.cuda.empty_cache()
        for name in PER_WORKLOAD:
            if name == spec.name:
                continue
            t0 = time.time()
            ow = DeviceWorkload(W.SPECS[name], tsv, dev, stream, overlap=not args.serial)
            ow.capture()
            ow.run_steps(max(3, args.warmup))
            of = ow.measure(200)
            t1 = time.time()
            per_workload[name] = workload_summary(W.SPECS[name], ow, of, of["graph_mean_ms"], num_sms)
            per_workload[name]["clocks"] = clocks.summary(t0, t1)
            del ow
            torch.cuda.empty_cache()
    clocks.stop()

    how = ("mean over the K timed steps; CUDA graph replay (one graph per %d steps, each step on the next of "
           "%d rotating input copies); verification launches %s" %
           (L, R, "after the attention launch on one stream" if args.serial else
            "after the attention launch on the same stream; greedy in the overlap mode (compact CTAs run "
            "beside the attention CTAs and complete after them)"))
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": spec.dtype, "data": "synthetic",
            "config": config_of(spec),
            "roofline": roofline, "roofline_step": roofline_step,
            "timing": dict(forms, value=how, rotating_copies=R, steps_per_graph=L,
                           verification_copies=Rv, verification_launches_per_graph=Lv),
            "e2e": e2e, "gpu_launches": kernels_per_step * args.steps, "clocks": timed_clocks}
    if per_workload is not None:
        line["per_workload"] = per_workload
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        trees, att, gi, si = workload_inputs(spec)
        line["cpu_baseline"] = oracle_baseline(spec, trees, att, gi, si, args.cpu_seconds,
                                               choose_heads_sample(spec, trees), N)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def graph_kernel_count(g):
    """Kernel nodes in a captured torch CUDA graph."""
    try:
        from cuda.bindings import runtime as cudart
        raw = g.raw_cuda_graph() if hasattr(g, "raw_cuda_graph") else None
        if raw is None:
            return None
        err, _, n = cudart.cudaGraphGetNodes(raw, 0)
        err, nodes, n = cudart.cudaGraphGetNodes(raw, n)
        count = 0
        for nd in nodes:
            err, t = cudart.cudaGraphNodeGetType(nd)
            if t == cudart.cudaGraphNodeType.cudaGraphNodeTypeKernel:
                count += 1
        return count
    except Exception:
        return None


def measure_e2e(args, spec, trees, att, gi, si, h, tsv, dev, stream, ws_attn, ws_g, ws_s):
    """Inputs copied from pinned host memory and results read back every step."""
    import torch
    B, N = spec.B, int(trees.node_offsets[-1])
    host = {"q": att.q, "k": att.k_cache, "v": att.v_cache, "parent": torch.from_numpy(trees.parent),
            "offs": torch.from_numpy(trees.node_offsets), "plen": torch.from_numpy(trees.prefix_len)}
    if gi is not None:
        host.update(logits=torch.from_numpy(gi.logits), gtok=torch.from_numpy(gi.tokens))
    if si is not None:
        host.update(llm=torch.from_numpy(si.llm_logits), ssm=torch.from_numpy(si.ssm_probs),
                    stok=torch.from_numpy(si.tokens), ua=torch.from_numpy(si.u_accept),
                    us=torch.from_numpy(si.u_sample))
    host = {k: t.contiguous().pin_memory() for k, t in host.items()}
    d = {k: torch.empty_like(t, device=dev) for k, t in host.items()}
    anc = torch.empty((N, tsv.TSV_ANC_WORDS), dtype=torch.int32, device=dev)
    status = torch.zeros(B, dtype=torch.int32, device=dev)
    out = torch.empty_like(d["q"])
    wsa = torch.zeros(max(ws_attn, 1), dtype=torch.uint8, device=dev)
    wsg = torch.zeros(max(ws_g, 1), dtype=torch.uint8, device=dev)
    wss = torch.zeros(max(ws_s, 1), dtype=torch.uint8, device=dev)
    res = {k: torch.empty(n, dtype=torch.int32, device=dev) for k, n in
           (("path", N), ("accept_len", B), ("bonus", B), ("n_tried", B), ("status", B))}
    res2 = {k: torch.empty_like(t) for k, t in res.items()}
    out_h = torch.empty_like(out, device="cpu").pin_memory()
    res_h = {k: torch.empty_like(t, device="cpu").pin_memory() for k, t in res.items()}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size()
    if gi is not None:
        d2h += sum(res_h[k].numel() * 4 for k in ("path", "accept_len", "bonus"))
    if si is not None:
        d2h += sum(res_h[k].numel() * 4 for k in ("path", "accept_len", "bonus"))

    # The largest inputs (K and V caches, logits rows) are copied on side
    # streams, so several copy engines share the host link; the main stream
    # waits for them before the kernels that read them.
    big = sorted(host, key=lambda k: -host[k].numel() * host[k].element_size())[:4]
    side = [torch.cuda.Stream(dev) for _ in big]

    def step():
        for k, s2 in zip(big, side):
            s2.wait_stream(stream)
            with torch.cuda.stream(s2):
                d[k].copy_(host[k], non_blocking=True)
        for k in host:
            if k not in big:
                d[k].copy_(host[k], non_blocking=True)
        for s2 in side:
            stream.wait_stream(s2)
        tsv.tree_attention(d["q"], d["k"], d["v"], trees.prefix_len, trees.node_offsets, d["plen"], d["offs"],
                           parent=d["parent"], anc=None, out=out, workspace=wsa, status=status)
        # The verification calls follow attention directly, in overlap mode as
        # in DeviceWorkload.step; the results are read back after all launches.
        kinds = 0 if args.serial else overlap_kinds(tsv, gi is not None)
        with tsv.verify_overlap(kinds, device=dev.index):
            if si is not None:
                tsv.tree_verify_stochastic(d["llm"], d["ssm"], d["stok"], d["parent"], d["offs"], d["ua"], d["us"],
                                           workspace=wss, out=res2, **WARP)
            if gi is not None:
                tsv.tree_verify_greedy(d["logits"], d["gtok"], d["parent"], d["offs"], workspace=wsg, out=res)
        out_h.copy_(out, non_blocking=True)
        if gi is not None:
            for k in ("path", "accept_len", "bonus"):
                res_h[k].copy_(res[k], non_blocking=True)
        if si is not None:
            for k in ("path", "accept_len", "bonus"):
                res_h[k].copy_(res2[k], non_blocking=True)

    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    steps = max(20, min(2000, args.steps // 10))
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"value": N / (ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": ms, "steps": steps,
            "api": "C ABI via the ctypes binding, pinned host buffers, the four largest inputs copied on side streams"}


def run_kv_commit(args, spec):
    """KV commit of the accepted path, timed alone on the workload's shapes: one
    accepted chain per request (the root-to-node chain of a seeded random node).
    Only the rows from prefix_len on are touched, so each of R rotating copies
    holds those rows (prefix 0 on a view of them); R copies exceed 4 x L2."""
    import torch
    import oracle
    import tree_speculative_verification_attention_gb300 as tsv
    import workloads as W

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    rng = np.random.default_rng(1234)
    offs = trees.node_offsets
    B = len(offs) - 1
    path = np.full(int(offs[-1]), -1, np.int32)
    lens = np.zeros(B, np.int32)
    for b in range(B):
        off, n = int(offs[b]), int(offs[b + 1] - offs[b])
        node, chain = int(rng.integers(0, n)), []
        while node >= 0:
            chain.append(node)
            node = int(trees.parent[off + node])
        path[off:off + len(chain)] = chain[::-1]
        lens[b] = len(chain) - 1
    nmax = int(np.diff(offs).max())
    rows_k = torch.stack([att.k_cache[b, int(trees.prefix_len[b]):int(trees.prefix_len[b]) + nmax]
                          for b in range(B)])
    rows_v = torch.stack([att.v_cache[b, int(trees.prefix_len[b]):int(trees.prefix_len[b]) + nmax]
                          for b in range(B)])
    esz = rows_k.element_size()
    per_copy = 2 * rows_k.numel() * esz
    R = max(4, int(math.ceil(4 * 129e6 / per_copy)))
    ks = [rows_k.to(dev) for _ in range(R)]
    vs = [rows_v.to(dev) for _ in range(R)]
    zero = torch.zeros(B, dtype=torch.int32, device=dev)
    d_offs, d_path, d_lens = (torch.as_tensor(x).to(dev) for x in (offs, path, lens))
    out = dict(new_len=torch.empty(B, dtype=torch.int32, device=dev),
               status=torch.empty(B, dtype=torch.int32, device=dev))
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup)):
            tsv.kv_commit(ks[i % R], vs[i % R], zero, d_offs, d_path, d_lens, stream=stream, out=out)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(R):
                tsv.kv_commit(ks[i], vs[i], zero, d_offs, d_path, d_lens, stream=stream, out=out)
    torch.cuda.synchronize()
    reps = max(1, args.steps // R)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (reps * R)
    assert out["status"].cpu().eq(0).all()
    moved = 2 * 2 * int(lens.sum()) * spec.Hkv * spec.D * esz  # K and V, read + write
    peak, _, peak_kind = measured_peaks()
    gbs = moved / (ms * 1e-3) / 1e9
    # The oracle on the host, same rows.
    kc, vc = rows_k.float().numpy(), rows_v.float().numpy()
    t0 = time.perf_counter()
    n_cpu = 0
    while time.perf_counter() - t0 < min(args.cpu_seconds, 2.0) or n_cpu == 0:
        oracle.kv_commit(kc, vc, np.zeros(B, np.int32), offs, path, lens)
        n_cpu += 1
    cpu_s = (time.perf_counter() - t0) / n_cpu
    print(json.dumps({
        "row": "kv_commit", "metric": "committed KV bytes/s (read + write)", "value": gbs, "unit": "GB/s",
        "n_gpus": 1, "steps": reps * R, "warmup": max(3, args.warmup), "ms_per_launch": ms,
        "higher_is_better": True, "dtype": spec.dtype, "data": "synthetic",
        "config": {"workload": spec.name, "B": B, "Hkv": spec.Hkv, "D": spec.D,
                   "accepted_rows": int(lens.sum()), "l2": "rotating %d copies of the touched rows" % R},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "traffic": None, "kernel": "kv_commit_kernel", "peak_kind": peak_kind + " hbm_gbs",
                     "algorithmic_bytes": moved},
        "gpu_launches": reps * R,
        "cpu_baseline": {"value": moved / cpu_s / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "%d full commits of the same rows (numpy, one core)" % n_cpu},
    }), flush=True)


def _attention_parts(q, k, v, trees, max_batch=128):
    """Splits a batch into slices of at most max_batch requests (one launch each)."""
    import workloads as W
    offs = trees.node_offsets
    parts = []
    for b0 in range(0, len(offs) - 1, max_batch):
        b1 = min(len(offs) - 1, b0 + max_batch)
        r0, r1 = int(offs[b0]), int(offs[b1])
        sub = W.Trees(trees.prefix_len[b0:b1], (offs[b0:b1 + 1] - offs[b0]).astype(np.int32),
                      trees.parent[r0:r1], trees.Lcap)
        parts.append((q[r0:r1], k[b0:b1], v[b0:b1], sub))
    return parts


def _time_attention(tsv, q, k, v, trees, dev, stream, reps):
    """Milliseconds per tree attention over the whole batch (one launch per
    slice of at most 128 requests, all replayed from one CUDA graph)."""
    import torch
    h = tsv.handle(dev.index)
    code = 1 if q.dtype == torch.bfloat16 else 0
    calls, outs, stats = [], [], []
    for qp, kp, vp, tp in _attention_parts(q, k, v, trees):
        plen, offs, parent = (torch.as_tensor(x).to(dev) for x in (tp.prefix_len, tp.node_offsets, tp.parent))
        need = tsv.tsv_tree_attention_workspace_size(h, code, len(tp.prefix_len), tp.prefix_len, tp.node_offsets,
                                                     qp.shape[1], kp.shape[2], qp.shape[2], 0, 0)
        ws = torch.zeros(max(16, need), dtype=torch.uint8, device=dev)
        out = torch.empty_like(qp)
        st = torch.empty(len(tp.prefix_len), dtype=torch.int32, device=dev)
        outs.append(out)
        stats.append(st)
        calls.append((qp, kp, vp, tp, plen, offs, parent, ws, out, st))

    def run_all():
        for qp, kp, vp, tp, plen, offs, parent, ws, out, st in calls:
            tsv.tree_attention(qp, kp, vp, tp.prefix_len, tp.node_offsets, plen, offs, parent=parent, out=out,
                               workspace=ws, status=st, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            run_all()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                run_all()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        for _ in range(3):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    assert all(st.cpu().eq(0).all() for st in stats)
    return e0.elapsed_time(e1) / (3 * reps), torch.cat(outs), len(calls)


def run_sequence_baseline(args, spec):
    """Tree attention against a sequence-based verifier doing the same work at
    the kernel level: every root-to-leaf path as its own request (tree width
    1) with its own copy of the prefix, through the same attention entry
    point.  Both caches exceed 4 x L2 or are timed over launches that each
    stream the whole cache."""
    import torch
    import tree_speculative_verification_attention_gb300 as tsv
    import workloads as W

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    trees = W.make_trees(spec)
    att = W.make_attention_inputs(spec, trees)
    att_d = W.AttentionInputs(att.q.to(dev), att.k_cache.to(dev), att.v_cache.to(dev))
    seq = W.sequence_decomposition(trees, att_d)
    stream = torch.cuda.Stream()
    reps = max(1, min(50, args.steps))
    t_tree, out_tree, n_tree = _time_attention(tsv, att_d.q, att_d.k_cache, att_d.v_cache, trees, dev, stream,
                                               reps)
    t_seq, out_seq, n_seq = _time_attention(tsv, seq.inputs.q, seq.inputs.k_cache, seq.inputs.v_cache, seq.trees,
                                            dev, stream, reps)
    diff = (out_seq.float() - out_tree[torch.as_tensor(seq.tree_row, device=dev)].float()).abs().max().item()
    b_tree, b_seq = attention_bytes(spec, trees), attention_bytes(spec, seq.trees)
    peak, _, peak_kind = measured_peaks()
    print(json.dumps({
        "row": "sequence_baseline", "metric": "attention speed-up of the tree over per-sequence attention",
        "value": t_seq / t_tree, "unit": "x", "higher_is_better": True, "n_gpus": 1, "dtype": spec.dtype,
        "data": "synthetic",
        "config": {"workload": spec.name, "tree_nodes": int(trees.node_offsets[-1]),
                   "sequences": int(len(seq.trees.prefix_len)), "sequence_tokens": int(seq.trees.node_offsets[-1])},
        "tree": {"ms": t_tree, "launches": n_tree, "algorithmic_bytes": b_tree,
                 "hbm_gbs": b_tree / (t_tree * 1e-3) / 1e9},
        "sequences": {"ms": t_seq, "launches": n_seq, "algorithmic_bytes": b_seq,
                      "hbm_gbs": b_seq / (t_seq * 1e-3) / 1e9},
        "peak_hbm_gbs": peak, "peak_kind": peak_kind, "max_abs_diff_sequence_vs_tree": diff,
    }), flush=True)


def _graph_ms(fn, stream, reps):
    import torch
    with torch.cuda.stream(stream):
        for _ in range(3):
            fn()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(reps):
                fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        e0.record(stream)
        for _ in range(5):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (5 * reps)


def run_tree_build(args, spec):
    """Token-tree construction: one expansion step (k = 4 children for 8
    frontier nodes per request, the workload's vocabulary) and the merge of
    three speculator trees per request (random-branching, 21 nodes each, as in
    the merge workload), each timed alone from a CUDA graph, the oracle beside."""
    import torch
    import oracle
    import tree_speculative_verification_attention_gb300 as tsv
    import workloads as W

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream()
    B, V, k = spec.B, spec.V, 4
    F = 8 * B
    z = W.normal_f32(spec.wid, 20, (F, V), 2.0)
    zd = torch.as_tensor(z).to(dev)
    tok = torch.empty((F, k), dtype=torch.int32, device=dev)
    ms_expand = _graph_ms(lambda: tsv.tree_expand(zd, k, stream=stream, out=tok), stream, 20)
    assert np.array_equal(tok.cpu().numpy(), oracle.tree_expand(z, k))
    rng = W._rng(spec.wid, 21)
    trees = []
    for b in range(B):
        for _ in range(3):
            par = W.random_tree(rng, 21, 8)
            t = rng.integers(0, 6, 21).astype(np.int32)  # small token range: paths repeat across speculators
            t[0] = 1
            trees.append((par.astype(np.int32), t))
    parent = torch.as_tensor(np.concatenate([t[0] for t in trees])).to(dev)
    tokens = torch.as_tensor(np.concatenate([t[1] for t in trees])).to(dev)
    toffs = torch.as_tensor(np.arange(0, 21 * 3 * B + 1, 21, dtype=np.int32)).to(dev)
    rtrees = torch.as_tensor(np.arange(0, 3 * B + 1, 3, dtype=np.int32)).to(dev)
    res = {}

    def merge():
        res.update(tsv.tree_merge(parent, tokens, toffs, rtrees, stream=stream))
    ms_merge = _graph_ms(merge, stream, 20)
    union = [oracle.tree_merge([t[0] for t in trees[3 * b:3 * b + 3]], [t[1] for t in trees[3 * b:3 * b + 3]])
             for b in range(B)]
    assert res["count"].cpu().tolist() == [len(u[0]) for u in union]
    t0 = time.perf_counter()
    oracle.tree_expand(z[:min(F, 8)], k)
    cpu_expand_ms = (time.perf_counter() - t0) * 1e3 * F / min(F, 8)
    t0 = time.perf_counter()
    for b in range(B):
        oracle.tree_merge([t[0] for t in trees[3 * b:3 * b + 3]], [t[1] for t in trees[3 * b:3 * b + 3]])
    cpu_merge_ms = (time.perf_counter() - t0) * 1e3
    peak, _, peak_kind = measured_peaks()
    gbs = F * V * 4 / (ms_expand * 1e-3) / 1e9
    print(json.dumps({
        "row": "tree_build", "metric": "expansion: frontier logits read per second", "value": gbs, "unit": "GB/s",
        "n_gpus": 1, "data": "synthetic",
        "config": {"workload": spec.name, "frontier_rows": F, "vocab": V, "k": k, "merge_requests": B,
                   "merge_trees_per_request": 3, "merge_nodes_per_tree": 21,
                   "union_nodes_mean": float(np.mean([len(u[0]) for u in union]))},
        "expand": {"ms": ms_expand, "bytes": F * V * 4,
                   "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                                "kernel": "tree_expand_kernel", "peak_kind": peak_kind + " hbm_gbs"}},
        "merge": {"ms": ms_merge, "bound": "latency (one CTA walks each request's input nodes in order)"},
        "cpu_baseline": {"expand_ms": cpu_expand_ms, "merge_ms": cpu_merge_ms, "cores": 1, "kind": "oracle",
                         "sample": "expansion of %d rows scaled to %d; merge of all %d requests" % (min(F, 8), F, B)},
    }), flush=True)


def main():
    args = parse_args()
    import workloads as W
    if args.workload not in W.SPECS:
        raise SystemExit("unknown workload %s (known: %s)" % (args.workload, ", ".join(W.SPECS)))
    spec = W.SPECS[args.workload]
    if args.top_k or args.top_p < 1.0:
        WARP.update(top_k=args.top_k, top_p=args.top_p)
    if args.row == "kv_commit":
        run_kv_commit(args, spec)
    elif args.row == "sequence_baseline":
        run_sequence_baseline(args, spec)
    elif args.row == "tree_build":
        run_tree_build(args, spec)
    elif args.impl == "reference":
        run_reference(args, spec)
    else:
        run_ours(args, spec)


if __name__ == "__main__":
    main()
