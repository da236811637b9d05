#!/usr/bin/env python
"""Throughput of token-tree verification on GB300: tree nodes verified per second.

One step = one pass of the whole hot path over one batch of synthetic input:
tree preparation (ancestor bitsets), one layer of tree attention, and the
verification of the workload (greedy and/or multi-step speculative sampling).
`value` = tree nodes verified / s over the whole job with inputs resident in
HBM; `e2e` = the same metric when every step also copies its inputs from
pinned host memory and reads its results back.

Timing: W untimed warm-up steps, then exactly K steps between CUDA events on
the launching stream, bracketed by barrier + synchronize; each step replays a
CUDA graph of the step on one of R input copies whose total size is at least
4x the L2 cache, so every step reads its inputs from HBM.  Under torchrun each
rank runs an independent replica (replicas only: no data exchange) and the
maximum time over ranks is reported.

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
DEFAULT_WORKLOAD = "llama7b-layer-P1024-n20"


def parse_args():
    p = argparse.ArgumentParser(description=__doc__)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--no-cpu-baseline", action="store_true")
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


def config_of(spec, extra=None):
    cfg = {"workload": spec.name, "B": spec.B, "Hq": spec.Hq, "Hkv": spec.Hkv, "D": spec.D,
           "prefix": list(spec.prefix) if isinstance(spec.prefix, tuple) else spec.prefix,
           "nodes_per_request": spec.nodes, "vocab": spec.V,
           "verify": "+".join(v for v, on in (("greedy", spec.greedy), ("stochastic", spec.stochastic)) if on),
           "tree": spec.tree}
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


def verify_bytes(spec, trees, n_rejected_rows=0):
    """Greedy: every logits row once.  Stochastic: every LLM row once plus the
    full proposal row of each rejected child (count from the oracle)."""
    N = int(trees.node_offsets[-1])
    b = 0
    if spec.greedy:
        b += N * spec.V * 4
    if spec.stochastic:
        b += (N + n_rejected_rows) * spec.V * 4
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


def measured_peaks():
    """(HBM GB/s, dense bf16 TFLOP/s for a kernel timed alone, which)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


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
            "config": config_of(spec, {"reference": "CPU fp64 oracle (the pages ship no code)"}),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "per step: " + sample, "single_core": base["single_core"],
                             "nproc": base["nproc"], "cpu_model": base["cpu_model"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU


def run_ours(args, spec):
    import torch
    import torch.distributed as dist

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import tree_speculative_verification_attention_gb300 as tsv

    trees, att, gi, si = workload_inputs(spec)
    B, N = spec.B, int(trees.node_offsets[-1])
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)

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
    per_copy = sum(t.numel() * t.element_size() for t in base.values())
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = int(min(64, max(1, math.ceil(4 * l2 / per_copy))))
    copies = [base] + [{k: t.clone() for k, t in base.items()} for _ in range(R - 1)]

    h = tsv.handle(local)
    ws_attn = tsv.tsv_tree_attention_workspace_size(h, tsv.TSV_BF16 if spec.dtype == "bf16" else tsv.TSV_F32,
                                                    B, trees.prefix_len, trees.node_offsets, spec.Hq,
                                                    spec.Hkv, spec.D, False)
    ws_g = tsv.tsv_tree_verify_greedy_workspace_size(h, B, N, spec.V)
    ws_s = tsv.tsv_tree_verify_stochastic_workspace_size(h, B, N, spec.V)
    ws_bytes = max(ws_attn, 1) + max(ws_g, 1) + max(ws_s, 1) + 3 * 256

    def make_state(c):
        st = {"anc": torch.empty((N, tsv.TSV_ANC_WORDS), dtype=torch.int32, device=dev),
              "depth": torch.empty(N, dtype=torch.int32, device=dev),
              "status": torch.zeros(B, dtype=torch.int32, device=dev),
              "out": torch.empty_like(c["q"]),
              "ws": torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)}
        st["ws_attn"] = st["ws"][:max(ws_attn, 1)]
        off = (max(ws_attn, 1) + 255) // 256 * 256
        st["ws_g"] = st["ws"][off:off + max(ws_g, 1)]
        off += (max(ws_g, 1) + 255) // 256 * 256
        st["ws_s"] = st["ws"][off:off + max(ws_s, 1)]
        mk = lambda: {k: torch.empty(n, dtype=torch.int32, device=dev) for k, n in
                      (("path", N), ("accept_len", B), ("bonus", B), ("n_tried", B), ("status", B))}
        st["g"], st["s"] = mk(), mk()
        return st

    def attention(c, st):
        # The kernel builds the ancestor masks from parent[] itself (and
        # validates the tree), so tree preparation runs inside this launch.
        tsv.tree_attention(c["q"], c["k"], c["v"], trees.prefix_len, trees.node_offsets, c["plen"],
                           c["offs"], parent=c["parent"], anc=None, out=st["out"],
                           workspace=st["ws_attn"], status=st["status"])

    def step(c, st):
        attention(c, st)
        if gi is not None:
            tsv.tree_verify_greedy(c["logits"], c["gtok"], c["parent"], c["offs"], workspace=st["ws_g"],
                                   out=st["g"])
        if si is not None:
            tsv.tree_verify_stochastic(c["llm"], c["ssm"], c["stok"], c["parent"], c["offs"], c["ua"],
                                       c["us"], workspace=st["ws_s"], out=st["s"], **WARP)

    states = [make_state(c) for c in copies]
    # Eager run once (also checks statuses), then capture one graph per input copy.
    for c, st in zip(copies, states):
        step(c, st)
    torch.cuda.synchronize()
    assert (states[0]["status"].cpu() == 0).all()
    # One graph holds one step on every input copy (R steps), so the host
    # replays one graph per R steps and stays ahead of the GPU.
    g_steps = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_steps, stream=stream):
        for c, st in zip(copies, states):
            step(c, st)
    g_one = []
    for c, st in zip(copies, states):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(c, st)
        g_one.append(g)
    g_attn = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_attn, stream=stream):
        for c, st in zip(copies, states):
            attention(c, st)
    torch.cuda.synchronize()
    # Kernels per step: one attention launch (masks built inside, splits merged
    # inside; the fp32 CUDA-core path first prepares the ancestor bitsets in a
    # launch of its own), one for greedy verification, one for stochastic
    # verification; checked against the captured graph when torch exposes it.
    attn_kernels = 1 if spec.dtype == "bf16" else 2
    kernels_per_step = attn_kernels + (1 if gi is not None else 0) + (1 if si is not None else 0)
    counted = graph_kernel_count(g_one[0])
    if counted is not None:
        assert counted == kernels_per_step, (counted, kernels_per_step)

    sampler = ClockSampler(local)
    sampler.start()
    def run_steps(k):
        for _ in range(k // R):
            g_steps.replay()
        for i in range(k % R):
            g_one[i].replay()

    run_steps(args.warmup)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    # ---------------------------------------------------------------- timed region
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record(stream)
    run_steps(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    ms_total = whole_job_ms(e0.elapsed_time(e1), world, dev)
    ms_step = ms_total / args.steps
    value = whole_job_value(ms_total, args.steps, N, world)

    # ---------------------------------------------------------------- attention kernel, per launch
    # Average launch duration of the attention call inside a graph of R
    # back-to-back launches (one per input copy), events on the launching stream.
    reps = max(1, min(2000, args.steps) // R)
    g_attn.replay()
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(reps):
        g_attn.replay()
    a1.record(stream)
    torch.cuda.synchronize()
    attn_ms = a0.elapsed_time(a1) / (reps * R)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    if args.no_e2e:
        print(json.dumps({"ms_per_step": ms_step, "attn_launch_ms": attn_ms}), flush=True)
        return

    # ---------------------------------------------------------------- end to end
    e2e = measure_e2e(args, spec, trees, att, gi, si, h, tsv, dev, stream, ws_attn, ws_g, ws_s)

    # ---------------------------------------------------------------- roofline
    peak, peak_tf, peak_kind = measured_peaks()
    abytes = attention_bytes(spec, trees)
    aflops = attention_flops(spec, trees)
    achieved = abytes / (attn_ms * 1e-3) / 1e9
    keys_kernel = all(int(n) * (spec.Hq // spec.Hkv) <= 64 for n in np.diff(trees.node_offsets)) and \
        64 % (spec.Hq // spec.Hkv) == 0
    G = spec.Hq // spec.Hkv
    tile_pairs = any(int(n) * G > 128 for n in np.diff(trees.node_offsets))  # some request has 2+ row tiles
    kernel_name = ("tree_attn_simt_kernel" if spec.dtype != "bf16" else
                   "tree_attn_keys_kernel" if keys_kernel else
                   "tree_attn_tc_kernel" if tile_pairs else "tree_attn_tc1_kernel")
    traffic = recorded_traffic(spec.name, kernel_name)
    # The bound is whichever of bytes / bandwidth and FLOPs / tensor peak takes longer.
    tensor_bound = spec.dtype == "bf16" and aflops / (peak_tf * 1e12) > abytes / (peak * 1e9)
    if tensor_bound:
        tf = aflops / (attn_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": tf, "peak": peak_tf, "unit": "TFLOP/s",
                    "frac": tf / peak_tf, "peak_kind": peak_kind + " bf16_tflops (burst)"}
    else:
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "peak_kind": peak_kind + " hbm_gbs"}
    roofline.update({"traffic": traffic, "kernel": kernel_name, "launch_ms": attn_ms,
                     "algorithmic_bytes": abytes, "algorithmic_flops": aflops,
                     "hbm_gbs": achieved, "hbm_frac": achieved / peak})
    step_bytes = abytes + verify_bytes(spec, trees)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": spec.dtype, "data": "synthetic",
            "config": config_of(spec, {"l2": "rotating %d input copies (%.0f MB > 4x L2)" % (R, R * per_copy / 1e6),
                                       "graph": "one CUDA graph per step", "parallelism": "replicas"}),
            "roofline": roofline,
            "step_hbm_gbs": step_bytes / (ms_step * 1e-3) / 1e9,
            "step_roofline_frac": step_bytes / (ms_step * 1e-3) / 1e9 / peak,
            "e2e": e2e, "gpu_launches": kernels_per_step * args.steps, "clocks": clocks}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
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
        out_h.copy_(out, non_blocking=True)
        if gi is not None:
            tsv.tree_verify_greedy(d["logits"], d["gtok"], d["parent"], d["offs"], workspace=wsg, out=res)
            for k in ("path", "accept_len", "bonus"):
                res_h[k].copy_(res[k], non_blocking=True)
        if si is not None:
            tsv.tree_verify_stochastic(d["llm"], d["ssm"], d["stok"], d["parent"], d["offs"], d["ua"], d["us"],
                                       workspace=wss, out=res2, **WARP)
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
