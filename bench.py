"""Benchmark of the paged decode attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

The default workload is the largest single-GPU decode configuration
(gqa6_d256_vllm_decode: 128 sequences, GQA-6, D = 256, vLLM layout); the same
run measures the other configurations (Llama-3-8B-shaped, long-context, FP8,
4-token and the MLA prefill) and reports them under "per_config", the
Llama-3-8B-shaped one with what the device plan costs there ("device_plan":
host plan, planning in phase 1, a reused plan at exact and capacity bounds).

One step = one full decode step of the workload (phase 1 + cross-split
combine) on synthetic inputs already resident in HBM.  Between timed steps a
256 MiB buffer is written to flush the 129 MB L2 and a second 256 MiB buffer is
read, so that the write's dirty lines reach HBM before the step instead of
during it; each step is timed with CUDA events on the launching stream, the K
step times are summed, and the maximum over ranks is taken.  The metric is
KV-cache bytes per second: live tokens x KV heads x head_dim x (K and V) x 2
bytes per step, divided by the step time.

N > 1 runs independent replicas (one process per GPU, launched by torchrun):
the decode step has no exchange between GPUs, so there is no collective on the
data path; the only collectives are the timing barrier and the max-over-ranks.

--impl reference times the fp64 CPU oracle on the host cores (bounded samples
of the same workload) and prints the same JSON line with "impl": "reference".
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
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention: KV-cache GB/s and % of GB300 HBM peak; µs/step"
FLUSH_BYTES = 256 << 20
L2_NOTE = "cold between steps: 256 MiB written, then another 256 MiB read (the write's dirty lines reach HBM first)"


class ColdL2:
    """Leaves the L2 cold and clean before a timed step.  Writing a buffer twice the
    L2's size evicts every line of the step's inputs but leaves the L2 full of that
    buffer's dirty lines, whose write-back would otherwise run during the step and
    take HBM bandwidth from it; reading a second buffer of the same size writes
    them back first."""

    def __init__(self, torch, device):
        self.torch = torch
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.ones(FLUSH_BYTES, dtype=torch.uint8, device=device)

    def __call__(self):
        self.w.zero_()
        self.torch.amax(self.r)


# committed ncu summaries per workload (their traffic is used only while the sources match)
PROFILE_SUMMARIES = {
    "llama3_8b_decode": os.path.join(ROOT, "profiles", "decode_phase1_llama3_8b_decode.md"),
    "llama3_8b_spec_decode_q4": os.path.join(ROOT, "profiles", "decode_phase1_llama3_8b_spec_decode_q4.md"),
    "llama3_8b_decode_fp8": os.path.join(ROOT, "profiles", "decode_phase1_llama3_8b_decode_fp8.md"),
    "long_context_decode": os.path.join(ROOT, "profiles", "decode_phase1_long_context_decode.md"),
    "gqa6_d256_vllm_decode": os.path.join(ROOT, "profiles", "decode_phase1_gqa6_d256_vllm_decode.md"),
}
MLA_PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "mla_prefill_kernel_mla_prefill_h16.md")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e nominal (context for the measured copy peak)


def kernel_source_hash(files=None) -> str:
    """sha256 over CUDA sources (the named csrc files, else all of them); a
    profile's counters are valid only for the sources they were taken on."""
    csrc = os.path.join(ROOT, "paged_kv_gqa_table_gb300", "csrc")
    if not files:
        files = sorted(f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")))
    h = hashlib.sha256()
    for f in files:
        h.update(f.encode())
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(summary):
    """Per-launch DRAM bytes of the profiled kernel from a committed ncu
    summary, if it was taken on the current kernel sources (the summary's
    `source_files`, else every csrc file); else None."""
    if not summary or not os.path.exists(summary):
        return None
    text = open(summary).read()
    m_hash = re.search(r"source_sha256:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    m_files = re.search(r"source_files:\s*(.+)", text)
    files = m_files.group(1).split() if m_files else None
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_source_hash(files):
        return None
    return int(m_bytes.group(1))


def profiled_field(summary, key):
    """A number `key: value` from a committed ncu summary taken on the current
    kernel sources (as profiled_traffic), else None."""
    if not summary or not os.path.exists(summary) or profiled_traffic(summary) is None:
        return None
    m = re.search(r"^%s:\s*([0-9.]+)" % re.escape(key), open(summary).read(), flags=re.M)
    return float(m.group(1)) if m else None


# ----------------------------------------------------------------- clocks ----

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the GPU works."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.proc = None
        self.lines = []
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "50"]
        if uuid:
            cmd[1:1] = ["-i", uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        # nvidia-smi's start-up (driver queries) can hold up kernel launches for
        # milliseconds: let it reach its first sample before anything is timed.
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < 10.0 and self.proc.poll() is None:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------- distributed ----

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ------------------------------------------------------------ CPU oracle ----

def oracle_decode_timed(case, seqs, threads):
    """Runs the fp64 oracle over the given sequences on `threads` host threads; returns seconds."""
    import oracle
    out = np.empty(case["q"].shape)
    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda b: oracle.decode(case, b, b + 1, out=out), seqs))
    return time.perf_counter() - t0


def kv_bytes_page_rounded(case):
    """KV bytes of whole pages: every live token's page read in full (the last page's unused slots too)."""
    e = 1 if tensors_fp8(case) else 2
    bs = case["block_size"]
    pages = (case["context_lens"].astype(np.int64) + bs - 1) // bs
    return int(pages.sum()) * bs * case["Hkv"] * case["D"] * 2 * e


def seq_kv_bytes(case, seqs):
    """KV bytes of the given sequences (K and V, the cache's element size)."""
    e = 1 if tensors_fp8(case) else 2
    return int(np.sum(case["context_lens"][list(seqs)], dtype=np.int64)) * case["Hkv"] * case["D"] * 2 * e


def cpu_baseline(case, budget_s: float = 15.0):
    """The oracle as it stands on all host cores over a bounded sample of the workload, and
    on one core over a smaller sample."""
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    order = np.random.default_rng(1).permutation(case["B"])
    # grow the sample until it takes about a second, then extrapolate within the budget
    n = min(len(order), threads)
    while True:
        secs = oracle_decode_timed(case, order[:n], threads)
        if n == len(order) or secs > 1.0:
            break
        n = min(len(order), n * 2)
    if secs < budget_s / 4 and n < len(order):
        m = min(len(order), int(n * budget_s / 4 / max(secs, 1e-3)))
        secs = oracle_decode_timed(case, order[:m], threads)
        n = m
    gbs = seq_kv_bytes(case, order[:n]) / secs / 1e9
    # one core: sequences in the same order until ~2 s
    m1, secs1 = 0, 0.0
    while m1 < len(order) and secs1 < 2.0:
        secs1 += oracle_decode_timed(case, [order[m1]], 1)
        m1 += 1
    return {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": "%d of %d sequences (all heads), one pass, %.1f s" % (n, case["B"], secs),
            "single_core": {"value": seq_kv_bytes(case, order[:m1]) / secs1 / 1e9, "unit": "GB/s",
                            "sample": "%d sequences, %.1f s" % (m1, secs1)}}


# ----------------------------------------------------------------- arms ----

def run_reference(args):
    """--impl reference: the CPU oracle timed on bounded samples, same metric and workload."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from paged_kv_gqa_table_gb300 import synth
    import oracle
    oracle.build()
    case = synth.decode_case(seed=0, **synth.WORKLOADS[args.workload])
    threads = os.cpu_count() or 1
    order = np.random.default_rng(2).permutation(case["B"])
    # step size: as many sequences as keep K + W steps within ~120 s
    probe = order[:min(len(order), threads)]
    t_probe = oracle_decode_timed(case, probe, threads)
    per_seq = t_probe / len(probe)
    per_step = max(1, min(len(order), int(120.0 / (args.steps + args.warmup) / max(per_seq, 1e-6))))
    cursor = 0

    def step():
        nonlocal cursor
        seqs = [order[(cursor + i) % len(order)] for i in range(per_step)]
        cursor += per_step
        return oracle_decode_timed(case, seqs, threads), seq_kv_bytes(case, seqs)

    for _ in range(args.warmup):
        step()
    tot_t, tot_b = 0.0, 0
    for _ in range(args.steps):
        t, b = step()
        tot_t += t
        tot_b += b
    value = tot_b / tot_t / 1e9
    sample = "%d of %d sequences (all heads) per step" % (per_step, case["B"])
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(case, args.workload, flushed=False, accumulate="fp64"),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def dtype_label(case):
    q = {0: "fp16", 1: "bf16"}[case["dtype"]]
    if tensors_fp8(case):
        return "%s q/out, fp8-e4m3 KV (k_scale %g, v_scale %g)" % (q, case["k_scale"], case["v_scale"])
    return q


def tensors_fp8(case):
    from paged_kv_gqa_table_gb300 import synth
    return case.get("kv_dtype", case["dtype"]) == synth.FP8_E4M3


def workload_config(case, name, flushed=True, accumulate="fp32"):
    from paged_kv_gqa_table_gb300 import synth
    ctx = case["context_lens"]
    q_len = int(case.get("q_len", 1))
    return {"workload": "%s: B=%d q_len=%d Hq=%d Hkv=%d D=%d block_size=%d %s %s layout, context_lens %d..%d (sum %d)" % (
        name, case["B"], q_len, case["Hq"], case["Hkv"], case["D"], case["block_size"],
        dtype_label(case), {0: "NHD", 1: "vLLM x-packed"}[case["layout"]],
        int(ctx.min()), int(ctx.max()), int(ctx.sum())),
        "seed": 0, "kv_bytes_per_step": synth.kv_bytes(case), "query_tokens_per_step": case["B"] * q_len,
        "kv_bytes_per_step_page_rounded": kv_bytes_page_rounded(case),
        "l2": L2_NOTE if flushed else "n/a (CPU)",
        "accumulate": accumulate}


def measure_decode(name, device, steps, warmup, world=1, rank=0, e2e_leg=True, cpu_leg=True, cpu_budget_s=15.0,
                   sample_clocks=False):
    """One decode workload: `warmup` untimed steps, then `steps` timed steps (cold L2
    before each), then the same steps again with events around the phase-1 kernel
    (the roofline's launch duration).  Returns (fields of the JSON line, case)."""
    import torch
    from paged_kv_gqa_table_gb300 import binding as B
    from paged_kv_gqa_table_gb300 import synth, tensors

    case = synth.decode_case(seed=0, **synth.WORKLOADS[name])
    kvb = synth.kv_bytes(case)
    dev = tensors.upload_decode_case(case, device)
    desc = tensors.decode_desc(case)
    ns, P = B.pkv_plan_splits(desc)
    out = torch.empty(case["q"].shape, dtype=tensors.TORCH_DTYPE[case["dtype"]], device=device)
    ws = tensors.workspace_for(desc, device=device)
    flush = ColdL2(torch, device)
    stream = torch.cuda.current_stream(device)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    p_start, p_stop = [ev() for _ in range(steps)], [ev() for _ in range(steps)]
    s_start, s_stop = [ev() for _ in range(steps)], [ev() for _ in range(steps)]
    for e in p_start + p_stop:
        e.record(stream)       # materialise the CUDA events before the library records them
    torch.cuda.synchronize(device)

    def step(opts=None):
        B.pkv_paged_decode_attention(desc, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"],
                                     dev["context_lens"], case["scale"], out, ws, opts=opts, stream=stream)

    sampler = None
    if sample_clocks:
        uuid = None
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            pass
        sampler = ClockSampler(uuid)
    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize(device)
    barrier(world, device)
    torch.cuda.synchronize(device)
    wall0 = time.perf_counter()
    for i in range(steps):
        flush()
        s_start[i].record(stream)
        step()
        s_stop[i].record(stream)
    torch.cuda.synchronize(device)
    barrier(world, device)
    torch.cuda.synchronize(device)
    wall = time.perf_counter() - wall0
    # Phase 1 alone, for the roofline: the same steps again with events the
    # library records around the phase-1 kernel (an event between the two
    # kernels stops the combine from overlapping phase 1, so these steps are
    # not the timed ones).
    for i in range(steps):
        flush()
        step(B.make_opts(event_start=p_start[i], event_stop=p_stop[i]))
    torch.cuda.synchronize(device)
    clocks = sampler.stop() if sampler else None
    step_ms = [a.elapsed_time(b) for a, b in zip(s_start, s_stop)]
    p1_ms = [a.elapsed_time(b) for a, b in zip(p_start, p_stop)]
    t_total = sum(step_ms) * 1e-3
    t_max = max_over_ranks(t_total, world, device)
    value = world * kvb * steps / t_max / 1e9

    # end to end: pinned host inputs -> device, the C-ABI call, result -> pinned host
    e2e = None
    if e2e_leg:
        host = {k: v.cpu().pin_memory() for k, v in dev.items()}
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out.numel() * out.element_size()
        n_e2e = max(3, min(steps, 30))
        for i in range(n_e2e + 2):
            if i == 2:
                torch.cuda.synchronize(device)
                barrier(world, device)
                e0 = ev()
                e0.record(stream)
            for k in dev:
                dev[k].copy_(host[k], non_blocking=True)
            step()
            out_h.copy_(out, non_blocking=True)
        e1 = ev()
        e1.record(stream)
        torch.cuda.synchronize(device)
        t_e2e = max_over_ranks(e0.elapsed_time(e1) * 1e-3, world, device)
        e2e = {"value": world * kvb * n_e2e / t_e2e / 1e9, "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": n_e2e, "copies_declared": True}

    peak, peak_kind = measured_peaks()
    p1_avg = float(np.mean(p1_ms)) * 1e-3
    achieved = kvb / p1_avg / 1e9
    summary = PROFILE_SUMMARIES.get(name)
    fields = {
        "value": value, "unit": "GB/s", "ms_per_step": t_max / steps * 1e3, "us_per_step": t_max / steps * 1e6,
        "steps": steps, "warmup": warmup, "dtype": dtype_label(case),
        "config": dict(workload_config(case, name), partition_tokens=P, num_splits=ns),
        "hbm_frac_of_measured_peak": value / peak, "hbm_frac_of_nominal_peak": value / NOMINAL_HBM_GBS,
        "gpu_launches": steps * (1 + (1 if ns > 1 else 0)),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "traffic": profiled_traffic(summary),
                     "ncu_dram_throughput_pct": profiled_field(summary, "dram_throughput_pct"),
                     "kernel": "decode_phase1_kernel", "peak_source": peak_kind,
                     "algorithmic_bytes_per_launch": kvb, "avg_launch_us": p1_avg * 1e6},
        "clocks": clocks, "e2e": e2e, "wall_s_timed_region": wall,
    }
    if cpu_leg and world == 1 and rank == 0:
        fields["cpu_baseline"] = cpu_baseline(case, budget_s=cpu_budget_s)
    return fields, case


DEVICE_PLAN_STEPS = 100


def measure_device_plan(name, device, steps, warmup):
    """What the device plan (PKV_DECODE_DEVICE_PLAN) costs on one decode workload: mean µs per
    step, cold L2 before each, with the host plan, with phase 1 planning from the device's
    context lengths, and with the plan an earlier call left in the workspace reused
    (PKV_DECODE_PLAN_READY, as the later layers of one decode step do) -- at exact bounds and at
    capacity bounds (every context may fill its block-table row, as in a captured graph)."""
    import torch
    from paged_kv_gqa_table_gb300 import binding as B
    from paged_kv_gqa_table_gb300 import synth, tensors

    case = synth.decode_case(seed=0, **synth.WORKLOADS[name])
    dev = tensors.upload_decode_case(case, device)
    out = torch.empty(case["q"].shape, dtype=tensors.TORCH_DTYPE[case["dtype"]], device=device)
    flush = ColdL2(torch, device)
    stream = torch.cuda.current_stream(device)
    legs = (("host_plan", False, None), ("device_plan", False, B.make_opts(device_plan=True)),
            ("plan_reused", False, B.make_opts(plan_ready=True)),
            ("plan_reused_capacity_bounds", True, B.make_opts(plan_ready=True)))
    res = {}
    for label, capacity, opts in legs:
        desc = tensors.decode_desc(case)
        if capacity:
            desc.max_context_len = desc.max_blocks_per_seq * desc.block_size
            desc.sum_context_len = desc.B * desc.max_context_len
        ws = tensors.workspace_for(desc, opts, device=device)

        def call(o):
            B.pkv_paged_decode_attention(desc, dev["q"], dev["k_cache"], dev["v_cache"], dev["block_table"],
                                         dev["context_lens"], case["scale"], out, ws, opts=o, stream=stream)
        if opts is not None and opts.flags & B.PKV_DECODE_PLAN_READY:
            call(B.make_opts(device_plan=True))   # the earlier layer, which plans
        for _ in range(warmup):
            flush()
            call(opts)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in evs:
            flush()
            a.record(stream)
            call(opts)
            b.record(stream)
        torch.cuda.synchronize(device)
        res[label + "_us"] = float(np.mean([a.elapsed_time(b) for a, b in evs])) * 1e3
        err = int(ws[:4].view(torch.int32).item())
        if err:   # reported, not raised: the rest of the line still prints
            res[label + "_device_error_word"] = err
    res["device_plan_overhead_us"] = res["device_plan_us"] - res["host_plan_us"]
    res["plan_reused_overhead_us"] = res["plan_reused_us"] - res["host_plan_us"]
    res["plan_reused_capacity_bounds_overhead_us"] = res["plan_reused_capacity_bounds_us"] - res["host_plan_us"]
    res["steps_per_leg"] = steps
    return res


# The headline workload is the largest single-GPU configuration; the others are
# measured in the same run and reported under "per_config".
HEADLINE = "gqa6_d256_vllm_decode"
DEVICE_PLAN_WORKLOAD = "llama3_8b_decode"
PER_CONFIG = ["llama3_8b_decode", "long_context_decode", "llama3_8b_decode_fp8", "llama3_8b_spec_decode_q4",
              "mla_prefill_h16"]
PER_CONFIG_STEPS = 300


def run_gpu(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from paged_kv_gqa_table_gb300 import binding as B
    B.load()
    fields, case = measure_decode(args.workload, device, args.steps, args.warmup, world, rank,
                                  e2e_leg=not args.skip_e2e, cpu_leg=not args.skip_cpu_baseline,
                                  sample_clocks=rank == 0)
    per_config = None
    if world == 1 and not args.skip_per_config and args.workload == HEADLINE:
        per_config = {}
        steps = min(args.steps, PER_CONFIG_STEPS)
        for name in PER_CONFIG:
            if name == "mla_prefill_h16":
                f = measure_mla(name, device, steps, args.warmup, e2e_leg=False,
                                cpu_leg=not args.skip_cpu_baseline, cpu_budget_s=8.0)
            else:
                f, _ = measure_decode(name, device, steps, args.warmup, e2e_leg=False,
                                      cpu_leg=not args.skip_cpu_baseline, cpu_budget_s=8.0)
            per_config[name] = {k: f[k] for k in ("value", "unit", "us_per_step", "steps", "dtype", "roofline",
                                                  "cpu_baseline", "gpu_launches", "config") if k in f}
            if "hbm_frac_of_measured_peak" in f:
                per_config[name]["hbm_frac_of_measured_peak"] = f["hbm_frac_of_measured_peak"]
            if name == DEVICE_PLAN_WORKLOAD:
                per_config[name]["device_plan"] = measure_device_plan(name, device, min(steps, DEVICE_PLAN_STEPS),
                                                                      args.warmup)
    if rank == 0:
        line = {"metric": METRIC, "n_gpus": world, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None,
                "data": "synthetic (seeded N(0,1) K/V/q, uniform context lengths, random page permutation)"}
        line.update(fields)
        line["config"] = dict(fields["config"], parallelism="replicas" if world > 1 else "1 GPU")
        if per_config is not None:
            line["per_config"] = per_config
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


MLA_METRIC = "MLA paged causal prefill: TFLOP/s (algorithmic) and µs/step"


def mla_pairs(case):
    """(query token, visible key) pairs of an MLA prefill batch (bottom-right causal)."""
    qo, kvp = case["qo_indptr"].astype(np.int64), case["kv_indptr"].astype(np.int64)
    total = 0
    for b in range(case["batch"]):
        q_len, kv_len = int(qo[b + 1] - qo[b]), int(kvp[b + 1] - kvp[b])
        if kv_len == 0:
            continue
        prefix = kv_len - q_len
        total += q_len * (prefix + 1) + q_len * (q_len - 1) // 2
    return total


def mla_flops(case):
    """Algorithmic flops: per pair and head, 2 x (576 + 512) for Q.K^T and P.V."""
    return mla_pairs(case) * case["H"] * 2 * (case["Dc"] + case["Dr"] + case["Dc"])


def mla_workload_config(case, name):
    qo, kvp = case["qo_indptr"], case["kv_indptr"]
    return {"workload": "%s: %d sequences, q_len %d..%d, kv_len %d..%d (total_q %d, %d cached rows), "
                        "16 heads, ckv 512 + kpe 64, bf16, page size 1" % (
                            name, case["batch"], int(np.diff(qo).min()), int(np.diff(qo).max()),
                            int(np.diff(kvp).min()), int(np.diff(kvp).max()), case["total_q"], int(kvp[-1])),
            "seed": 0, "flops_per_step": int(mla_flops(case)), "pairs": int(mla_pairs(case)),
            "sm_scale": case["sm_scale"], "l2": L2_NOTE, "accumulate": "fp32",
            "s_per_row_tile": "once (max_kv_len given: the second output half replays the first's softmax weights)"}


def mla_oracle_timed(case, tokens, threads):
    """The oracle on the given query tokens (all heads) on `threads` host threads:
    (algorithmic flops of those tokens, seconds)."""
    import oracle
    out = np.empty((case["total_q"], case["H"], case["Dc"]))
    lse = np.empty((case["total_q"], case["H"]))
    t0 = time.perf_counter()
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda t: oracle.mla(case, int(t), int(t) + 1, out=out, lse=lse), tokens))
    secs = time.perf_counter() - t0
    qo, kvp = case["qo_indptr"], case["kv_indptr"]
    b_of = np.searchsorted(qo, tokens, side="right") - 1
    pairs = 0
    for t, b in zip(tokens, b_of):
        q_len, kv_len = qo[b + 1] - qo[b], kvp[b + 1] - kvp[b]
        pairs += (kv_len - q_len) + (t - qo[b]) + 1
    return pairs * case["H"] * 2 * (2 * case["Dc"] + case["Dr"]), secs


def mla_cpu_baseline(case, budget_s: float = 15.0):
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    T = case["total_q"]
    order = np.random.default_rng(3).permutation(T)
    n = min(T, threads * 2)
    flops, secs = mla_oracle_timed(case, order[:n], threads)
    m = min(T, max(n, int(n * budget_s / 4 / max(secs, 1e-3))))
    if m > n:
        n = m
        flops, secs = mla_oracle_timed(case, order[:n], threads)
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": "%d of %d query tokens (all heads), %.1f s" % (n, T, secs)}


def run_mla_reference(args):
    """--impl reference on the MLA workload: the CPU oracle timed on bounded samples of query
    tokens (a different sample each step), same metric and workload as run_mla."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    from paged_kv_gqa_table_gb300 import synth
    import oracle
    oracle.build()
    case = synth.mla_case(seed=0, **synth.MLA_WORKLOADS[args.workload])
    threads = os.cpu_count() or 1
    T = case["total_q"]
    order = np.random.default_rng(3).permutation(T)
    # step size: as many tokens as keep K + W steps within ~60 s
    n0 = min(T, threads * 2)
    _, secs0 = mla_oracle_timed(case, order[:n0], threads)
    per_step = int(min(T, max(n0, n0 * 60.0 / (args.steps + args.warmup) / max(secs0, 1e-3))))
    cursor = 0

    def step():
        nonlocal cursor
        toks = order[np.arange(cursor, cursor + per_step) % T]
        cursor += per_step
        return mla_oracle_timed(case, toks, threads)

    for _ in range(args.warmup):
        step()
    tot_f, tot_t = 0, 0.0
    for _ in range(args.steps):
        f, t = step()
        tot_f += f
        tot_t += t
    value = tot_f / tot_t / 1e12
    sample = "%d of %d query tokens (all heads) per step" % (per_step, T)
    line = {"impl": "reference", "metric": MLA_METRIC, "value": value,
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": dict(mla_workload_config(case, args.workload), l2="n/a (CPU)", accumulate="fp64"),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def measure_mla(name, device, steps, warmup, e2e_leg=True, cpu_leg=True, cpu_budget_s=15.0, sample_clocks=False):
    """The MLA prefill workload (one call per step), same timing rules as the decode arm."""
    import torch
    from paged_kv_gqa_table_gb300 import synth, tensors
    case = synth.mla_case(seed=0, **synth.MLA_WORKLOADS[name])
    flops = mla_flops(case)
    dev = tensors.upload_mla_case(case, device)
    T, H, Dc = case["total_q"], case["H"], case["Dc"]
    out = torch.empty((T, H, Dc), dtype=torch.bfloat16, device=device)
    lse = torch.empty((T, H), dtype=torch.float32, device=device)
    desc = tensors.mla_desc(case)
    ws = tensors.mla_workspace_for(desc, device=device)
    flush = ColdL2(torch, device)
    stream = torch.cuda.current_stream(device)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    starts, stops = [ev() for _ in range(steps)], [ev() for _ in range(steps)]
    step = lambda: tensors.mla_paged_prefill(case, dev, out, lse, workspace=ws, stream=stream, desc=desc)
    sampler = None
    if sample_clocks:
        uuid = None
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            pass
        sampler = ClockSampler(uuid)
    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize(device)
    wall0 = time.perf_counter()
    for i in range(steps):
        flush()
        starts[i].record(stream)
        step()
        stops[i].record(stream)
    torch.cuda.synchronize(device)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop() if sampler else None
    t = sum(a.elapsed_time(b) for a, b in zip(starts, stops)) * 1e-3
    e2e = None
    if e2e_leg:
        host = {k: v.cpu().pin_memory() for k, v in dev.items()}
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        h2d = sum(x.numel() * x.element_size() for x in host.values())
        d2h = out.numel() * out.element_size() + lse.numel() * lse.element_size()
        n_e2e = max(3, min(steps, 30))
        for i in range(n_e2e + 2):
            if i == 2:
                torch.cuda.synchronize(device)
                e0 = ev()
                e0.record(stream)
            for k in dev:
                dev[k].copy_(host[k], non_blocking=True)
            step()
            out_h.copy_(out, non_blocking=True)
            lse_h.copy_(lse, non_blocking=True)
        e1 = ev()
        e1.record(stream)
        torch.cuda.synchronize(device)
        t_e2e = e0.elapsed_time(e1) * 1e-3
        e2e = {"value": flops * n_e2e / t_e2e / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": n_e2e, "copies_declared": True}
    pk = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = float(pk.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    achieved = flops / (t / steps) / 1e12
    fields = {"value": achieved, "unit": "TFLOP/s", "steps": steps, "warmup": warmup, "ms_per_step": t / steps * 1e3,
              "us_per_step": t / steps * 1e6, "dtype": "bf16", "config": mla_workload_config(case, name),
              "clocks": clocks, "e2e": e2e, "gpu_launches": 3 * steps,
              "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                           "frac": achieved / peak, "traffic": profiled_traffic(MLA_PROFILE_SUMMARY),
                           "ncu_tensor_pipe_pct": profiled_field(MLA_PROFILE_SUMMARY, "tensor_pipe_pct"),
                           "kernel": "mla_prefill_kernel",
                           "timed": "whole step: mla_stage_kernel, mla_prefill_kernel (S once per row tile, the "
                                    "first 256 output columns; exports P) and mla_replay_kernel (the other 256 "
                                    "columns from the export), each the programmatic dependent of the one before",
                           "peak_source": "measured" if pk else "fallback",
                           "algorithmic_flops_per_launch": int(flops), "avg_launch_us": t / steps * 1e6},
              "wall_s_timed_region": wall}
    if cpu_leg:
        fields["cpu_baseline"] = mla_cpu_baseline(case, budget_s=cpu_budget_s)
    return fields


def run_mla(args):
    import torch
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    from paged_kv_gqa_table_gb300 import binding as B
    B.load()
    fields = measure_mla(args.workload, device, args.steps, args.warmup, e2e_leg=not args.skip_e2e,
                         cpu_leg=not args.skip_cpu_baseline, sample_clocks=True)
    line = {"metric": MLA_METRIC, "n_gpus": 1, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "data": "synthetic (seeded N(0,1) bf16)"}
    line.update(fields)
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE,
                    choices=["llama3_8b_decode", "long_context_decode", "gqa6_d256_vllm_decode", "tiny",
                             "llama3_8b_decode_fp8", "llama3_8b_spec_decode_q4", "mla_prefill_h16"])
    ap.add_argument("--skip-e2e", action="store_true", help="omit the end-to-end leg (profiling runs)")
    ap.add_argument("--skip-cpu-baseline", action="store_true", help="omit the CPU oracle leg (profiling runs)")
    ap.add_argument("--skip-per-config", action="store_true",
                    help="measure the headline workload only (profiling runs)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.workload == "mla_prefill_h16":
        return run_mla_reference(args) if args.impl == "reference" else run_mla(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
