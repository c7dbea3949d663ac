#!/usr/bin/env python
"""Benchmark of the SPRINT block-decode step on B300.

One bench step decodes one block: the step-0 prefix pass (LM-head
confidences of every prefix row, key-norm scoring and per-modality
selection, KV compaction), then every denoising step (block attention over
the full prefix at step 0 and the pruned prefix afterwards, block LM head,
adaptive unmasking) until the block is unmasked.  The metric is decode
steps per second (tokens per second alongside), whole job, inputs resident
in HBM; `e2e` repeats it through the same public API with the inputs coming
from pinned host memory each block.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...    # the CPU oracle, timed on a sample

Multi-GPU (torchrun, one rank per GPU): every rank decodes its own
independent sequence; there is no data-path collective (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "block-decode steps/s and tokens/s at 32K prefix; % tensor peak / % HBM BW"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100, help="timed blocks")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="prefix-32k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-compare", action="store_true",
                    help="skip the full-retention (r = 1) comparison runs")
    ap.add_argument("--selection", default="modality", choices=["modality", "per_image", "global"],
                    help="keep pools: the two modalities (the paper's), text plus one pool per "
                         "image, or one pool over the whole prefix at --r-global")
    ap.add_argument("--r-global", type=float, default=0.5)
    ap.add_argument("--residual", action="store_true",
                    help="the block LM head reads h + O of the last layer (residual chain)")
    ap.add_argument("--prefix-attn", action="store_true",
                    help="step 0 also runs the prefix's own attention of the full forward "
                         "pass (sprint_prefix_attn) on seeded prefix queries")
    ap.add_argument("--prefix-layout", default="compacted", choices=["compacted", "indexed"],
                    help="later steps read a compacted copy of the kept rows, or the kept "
                         "rows of the full cache through their indices")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- ranks
def rank_info():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend)
    return dist


def barrier(world):
    import torch.distributed as dist
    if world > 1:
        dist.barrier()


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """Largest value of x over all ranks (the job's wall time)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device="cpu") -> float:
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 50 ms) of one GPU while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.f = None

    def __enter__(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.f.flush()
        rows = []
        with open(self.f.name) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 8:
                    rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i] == "Active"})
        pw = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


# Kernel sources whose ncu DRAM counters a profile summary records; the
# bench reports that traffic only while the sources are unchanged.
TRAFFIC_SOURCES = {
    "lmhead_prefix": ["lmhead_tc.cu", "lmhead.cu", "lmhead.cuh", "tc_ptx.cuh", "common.cuh"],
    "lmhead_block": ["lmhead_tc.cu", "lmhead.cu", "lmhead.cuh", "unmask.cuh", "tc_ptx.cuh",
                     "common.cuh"],
    "attn_full": ["attention_tc.cu", "attention.cu", "attention.cuh", "tc_ptx.cuh", "common.cuh"],
    "attn_pruned": ["attention_tc.cu", "attention.cu", "attention.cuh", "tc_ptx.cuh",
                    "common.cuh"],
    "keynorm": ["score_prune.cu", "common.cuh"],
    "score_prune": ["score_prune.cu", "common.cuh"],
    "compact": ["compact.cu", "common.cuh"],
}


def source_digest(stage):
    import hashlib
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES[stage]:
        with open(os.path.join(ROOT, "kv_cache_pruning_step_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(stage, workload):
    """DRAM bytes per launch of `stage` from the committed ncu summary
    profiles/traffic_<workload>.txt (lines: stage bytes source-digest), or
    None when absent or captured from other kernel sources."""
    p = os.path.join(ROOT, "profiles", f"traffic_{workload}.txt")
    if not os.path.exists(p) or stage not in TRAFFIC_SOURCES:
        return None
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 3 and parts[0] == stage:
                return float(parts[1]) if parts[2] == source_digest(stage) else None
    return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- inputs
def build_inputs(w, seqs, device, prefix_attn=False):
    """Seeded prefix and per-step inputs of sequences `seqs` (CSR layout);
    prefix_attn adds the prefix queries Qp of the prefix's own attention."""
    import torch

    from workload import lm_head_weight, prefix_inputs, prefix_queries, step_inputs
    pres = [prefix_inputs(w, seq=s, device="cpu") for s in seqs]
    prefix = {
        "K": torch.cat([p["K"].reshape(-1) for p in pres]),
        "V": torch.cat([p["V"].reshape(-1) for p in pres]),
        "H": torch.cat([p["H"] for p in pres]),
        "theta": torch.cat([p["theta"] for p in pres]),
        "modality": torch.cat([p["modality"] for p in pres]),
        "image": torch.cat([p["image"] for p in pres]),
    }
    if prefix_attn:
        prefix["Qp"] = torch.cat([prefix_queries(w, seq=s, device="cpu").reshape(-1)
                                  for s in seqs])
    counts = [(int((p["modality"] == 0).sum()), int((p["modality"] != 0).sum())) for p in pres]
    steps = []
    for t in range(w.T):
        xs = [step_inputs(w, s, 0, t, device="cpu") for s in seqs]
        steps.append({
            "Q": torch.stack([x["Q"] for x in xs]).contiguous(),
            "Kb": torch.stack([x["Kb"] for x in xs]).contiguous(),
            "Vb": torch.stack([x["Vb"] for x in xs]).contiguous(),
            "h": torch.cat([x["h"] for x in xs]).contiguous(),
            "theta": torch.cat([x["theta"] for x in xs]).contiguous(),
        })
    W = lm_head_weight(w, device="cpu")
    return prefix, steps, W, counts, pres


def selection_args(args, prefix, pres=None):
    """BlockDecoder keywords for the --selection keep pools."""
    out = {"selection": args.selection, "r_global": args.r_global, "residual": args.residual}
    if args.selection == "per_image":
        import torch
        if pres is None:
            raise ValueError("per-image pool sizes need the per-sequence prefixes")
        out["pool_sizes"] = [torch.bincount(p["image"].long().cpu()).tolist() for p in pres]
    return out


def to_device(d, device, non_blocking=False):
    return {k: v.to(device, non_blocking=non_blocking) for k, v in d.items()}


def nbytes(d):
    return sum(v.numel() * v.element_size() for v in d.values())


# ---------------------------------------------------------------- oracle timing
# Prefix rows whose LM-head confidences the CPU legs compute per sample; the
# cpu_baseline leg and the reference arm use the same sample.
CPU_SAMPLE_ROWS = 128


def host_f64(t):
    """fp64 numpy copy of a host tensor (bf16 widened exactly)."""
    import numpy as np
    if hasattr(t, "detach"):
        t = t.detach().cpu()
        if str(t.dtype) in ("torch.bfloat16", "torch.float16"):
            t = t.float()
        t = t.numpy()
    return np.asarray(t, dtype=np.float64)


def cpu_inputs(pres, steps_host, W):
    """Inputs of the CPU legs, widened to fp64 once, before any timing.

    The oracle expands what it is given to fp64 on entry.  Handing it
    bf16 tensors would charge every call the widening of all of W (2.6 GB
    in fp64) or of every layer's keys, and the sample's scale factors would
    then multiply that fixed cost as if it were per-row work."""
    p = pres[0]
    x = steps_host[0]
    one = lambda a: host_f64(a[0])  # noqa: E731  (first sequence of the stacked inputs)
    return {
        "K": host_f64(p["K"]), "V": host_f64(p["V"]), "H": host_f64(p["H"]),
        "theta": host_f64(p["theta"]), "modality": p["modality"].numpy(),
        "image": p["image"].numpy() if "image" in p else None,
        "W": host_f64(W),
        "Q": one(x["Q"]), "Kb": one(x["Kb"]), "Vb": one(x["Vb"]),
        "h": host_f64(x["h"]), "theta_b": host_f64(x["theta"]),
    }


def cpu_baseline(w, ci, steps_per_block, sample_rows=CPU_SAMPLE_ROWS,
                 selection="modality", r_global=0.5):
    """The oracle, as it stands, on a bounded sample of one block.

    `ci` are the fp64 inputs of cpu_inputs (widened before this call).
    Measured: key-norm importance, selection and compaction of the whole
    prefix; prefix confidences of `sample_rows` rows (scaled to all rows:
    the work per row is one row of the logits and its softmax); block
    attention of layer 0 at the full and at the pruned prefix (scaled to
    all layers); the block LM head and unmask of one step (whole)."""
    import numpy as np

    from oracle import sprint_oracle as orc
    try:
        from threadpoolctl import threadpool_info
        cores = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:  # noqa: BLE001
        cores = os.cpu_count()
    n = ci["modality"].size
    t0 = time.perf_counter()
    imp = orc.key_norm_importance(ci["K"])
    t_imp = time.perf_counter() - t0
    rows = np.linspace(0, n - 1, min(sample_rows, n)).astype(np.int64)
    t0 = time.perf_counter()
    c_s, _, _ = orc.lm_confidence(ci["H"], ci["W"], ci["theta"], rows=rows)
    t_conf_sample = time.perf_counter() - t0
    t_conf = t_conf_sample * n / len(rows)
    conf_all = np.full(n, float(np.mean(c_s)))
    conf_all[rows] = c_s
    t0 = time.perf_counter()
    score = orc.composite_score(imp, conf_all, w.alpha)
    if selection == "modality":
        kept = orc.select_kept(score, ci["modality"], w.r_text, w.r_img)
    else:
        pool = ci["image"] if selection == "per_image" else np.zeros(n, np.int64)
        sizes = np.bincount(pool).tolist()
        keep = orc.pool_keep_counts(sizes, selection, w.r_text, w.r_img, r_global)
        kept = orc.select_kept_pools(score, pool, keep)
    Kp = orc.compact(ci["K"], kept)
    Vp = orc.compact(ci["V"], kept)
    t_sel = time.perf_counter() - t0
    t0 = time.perf_counter()
    orc.block_attention(ci["Q"], ci["K"], ci["V"], ci["Kb"], ci["Vb"], layers=[0])
    t_attn_full_l0 = time.perf_counter() - t0
    t0 = time.perf_counter()
    orc.block_attention(ci["Q"], Kp, Vp, ci["Kb"], ci["Vb"], layers=[0])
    t_attn_pruned_l0 = time.perf_counter() - t0
    t0 = time.perf_counter()
    c_b, am_b, _ = orc.lm_confidence(ci["h"][:w.LB], ci["W"], ci["theta_b"][:w.LB])
    orc.unmask_step(c_b, am_b, np.ones(w.LB, bool), np.full(w.LB, -1), 0, w.T, w.tau)
    t_step_head = time.perf_counter() - t0
    extra = max(steps_per_block - 1, 0)
    t_block = (t_imp + t_conf + t_sel + t_attn_full_l0 * w.NL + t_step_head
               + extra * (t_attn_pruned_l0 * w.NL + t_step_head))
    measured = (t_imp + t_conf_sample + t_sel + t_attn_full_l0 + t_attn_pruned_l0
                + t_step_head)
    return {
        "value": steps_per_block / t_block,
        "unit": "steps/s",
        "cores": cores,
        "kind": "oracle",
        "tokens_per_s": w.LB / t_block,
        "block_s_extrapolated": t_block,
        "measured_s": measured,
        "extrapolation": round(t_block / measured, 2),
        "sample": (f"one block of sequence 0 ({n}-row prefix), inputs widened to fp64 once "
                   f"before timing (widening excluded): key norms, selection and "
                   f"compaction of the whole prefix; LM-head confidences of {len(rows)} of "
                   f"{n} prefix rows scaled x{n / len(rows):.0f}; attention of layer 0 of "
                   f"{w.NL} scaled x{w.NL} (full prefix, then pruned); one step's block LM "
                   f"head and unmask; block = step 0 + {extra} pruned steps"),
    }


# ---------------------------------------------------------------- r = 1 comparison
def compare_full_retention(args, w, prefix, steps, counts, W, ms_block, later_ms, pres=None):
    """SPRINT at the workload's keep ratios against full prefix retention
    (r_text = r_img = 1), adaptive and fixed schedule, on the same inputs;
    plus the exactness of r = 1: attention over the "pruned" cache equals
    attention over the full prefix bit for bit."""
    import torch

    from kv_cache_pruning_step_b300 import BlockDecoder
    from kv_cache_pruning_step_b300 import sprint as sp
    step_fn = lambda t: steps[t]  # noqa: E731
    reps = max(3, args.steps // 4)
    indexed = args.prefix_layout == "indexed"
    out = {"sprint": {"r_text": w.r_text, "r_img": w.r_img, "mode": "adaptive",
                      "prefix_layout": args.prefix_layout,
                      "ms_per_block": ms_block, "ms_per_later_step": later_ms}}
    # The same SPRINT decode with the other layout of the pruned prefix.
    other = "compacted" if indexed else "indexed"
    dl = BlockDecoder(W, NL=w.NL, Hq=w.Hq, Hkv=w.Hkv, d=w.d, LB=w.LB, T=w.T, tau=w.tau,
                      r_text=w.r_text, r_img=w.r_img, alpha=w.alpha, modality_counts=counts,
                      indexed=not indexed, **selection_args(args, prefix, pres))
    dl.decode(prefix, step_fn)
    torch.cuda.synchronize()
    dl.timing = {}
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        dl.decode(prefix, step_fn)
    b.record()
    torch.cuda.synchronize()
    assert dl.status.item() == 0, f"device status {dl.status.item()}"
    out[f"sprint_{other}"] = {
        "prefix_layout": other, "ms_per_block": a.elapsed_time(b) / reps,
        "ms_per_later_step": _later_step_ms(dl),
        "stages_ms": {k: statistics.mean(v) for k, v in dl.timing.items()}}
    del dl
    r1_equal = None
    for mode_name, mode in (("adaptive", sp.UNMASK_ADAPTIVE), ("fixed", sp.UNMASK_FIXED)):
        d1 = BlockDecoder(W, NL=w.NL, Hq=w.Hq, Hkv=w.Hkv, d=w.d, LB=w.LB, T=w.T, tau=w.tau,
                          r_text=1.0, r_img=1.0, alpha=w.alpha, mode=mode,
                          modality_counts=counts)
        caught = {}

        def on_step(t, dd):
            if t == 1:
                caught["O"] = dd.O.clone()
        d1.decode(prefix, step_fn, on_step=on_step if r1_equal is None else None)
        if r1_equal is None and "O" in caught:
            x = steps[1]
            O_full = sp.sprint_block_attn(x["Q"], prefix["K"], prefix["V"], d1.prefix_off,
                                          d1.max_rows, d1.total_rows, x["Kb"], x["Vb"],
                                          status=d1.status)
            r1_equal = bool(torch.equal(O_full, caught["O"]))
        torch.cuda.synchronize()
        d1.timing = {}
        n_steps = 0
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            n_steps += d1.decode(prefix, step_fn).steps
        b.record()
        torch.cuda.synchronize()
        assert d1.status.item() == 0, f"device status {d1.status.item()}"
        ms = a.elapsed_time(b) / reps
        out[f"full_retention_{mode_name}"] = {
            "r_text": 1.0, "r_img": 1.0, "mode": mode_name, "ms_per_block": ms,
            "steps_per_block": n_steps / reps, "ms_per_later_step": _later_step_ms(d1)}
        d1.timing = None
        del d1
    out["block_speedup_vs_full_retention_fixed"] = (
        out["full_retention_fixed"]["ms_per_block"] / ms_block)
    out["later_step_speedup_vs_full_retention"] = (
        out["full_retention_fixed"]["ms_per_later_step"] / out["sprint"]["ms_per_later_step"])
    out["r1_pruned_attention_equals_full_bitwise"] = r1_equal
    out["note"] = ("the step-0 prefix LM head (all prefix rows) is part of every SPRINT block "
                   "and of neither full-retention block's later steps; with these synthetic "
                   "confidences the adaptive schedule takes its ceil(m/(T-t)) minimum, so "
                   "step counts equal the fixed schedule's")
    return out


def _later_step_ms(dec):
    """Mean CUDA-event time of one step after step 0 (attention over the
    pruned cache, block LM head, unmask) from the decoder's stage timers."""
    import statistics as st
    tm = dec.timing or {}
    tot = 0.0
    for k in ("attn_pruned", "lmhead_block", "unmask"):
        if k in tm and tm[k]:
            tot += st.mean(tm[k])
    return tot


# ---------------------------------------------------------------- our arm
def run_ours(args):
    import torch

    from kv_cache_pruning_step_b300 import BlockDecoder
    from kv_cache_pruning_step_b300 import sprint as sp
    from workload import WORKLOADS

    rank, world, local = rank_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    w = WORKLOADS[args.workload]
    seqs = [rank * w.S + s for s in range(w.S)]
    prefix_h, steps_h, W_h, counts, pres = build_inputs(w, seqs, "cpu",
                                                        prefix_attn=args.prefix_attn)
    W = W_h.to(dev)
    prefix = to_device(prefix_h, dev)
    steps = [to_device(x, dev) for x in steps_h]
    dec = BlockDecoder(W, NL=w.NL, Hq=w.Hq, Hkv=w.Hkv, d=w.d, LB=w.LB, T=w.T, tau=w.tau,
                       r_text=w.r_text, r_img=w.r_img, alpha=w.alpha, modality_counts=counts,
                       indexed=args.prefix_layout == "indexed",
                       prefix_attn=args.prefix_attn,
                       **selection_args(args, prefix_h, pres))
    step_fn = lambda t: steps[t]  # noqa: E731

    for _ in range(args.warmup):
        dec.decode(prefix, step_fn)
    torch.cuda.synchronize()
    assert dec.status.item() == 0, f"device status {dec.status.item()}"

    props = torch.cuda.get_device_properties(dev)
    gpu_id = f"GPU-{props.uuid}" if getattr(props, "uuid", None) else str(local)
    # Inside the timed region CUDA events bracket only the prefix LM head
    # (the roofline kernel): an event between two kernels would keep the
    # second from launching before the first ends.  Every stage's time comes
    # from a separate pass after the timed region.
    dec.timing = {}
    dec.timing_stages = {"lmhead_prefix"}
    n_steps = 0
    hist = {}
    launches0 = sp.sprint_kernel_launches()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_id) as clk:
        barrier(world)
        torch.cuda.synchronize()
        start.record()
        # Block i+1 is enqueued before block i's step counts are read, so the
        # GPU never waits for the host between blocks.
        pend = None
        for i in range(args.steps + 1):
            cur = dec.decode(prefix, step_fn, wait=False) if i < args.steps else None
            if pend is not None:
                res = dec.finish(pend)
                n_steps += res.steps
                for a in res.accepted_per_step:
                    for v in a:
                        hist[v] = hist.get(v, 0) + 1
            pend = cur
        end.record()
        torch.cuda.synchronize()
        barrier(world)
    launches = sp.sprint_kernel_launches() - launches0
    elapsed = start.elapsed_time(end) / 1e3
    timed_ms = {k: statistics.mean(v) for k, v in dec.timing.items()}
    # Stage breakdown: a separate pass with events around every stage.
    dec.timing = {}
    dec.timing_stages = None
    breakdown_blocks = max(3, args.steps // 10)
    for _ in range(breakdown_blocks):
        dec.decode(prefix, step_fn)
    torch.cuda.synchronize()
    stage_ms = {k: statistics.mean(v) for k, v in dec.timing.items()}
    stage_launches = {k: len(v) for k, v in dec.timing.items()}
    stage_ms.update(timed_ms)  # the roofline kernel: measured inside the timed region
    dec.timing = None
    # Confidence histograms, outside the timed region: every prefix c_i of
    # the last block, and the block's c_n at every step of one stepwise
    # decode of the same block (the unmask rule sees these).
    blk_conf = []
    dec.decode_stepwise(prefix, step_fn,
                        on_step=lambda t, d: blk_conf.append(d.conf_blk.clone()))

    def histo(x):
        return [int(v) for v in torch.histc(x.float(), bins=10, min=0.0, max=1.0).tolist()]
    blk_all = torch.cat(blk_conf)
    conf_hist = {"bins": "10 equal bins over [0, 1]", "prefix_c": histo(dec.conf_prefix),
                 "block_c_every_step": histo(blk_all),
                 "block_c_above_tau": int((blk_all > w.tau).sum().item()),
                 "block_c_max": float(blk_all.max().item())}
    assert dec.status.item() == 0, f"device status {dec.status.item()}"

    t_job = max_over_ranks(elapsed, world, dev)
    total_steps = sum_over_ranks(n_steps, world, dev)
    blocks = args.steps * world
    value = total_steps / t_job
    tokens_per_s = blocks * w.S * w.LB / t_job

    # e2e: the same decode with every block's inputs copied from pinned host
    # memory and the decoded tokens read back.  Copies run on their own
    # stream into two alternating device buffer sets, so block i+1's inputs
    # travel while block i computes; the first copy is inside the timed region.
    # As above, block i's step counts are read after block i+1 is enqueued.
    e2e = None
    if not args.no_e2e:
        pin = lambda d: {k: v.pin_memory() for k, v in d.items()}  # noqa: E731
        prefix_p = pin(prefix_h)
        steps_p = [pin(x) for x in steps_h]
        tok_host = torch.empty((w.S, w.LB), dtype=torch.int32, pin_memory=True)
        h2d = nbytes(prefix_h) + sum(nbytes(x) for x in steps_h)
        d2h = tok_host.numel() * 4
        bufs = [({k: torch.empty_like(v, device=dev) for k, v in prefix_h.items()},
                 [{k: torch.empty_like(v, device=dev) for k, v in x.items()} for x in steps_h])
                for _ in range(2)]
        copy_stream = torch.cuda.Stream(device=dev)
        compute = torch.cuda.current_stream(dev)
        ready = [torch.cuda.Event() for _ in range(2)]
        free = [torch.cuda.Event() for _ in range(2)]

        def enqueue_copy(b):
            copy_stream.wait_event(free[b])
            with torch.cuda.stream(copy_stream):
                for k, v in prefix_p.items():
                    bufs[b][0][k].copy_(v, non_blocking=True)
                for xd, xp in zip(bufs[b][1], steps_p):
                    for k, v in xp.items():
                        xd[k].copy_(v, non_blocking=True)
            ready[b].record(copy_stream)

        for b in range(2):
            free[b].record(compute)
        e_steps = 0
        barrier(world)
        torch.cuda.synchronize()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(compute)
        copy_stream.wait_event(s2)
        enqueue_copy(0)
        pend = None
        for i in range(args.steps):
            b = i % 2
            if i + 1 < args.steps:
                enqueue_copy(1 - b)
            compute.wait_event(ready[b])
            pre_b, steps_b = bufs[b]
            cur = dec.decode(pre_b, lambda t, s=steps_b: s[t], wait=False)
            tok_host.copy_(cur.tokens, non_blocking=True)
            free[b].record(compute)
            if pend is not None:
                e_steps += dec.finish(pend).steps
            pend = cur
        e_steps += dec.finish(pend).steps
        e2.record(compute)
        torch.cuda.synchronize()
        barrier(world)
        t_e2e = max_over_ranks(s2.elapsed_time(e2) / 1e3, world, dev)
        e2e = {"value": sum_over_ranks(e_steps, world, dev) / t_e2e, "unit": "steps/s",
               "tokens_per_s": blocks * w.S * w.LB / t_e2e,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h + 4 * w.S * w.T,
               "copies": "pinned host -> device on a copy stream, double-buffered: block i+1's "
                         "inputs copy while block i decodes"}

    peaks, peak_kind = load_peaks()
    n_rows = dec.total_rows
    kept = dec.total_kept
    row_b = w.NL * w.Hkv * w.d * 2
    seq_rows = [dec.prefix_off_host[i + 1] - dec.prefix_off_host[i] for i in range(dec.S)]
    work = {  # algorithmic work per launch of each stage
        "lmhead_prefix": ("tensor", 2.0 * n_rows * w.D * w.V),
        # QK^T and PV over every (query, key) pair of each prefix, all heads and layers
        "prefix_attn": ("tensor", sum(4.0 * n * n * w.Hq * w.d * w.NL for n in seq_rows)),
        "keynorm": ("hbm", n_rows * row_b),
        # with the key norms on a side stream under the prefix LM head, the
        # stage is the selection alone: a chain of cluster barriers
        "score_prune": (("latency", None) if "keynorm" in stage_ms else ("hbm", n_rows * row_b)),
        "compact": ("hbm", 2 * 2 * kept * row_b),
        "attn_full": ("hbm", 2 * (n_rows + w.S * w.LB) * row_b),
        "attn_pruned": ("hbm", 2 * (kept + w.S * w.LB) * row_b),
        # the block LM head streams W once: HBM-bound for few rows, tensor-bound
        # once its arithmetic intensity (about S * LB flop per byte) passes
        # the machine's ridge (peak flop/s over copy bytes/s)
        "lmhead_block": (("tensor", 2.0 * w.S * w.LB * w.D * w.V)
                         if w.S * w.LB > peaks["bf16_tflops"] * 1e3 / peaks["hbm_gbs"]
                         else ("hbm", w.V * w.D * 2)),
    }
    kernels = {}
    for k, (bound, amount) in work.items():
        if k not in stage_ms:
            continue
        sec = stage_ms[k] / 1e3
        traffic = profiled_traffic(k, w.name)
        if bound == "latency":
            kernels[k] = {"bound": "latency", "ms": stage_ms[k], "traffic": traffic}
        elif bound == "tensor":
            ach = amount / sec / 1e12
            pk = peaks["bf16_tflops"]
            kernels[k] = {"bound": "tensor", "achieved": ach, "peak": pk, "unit": "TFLOP/s",
                          "frac": ach / pk,
                          "frac_of_sustained": ach / peaks["bf16_tflops_sustained"],
                          "ms": stage_ms[k], "traffic": traffic}
        else:
            ach = amount / sec / 1e9
            pk = peaks["hbm_gbs"]
            kernels[k] = {"bound": "hbm", "achieved": ach, "peak": pk, "unit": "GB/s",
                          "frac": ach / pk, "ms": stage_ms[k], "traffic": traffic,
                          "algorithmic_bytes": amount}
    dom = max(stage_ms, key=lambda k: stage_ms[k] * stage_launches[k])
    r = kernels.get(dom, {})
    roofline = {"kernel": dom, "bound": r.get("bound"), "achieved": r.get("achieved"),
                "peak": r.get("peak"), "unit": r.get("unit"), "frac": r.get("frac"),
                "traffic": r.get("traffic"),
                "peak_source": f"{peak_kind} ("
                + ("bf16 burst; frac_of_sustained against the sustained figure"
                   if r.get("bound") == "tensor" else "copy bandwidth") + ")"}
    if r.get("bound") == "tensor":
        roofline["frac_of_sustained"] = r.get("frac_of_sustained")

    compare = None
    if not args.no_compare:
        later = sum(stage_ms.get(k, 0.0) for k in ("attn_pruned", "lmhead_block", "unmask"))
        compare = compare_full_retention(args, w, prefix, steps, counts, W,
                                         1e3 * elapsed / args.steps, later, pres=pres)

    out = {
        "metric": METRIC, "value": value, "unit": "steps/s", "tokens_per_s": tokens_per_s,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * t_job / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded; shapes and modality layout of the workload)",
        "config": {"workload": w.name, "description": w.description,
                   "prefix_rows": n_rows, "kept_rows": kept, "sequences": w.S,
                   "prefix_attn": bool(args.prefix_attn),
                   "LB": w.LB, "T": w.T, "tau": w.tau, "r_text": w.r_text, "r_img": w.r_img,
                   "alpha": w.alpha, "NL": w.NL, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "D": w.D,
                   "V": w.V, "bench_step": "one block decoded to completion",
                   "prefix_layout": args.prefix_layout, "selection": args.selection,
                   "residual_chain": args.residual,
                   **({"r_global": args.r_global} if args.selection == "global" else {}),
                   "l2": "inputs larger than L2 (K+V+W+H well above 126 MB)",
                   "parallelism": f"replicas x{world}, one sequence set per GPU"},
        "decode_steps_per_block": n_steps / args.steps,
        "accepted_per_step_hist": {str(k): v for k, v in sorted(hist.items())},
        "confidence_hist": conf_hist,
        "stages_ms": stage_ms, "stage_launches": stage_launches,
        "stages_ms_source": (f"lmhead_prefix: CUDA events inside the timed region; other stages: "
                             f"{breakdown_blocks} further blocks with events around every stage"),
        "kernels": kernels,
        "roofline": roofline, "gpu_launches": launches, "clocks": clk.summary(),
        "e2e": e2e, "full_retention_comparison": compare,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ci = cpu_inputs(pres, steps_h, W_h)
        # one untimed pass first (thread pools, first touch of the widened
        # inputs), as the reference arm's warm-up does
        cpu_baseline(w, ci, n_steps / args.steps, selection=args.selection,
                     r_global=args.r_global)
        out["cpu_baseline"] = cpu_baseline(w, ci, n_steps / args.steps,
                                           selection=args.selection, r_global=args.r_global)
        out["cpu_baseline"]["warmup"] = 1
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        dist.destroy_process_group()


# ---------------------------------------------------------------- sequential blocks
def run_sequential(args):
    """Workloads of several blocks decoded in order on one sequence whose
    prefix grows by the generated block each time (the 64-block workload).
    One bench step decodes every block; with the prefix-confidence cache on,
    a block's step-0 LM head runs only on the rows added since the previous
    block (bit-identical results below 4096 prefix rows).  The same pass
    without the cache is timed alongside."""
    import torch

    from kv_cache_pruning_step_b300 import BlockDecoder
    from kv_cache_pruning_step_b300 import sprint as sp
    from workload import WORKLOADS, lm_head_weight, prefix_inputs, step_inputs

    rank, world, local = rank_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    w = WORKLOADS[args.workload]
    W = lm_head_weight(w, device="cpu").to(dev)
    pres, steps, counts = [], [], []
    for b in range(w.blocks):
        p = prefix_inputs(w, seq=rank, block=b, device="cpu")
        pres.append({k: v.to(dev) for k, v in p.items()})
        m = p["modality"]
        counts.append([(int((m == 0).sum()), int((m != 0).sum()))])
        xs = [step_inputs(w, rank, b, t, device="cpu") for t in range(w.T)]
        steps.append([{"Q": x["Q"][None].contiguous().to(dev),
                       "Kb": x["Kb"][None].contiguous().to(dev),
                       "Vb": x["Vb"][None].contiguous().to(dev),
                       "h": x["h"].to(dev), "theta": x["theta"].to(dev)} for x in xs])
    dec = BlockDecoder(W, NL=w.NL, Hq=w.Hq, Hkv=w.Hkv, d=w.d, LB=w.LB, T=w.T, tau=w.tau,
                       r_text=w.r_text, r_img=w.r_img, alpha=w.alpha,
                       modality_counts=counts[-1],  # the largest: no buffer growth
                       indexed=args.prefix_layout == "indexed")

    def one_pass(cache):
        # Blocks are enqueued without waiting: block b's step count is read
        # after block b+1 is on the stream, so the GPU never waits for the
        # host between blocks (the blocks still run in stream order).
        n_steps, prev, pend = 0, 0, None
        for b in range(w.blocks):
            dec.set_prefix(counts[b])
            cur = dec.decode(pres[b], lambda t, s=steps[b]: s[t],
                             conf_from=prev if cache and b > 0 else 0, wait=False)
            if pend is not None:
                n_steps += dec.finish(pend).steps
            pend = cur
            prev = dec.total_rows
        return n_steps + dec.finish(pend).steps

    for _ in range(args.warmup):
        one_pass(True)
    torch.cuda.synchronize()
    timings = {}
    # In the timed passes CUDA events bracket only the block LM head (the
    # roofline kernel of this workload): an event between two kernels would
    # keep the second from launching before the first ends.  Every stage's
    # time comes from one more pass afterwards.
    for cache in (True, False):
        dec.timing = {} if cache else None
        dec.timing_stages = {"lmhead_block"}
        launches0 = sp.sprint_kernel_launches()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_steps = 0
        reps = args.steps if cache else max(1, args.steps // 4)
        with ClockSampler(str(local)) as clk:
            barrier(world)
            torch.cuda.synchronize()
            a.record()
            for _ in range(reps):
                n_steps += one_pass(cache)
            b.record()
            torch.cuda.synchronize()
        timings[cache] = (a.elapsed_time(b) / 1e3, n_steps, reps,
                          sp.sprint_kernel_launches() - launches0, clk.summary(),
                          dict(dec.timing or {}))
    dec.timing, dec.timing_stages = {}, None
    one_pass(True)
    torch.cuda.synchronize()
    breakdown = {k: statistics.mean(v) for k, v in dec.timing.items()}
    dec.timing = None
    assert dec.status.item() == 0, f"device status {dec.status.item()}"
    t, n_steps, reps, launches, clocks, stage = timings[True]
    t_job = max_over_ranks(t, world, dev)
    total = sum_over_ranks(n_steps, world, dev)
    stage_ms = dict(breakdown)
    stage_ms.update({k: statistics.mean(v) for k, v in stage.items()})
    peaks, peak_kind = load_peaks()
    ach = w.V * w.D * 2 / (stage_ms["lmhead_block"] / 1e3) / 1e9
    t0, s0, r0, _, _, _ = timings[False]
    out = {
        "metric": METRIC, "value": total / t_job, "unit": "steps/s",
        "tokens_per_s": reps * world * w.blocks * w.LB / t_job, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_job / reps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded; shapes and modality layout of the workload)",
        "config": {"workload": w.name, "description": w.description, "blocks": w.blocks,
                   "bench_step": f"all {w.blocks} blocks in order, prefix growing by LB",
                   "prefix_confidence_cache": True, "prefix_layout": args.prefix_layout,
                   "parallelism": f"replicas x{world}, one sequence per GPU"},
        "decode_steps_per_pass": n_steps / reps, "stages_ms": stage_ms,
        "stages_ms_source": ("lmhead_block: CUDA events inside the timed region; other "
                             "stages: one further pass with events around every stage"),
        "roofline": {"kernel": "lmhead_block", "bound": "hbm", "achieved": ach,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
                     "traffic": None, "peak_source": f"{peak_kind} (copy bandwidth)"},
        "without_cache": {"ms_per_pass": 1e3 * t0 / r0, "steps_per_pass": s0 / r0,
                          "speedup_of_cache": (t0 / r0) / (t / reps)},
        "gpu_launches": launches, "clocks": clocks, "e2e": None,
    }
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        dist.destroy_process_group()


# ---------------------------------------------------------------- reference arm
def run_reference(args):
    """The CPU oracle as the reference arm: each bench step is one bounded
    sample of a block (the cpu_baseline sample), timed on the host cores;
    the line's value is the block rate extrapolated from the samples."""
    rank, world, local = rank_info()
    if rank != 0:
        return
    from workload import WORKLOADS
    w = WORKLOADS[args.workload]
    prefix_h, steps_h, W_h, counts, pres = build_inputs(w, [0], "cpu")
    ci = cpu_inputs(pres, steps_h, W_h)
    for _ in range(args.warmup):
        cpu_baseline(w, ci, w.T)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline(w, ci, w.T))
    wall = time.perf_counter() - t0
    block_s = statistics.mean(v["block_s_extrapolated"] for v in vals)
    value = w.T / block_s
    cb = dict(vals[-1])
    cb["value"] = value
    cb["block_s_extrapolated"] = block_s
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s",
        "tokens_per_s": w.LB / block_s, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * wall / max(args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "description": w.description,
                   "bench_step": ("one bounded sample of a block (the oracle on the sample "
                                  "cpu_baseline describes); ms_per_step is the measured time "
                                  "of one sample, value the block rate extrapolated from it")},
        "samples": args.steps, "measured_s": wall,
        "extrapolated_ms_per_block": 1e3 * block_s,
        "cpu_baseline": cb, "wall_s": wall,
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


def launch_plan(gpus: int, env=None):
    """How `--gpus N` runs: 'run' in this process, 'spawn' N ranks under
    torch.distributed.run (N > 1 and no launcher around this process), or
    an error when a launcher gave a world size other than N."""
    env = os.environ if env is None else env
    if gpus < 1:
        raise SystemExit(f"--gpus must be at least 1, got {gpus}")
    if "WORLD_SIZE" in env:
        world = int(env["WORLD_SIZE"])
        if world != gpus:
            raise SystemExit(f"--gpus {gpus} but the launcher started {world} rank(s)")
        return "run"
    return "spawn" if gpus > 1 else "run"


def spawn_ranks(gpus: int, argv) -> int:
    """Run this script as `gpus` local ranks (one per GPU) and return the
    launcher's exit code."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={gpus}", "--master-addr", "127.0.0.1", "--master-port",
           str(port), os.path.abspath(__file__), *argv]
    return subprocess.run(cmd).returncode


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    args = parse_args(argv)
    if launch_plan(args.gpus) == "spawn":
        sys.exit(spawn_ranks(args.gpus, argv))
    if args.impl == "reference":
        run_reference(args)
    else:
        from workload import WORKLOADS
        if WORKLOADS[args.workload].blocks > 1:
            run_sequential(args)
        else:
            run_ours(args)


if __name__ == "__main__":
    main()
