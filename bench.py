"""Benchmark: chunked-prefill tokens/s per layer for one 4096-token chunk.

One step is the whole hot path for one chunk of one attention layer:
  bsx_xattn_estimate (scores, softmax, block sums, selection)
  -> bsx_bsa_prefill on the history key blocks
  -> bsx_bsa_prefill on the current chunk's key blocks
  -> bsx_merge_attn of the two (O, LSE) pairs
  -> bsx_map_mask_to_cpu_blocks (1024-token CPU blocks)
on the default workload "llama8b-32k-chunk4096" (32 q-heads, 8 kv-heads,
head_dim 128, bf16, a 4096-token chunk at q_start_pos 28672 against 32768
causal keys, stride 8, threshold 0.95, seeded planted-direction inputs).

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events
on the launching stream; L2 is flushed (a 256 MiB write) between timed steps,
outside the events.  value = tokens/s/layer over all ranks (each rank runs an
independent replica; the path has no cross-GPU exchange).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--step chunk|fused|offload|prefill|chunked]
    python bench.py --sweep              # density sweep, one JSON line per point
    python bench.py --sparse             # the sparse-regime workloads, one line each
    python bench.py --impl reference     # the fp64 CPU oracle, timed on a sample
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_sparse_long_xattn_gb300.inputs import CONFIGS, make_workload  # noqa: E402

DEFAULT_WORKLOAD = "llama8b-32k-chunk4096"
METRIC = "chunked-prefill tokens/s/layer at 32K ctx; % of bf16 TC / HBM roofline"
UNIT = "tokens/s/layer"
DOMINANT = "bsa_prefill"
# Dense bf16 tensor-core figures for the clock-normalised and datasheet
# fractions: a tcgen05 kind::f16 MMA of M128 N128 K16 retires in 64 SM cycles
# (8192 flop per cycle per SM, measured in isolation on this part), and the
# datasheet's dense bf16 figure for the whole GPU.
MMA_FLOP_PER_CLK_SM = 8192
DATASHEET_BF16_TFLOPS = 2250.0
BSA_SOURCES = ("bsa_tc.cu", "bsa_tc.cuh", "bsa_simt.cu", "common.cuh", "tc_common.cuh")
FUSED_SOURCES = ("fused_tc.cuh", "fused_tc.cu", "fused_d128_e2.cu", "fused_two_d128_e2.cu",
                 "estimate_tc.cuh", "bsa_tc.cuh", "common.cuh", "tc_common.cuh")


def _env_rank():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def _peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained or None, source)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return (p["hbm_gbs"], p["bf16_tflops"], p.get("bf16_tflops_sustained"),
                "measured (MEASURED_PEAKS.json, burst)")
    return 6800.0, 1900.0, 1700.0, "fallback"


def _source_sha(names):
    h = hashlib.sha256()
    for n in names:
        p = os.path.join(ROOT, "block_sparse_long_xattn_gb300", "csrc", n)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def _traffic_per_launch(kernel_key, sources=BSA_SOURCES):
    """DRAM bytes per launch of the dominant kernel from a committed ncu
    summary, or None when it is absent or was taken on different source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    e = t.get(kernel_key)
    if not e or e.get("source_sha") != _source_sha(sources):
        return None
    return e.get("bytes_per_launch_full")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.window = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            # 20 ms is about as often as the driver refreshes these values
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def mark(self, t0, t1):
        """Host wall-clock bounds of the timed region: only samples taken
        inside it are summarised."""
        self.window = (t0, t1)

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), float(parts[4]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if self.window is not None:
            t0, t1 = self.window
            rows = [r for r in rows if t0 <= r[0] <= t1]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "samples": 0,
                    "reasons": ["no samples inside the timed region"]}
        reasons = sorted({self.REASONS[i] for r in rows for i, v in enumerate(r[4])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in rows),
                "sm_mhz_min": min(r[1] for r in rows),
                "sm_max_mhz": max(r[2] for r in rows),
                "power_w_max": max(r[3] for r in rows), "samples": len(rows),
                "reasons": reasons}


def bsa_flops(mask: np.ndarray, q_start_pos: int, kb_begin: int, kb_end: int, d: int) -> float:
    """4*d flops per (query, key) pair the block-sparse attention computes:
    whole 128x128 tiles below the diagonal, the causal half on it."""
    B, Hq, nqb, nkb = mask.shape
    cur = q_start_pos // 128
    m = mask[..., kb_begin:kb_end].astype(bool)
    kb = np.arange(kb_begin, kb_end)[None, None, None, :]
    diag = cur + np.arange(nqb)[None, None, :, None]
    pairs = np.where(kb < diag, 128 * 128, np.where(kb == diag, 128 * 129 // 2, 0))
    return float(4 * d * (m * pairs).sum())


def estimate_flops(cfg, q_len, q_start_pos, stride):
    """2*d*S flops per allowed reshaped (I, J) pair and q-head."""
    R = q_len // stride
    I = q_start_pos // stride + np.arange(R)
    pairs = float((I + 1).sum())
    return 2.0 * cfg["d"] * stride * pairs * cfg["Hq"] * cfg["B"]


def aggregate_ranks(local_ms, tokens_per_rank, world, device):
    """Whole-job throughput: every rank runs its own replica, so the job
    takes the slowest rank's time (max over ranks) and processes
    tokens_per_rank on each rank.  Returns (max times, total tokens,
    tokens/s from the first time)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(local_ms, dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    times = t.tolist()
    tokens = tokens_per_rank * world
    return times, tokens, tokens / (times[0] / 1e3)


# ---------------------------------------------------------------------------
def run_gpu(args):
    import torch
    import torch.distributed as dist

    import block_sparse_long_xattn_gb300 as bsx

    rank, world, local = _env_rank()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = dict(CONFIGS[args.workload])
    S, tau = cfg.pop("stride"), cfg.pop("threshold")
    cfg.pop("chunk", None)
    w = make_workload(seed=args.seed + rank, **cfg)
    B, Lq, Hq, d = w.q.shape
    P, Lk, Hkv = w.q_start_pos, w.k.shape[1], cfg["Hkv"]
    cur, nkb = P // 128, Lk // 128
    cpu_tokens = 1024
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    host = {n: torch.from_numpy(x).to(tdt).pin_memory() for n, x in
            (("q", w.q), ("k", w.k), ("v", w.v))}
    dq, dk, dv = (host[n].to(dev) for n in ("q", "k", "v"))
    mask = torch.empty((B, Hq, Lq // 128, nkb), dtype=torch.uint8, device=dev)
    omask = torch.empty_like(mask)
    ws = torch.empty(bsx.bsx_estimate_workspace_bytes(bsx.shape_of(dq, dk), Lq, P, S),
                     dtype=torch.uint8, device=dev)
    oh = torch.empty_like(dq)
    oc = torch.empty_like(dq)
    lh = torch.empty((B, Hq, Lq), dtype=torch.float32, device=dev)
    lc = torch.empty_like(lh)
    keep = torch.empty((B, P // cpu_tokens), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    e4m3 = args.estimator == "e4m3"
    if e4m3:
        # e4m3 copies of Q and K for the estimator: the history's K is kept in
        # e4m3 next to the bf16 KV (made once here); each step quantizes the
        # chunk's Q and the chunk's own keys
        if B != 1:
            raise SystemExit("--estimator e4m3 runs batch 1 (the chunk's keys are one slice)")
        q8 = torch.empty(dq.shape, dtype=torch.float8_e4m3fn, device=dev)
        k8 = bsx.bsx_quantize_e4m3(dk)
        torch.cuda.synchronize()

    def est(q, k, v):
        if e4m3:
            bsx.bsx_quantize_e4m3(q, out=q8, stream=stream)
            bsx.bsx_quantize_e4m3(k[:, P:], out=k8[:, P:], stream=stream)
            q, k = q8, k8
        bsx.bsx_xattn_estimate(q, k, P, S, tau, mask=mask, workspace=ws, stream=stream)

    def bsa(m, kb0, kb1, o, lse):
        return lambda q, k, v: bsx.bsx_bsa_prefill(q, k, v, m, P, kb0, kb1, o=o, lse=lse,
                                                   stream=stream)

    def bsa_split(m):
        # history and current chunk, one launch, each into its own (O, LSE)
        return lambda q, k, v: bsx.bsx_bsa_prefill_split(q, k, v, m, P, o_hist=oh, lse_hist=lh,
                                                         o_curr=oc, lse_curr=lc, stream=stream)

    def merge_map(q, k, v):
        bsx.bsx_merge_attn(oh, lh, oc, lc, stream=stream)
        if P >= cpu_tokens:
            bsx.bsx_map_mask_to_cpu_blocks(mask, P, cpu_tokens, keep=keep, stream=stream)

    def offload_mask(q, k, v):
        bsx.bsx_map_mask_to_cpu_blocks(mask, P, cpu_tokens, True, keep=keep, stream=stream)
        bsx.bsx_cpu_block_mask(keep, Lq, P, Hq, cpu_tokens, mask=omask, stream=stream)

    def merge_only(q, k, v):
        bsx.bsx_merge_attn(oh, lh, oc, lc, stream=stream)

    one_kernel = w.dtype == "bf16" and nkb <= 1024 and not e4m3
    # phases of one step, timed separately; the BSA phases give the roofline
    if args.step == "chunk_kernel" and one_kernel:
        # bsx_chunk_step: estimate, selection, attention on the history and
        # on the current chunk, merge and CPU-block flags in one kernel
        wsc = torch.empty(bsx.bsx_chunk_prefill_workspace_bytes(bsx.shape_of(dq, dk), Lq, P, S),
                          dtype=torch.uint8, device=dev)

        def chunk_step(q, k, v):
            bsx.bsx_chunk_step(q, k, v, P, S, tau, cpu_block_tokens=cpu_tokens, mask=mask,
                               o=oh, lse=lh, o_curr=oc, lse_curr=lc,
                               keep=keep if P >= cpu_tokens else None, workspace=wsc,
                               stream=stream)
        phases = [("chunk_step", chunk_step)]
        launches = 1
    elif args.step in ("chunk", "chunk_kernel"):
        phases = [("estimate", est), ("bsa_split", bsa_split(mask)), ("merge_map", merge_map)]
        launches = 5
    elif args.step in ("fused", "prefill") and not e4m3:
        # bsx_chunk_prefill: one launch (estimate, selection and attention in
        # one kernel where it applies; else the three launches it falls back to)
        wsf = torch.empty(bsx.bsx_chunk_prefill_workspace_bytes(bsx.shape_of(dq, dk), Lq, P, S),
                          dtype=torch.uint8, device=dev)

        def fused_step(q, k, v):
            bsx.bsx_chunk_prefill(q, k, v, P, S, tau, mask=mask, o=oh, lse=lh, workspace=wsf,
                                  stream=stream)
        phases = [("fused_step", fused_step)]
        launches = 1 if one_kernel else 3
    elif args.step in ("fused", "prefill"):
        # e4m3 estimator operands: the estimate and one attention launch
        phases = [("estimate", est), ("bsa_all", bsa(mask, 0, nkb, oh, lh))]
        launches = 3
    elif args.step == "offload":
        phases = [("estimate", est), ("cpu_blocks", offload_mask),
                  ("bsa_split", bsa_split(omask)), ("merge", merge_only)]
        launches = 6
    else:
        raise ValueError(args.step)

    def step(q, k, v, ev=None):
        if ev:
            ev[0].record(stream)
        for i, (name, fn) in enumerate(phases):
            if args.nvtx:
                torch.cuda.nvtx.range_push(name)
            fn(q, k, v)
            if args.nvtx:
                torch.cuda.nvtx.range_pop()
            if ev:
                ev[i + 1].record(stream)

    for _ in range(args.warmup):
        step(dq, dk, dv)
    torch.cuda.synchronize()
    bsa_mask = (omask if args.step == "offload" else mask).cpu().numpy()
    causal_blocks = sum(cur + qb + 1 for qb in range(Lq // 128)) * B * Hq
    density = float(mask.cpu().numpy().astype(bool).sum()) / causal_blocks
    if e4m3:
        launches += 2   # the two quantize launches of each step
    ranges = {"bsa_split": ((0, cur), (cur, nkb)), "bsa_all": ((0, nkb),),
              "fused_step": ((0, nkb),), "chunk_step": ((0, cur), (cur, nkb))}
    flops = {n: sum(bsa_flops(bsa_mask, P, r0, r1, d) for r0, r1 in ranges[n])
             for n, _ in phases if n in ranges}
    est_fl = estimate_flops(cfg, Lq, P, S)
    for n in ("fused_step", "chunk_step"):   # one kernel: the estimate's MMAs and the attention's
        if n in flops:
            flops[n] += est_fl

    np_ = len(phases)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(np_ + 1)]
           for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall0 = time.time()
        for i in range(args.steps):
            flush.zero_()
            step(dq, dk, dv, evs[i])
        torch.cuda.synchronize()
        clk.mark(t_wall0, time.time())
    clocks = clk.summary()
    t_step = [evs[i][0].elapsed_time(evs[i][np_]) for i in range(args.steps)]
    t_phase = {n: float(np.mean([evs[i][j].elapsed_time(evs[i][j + 1])
                                 for i in range(args.steps)]))
               for j, (n, _) in enumerate(phases)}
    ms_step = float(np.mean(t_step))

    # End to end through the C ABI's host-buffer entry point: every step
    # uploads its pinned host Q/K/V (the whole K/V, as if none were resident)
    # and reads O/LSE(/flags) back.  bsx_chunk_step_host puts the uploads, the
    # launches and the read-back on three streams ordered by events.  Two
    # buffer sets alternate, so that one step's copies overlap the other's
    # launches, as an engine prefilling chunk after chunk would run them; the
    # timed region spans all steps, from before the first upload to after
    # the last read-back.  The same steps run one at a time (each synchronised
    # and timed alone) give ms_per_step_serial.
    fused = args.step in ("fused", "prefill")
    offload = args.step == "offload"
    with_keep = keep.numel() > 0 and not fused
    out_host = [torch.empty(oh.shape, dtype=oh.dtype).pin_memory() for _ in range(2)]
    lse_host = [torch.empty(lh.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    keep_host = [torch.empty(keep.shape, dtype=torch.uint8).pin_memory() if with_keep else None
                 for _ in range(2)]
    sets = [bsx.make_chunk_buffers(host["q"], host["k"], P, S, cpu_tokens, offload=offload,
                                   e4m3_estimate=e4m3, fused=fused, with_keep=with_keep,
                                   device=dev) for _ in range(2)]
    up_stream = torch.cuda.Stream(device=dev)
    dn_stream = torch.cuda.Stream(device=dev)

    def host_step(i, up, dn):
        bsx.bsx_chunk_step_host(host["q"], host["k"], host["v"], P, S, tau, buffers=sets[i % 2],
                                o_host=out_host[i % 2], lse_host=lse_host[i % 2],
                                keep_host=keep_host[i % 2], cpu_block_tokens=cpu_tokens,
                                force_first_last=offload, offload=offload, e4m3_estimate=e4m3,
                                fused=fused, stream=stream, upload_stream=up,
                                download_stream=dn)

    n_e2e = max(3, args.steps // 2)
    serial_ms = []
    for i in range(n_e2e):
        flush.zero_()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(up_stream)
        host_step(i, up_stream, dn_stream)
        e1.record(dn_stream)
        torch.cuda.synchronize()
        serial_ms.append(e0.elapsed_time(e1))
    flush.zero_()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(up_stream)
    for i in range(n_e2e):
        host_step(i, up_stream, dn_stream)
    e1.record(dn_stream)
    torch.cuda.synchronize()
    e2e_ms = [e0.elapsed_time(e1) / n_e2e]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in (out_host[0], lse_host[0]))
    if with_keep:
        d2h += keep_host[0].numel()

    (ms_step, ms_e2e), tokens, value = aggregate_ranks(
        [ms_step, float(np.mean(e2e_ms))], B * Lq, world, dev)

    hbm_peak, tc_peak, tc_sustained, peak_src = _peaks()
    bsa_names = [n for n, _ in phases if n in ranges]
    bsa_ms = float(np.mean([t_phase[n] for n in bsa_names]))        # mean launch
    bsa_flops_launch = float(np.mean([flops[n] for n in bsa_names]))
    achieved = bsa_flops_launch / (bsa_ms / 1e3) / 1e12
    traffic = None
    if args.workload == DEFAULT_WORKLOAD and "chunk_step" in t_phase:
        traffic = _traffic_per_launch("chunk_step", FUSED_SOURCES)
    elif args.workload == DEFAULT_WORKLOAD and "bsa_split" in t_phase:
        traffic = _traffic_per_launch("bsa_prefill")
    elif args.workload == DEFAULT_WORKLOAD and "fused_step" in t_phase:
        traffic = _traffic_per_launch("fused_step", FUSED_SOURCES)
    est_bytes = (dq.numel() + dk.numel()) * dq.element_size() + mask.numel()

    kernels = {f"{n}_ms": t for n, t in t_phase.items()}
    if "estimate" in t_phase:
        est_ms = t_phase["estimate"]
        kernels.update({
            "estimate_tflops": est_fl / (est_ms / 1e3) / 1e12,
            "estimate_tc_frac": est_fl / (est_ms / 1e3) / 1e12 / tc_peak,
            "estimate_gbs": est_bytes / (est_ms / 1e3) / 1e9,
            "estimate_hbm_frac": est_bytes / (est_ms / 1e3) / 1e9 / hbm_peak,
        })
    for n in bsa_names:
        kernels[f"{n}_tflops"] = flops[n] / (t_phase[n] / 1e3) / 1e12

    # the step's roofline: every launch at its own bound (estimate at the
    # larger of its tensor and HBM times, attention at the tensor peak, merge
    # and map at the copy bandwidth), summed; tokens/s at that time against
    # the measured tokens/s
    merge_bytes = 3 * oh.numel() * oh.element_size() + 3 * lh.numel() * 4
    roof_ms = {}
    if "estimate" in t_phase:
        roof_ms["estimate"] = max(est_fl / (tc_peak * 1e12), est_bytes / (hbm_peak * 1e9)) * 1e3
    for n in bsa_names:
        roof_ms[n] = flops[n] / (tc_peak * 1e12) * 1e3
    if "merge_map" in t_phase or "merge" in t_phase or "chunk_step" in t_phase:
        roof_ms["merge"] = merge_bytes / (hbm_peak * 1e9) * 1e3
    if ("merge_map" in t_phase or "chunk_step" in t_phase) and P >= cpu_tokens:
        roof_ms["map"] = mask.numel() / (hbm_peak * 1e9) * 1e3
    if "cpu_blocks" in t_phase:
        roof_ms["cpu_blocks"] = 2 * mask.numel() / (hbm_peak * 1e9) * 1e3
    roof_step_ms = sum(roof_ms.values())
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    at_clock = (MMA_FLOP_PER_CLK_SM * n_sm * clocks["sm_mhz"] * 1e6 / 1e12
                if clocks.get("sm_mhz") else None)

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded planted-direction N(0,1) inputs)",
        "config": config_dict(args, world),
        "roofline": {"kernel": next((n for n in ("chunk_step", "fused_step") if n in t_phase),
                                    DOMINANT),
                     "bound": "tensor", "achieved": achieved,
                     "peak": tc_peak, "unit": "TFLOP/s", "frac": achieved / tc_peak,
                     "traffic": traffic, "peak_source": peak_src,
                     # the same launch against the cuBLAS figure sustained under
                     # the power cap (the timed region's clock record says
                     # whether the cap was reached: clocks.reasons)
                     "peak_sustained": tc_sustained,
                     "frac_vs_sustained": achieved / tc_sustained if tc_sustained else None,
                     "flops_per_launch": bsa_flops_launch, "ms_per_launch": bsa_ms,
                     # the same launch against the tensor pipe's own rate at
                     # the median SM clock of the timed region, and against
                     # the datasheet's dense bf16 figure
                     "peak_at_clock": at_clock,
                     "frac_at_clock": achieved / at_clock if at_clock else None,
                     "frac_of_datasheet": achieved / DATASHEET_BF16_TFLOPS},
        "kernels": kernels,
        "density": density,
        # tokens/s as a fraction of its roofline: the step's launches each at
        # their own bound (roofline_ms_per_launch), summed, against the step
        "tokens_roofline_frac": roof_step_ms / ms_step,
        "tokens_roofline": {"value": B * Lq / (roof_step_ms / 1e3), "unit": UNIT,
                            "roofline_ms_per_step": roof_step_ms,
                            "roofline_ms_per_launch": roof_ms},
        "e2e": {"value": tokens / (ms_e2e / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
                "steps": n_e2e, "ms_per_step_serial": float(np.mean(serial_ms)),
                "overlap": "two buffer sets alternate: one step's uploads and read-back "
                           "overlap the other's launches; inputs (160 MiB at 32K) exceed L2"},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline and args.step == "chunk":
        result["cpu_baseline"], ests, heads = oracle_baseline(w, S, tau, args.cpu_heads,
                                                              keep_estimates=True)
        result["near_threshold_rows"] = mask_rows_vs_oracle(mask.cpu().numpy(), ests, heads)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_chunked(args):
    """Chunked prefill of a whole sequence (the 64K / 16 x 4096 workload): one
    step runs the chunk step (estimate over history + chunk, attention on
    history and current chunk in one launch, merge, CPU-block map) for every
    chunk in order, each chunk's queries against all keys before its end.
    value = sequence tokens / step time.  With --step chunk_kernel each
    chunk's step is bsx_chunk_step, one kernel.  The end-to-end leg uploads
    each chunk's Q, K and V rows from pinned host memory (appending to the
    device KV, as a prefill does), runs the chunk step after its upload and
    reads the chunk's O and LSE back, on three streams."""
    import torch
    import torch.distributed as dist

    import block_sparse_long_xattn_gb300 as bsx

    rank, world, local = _env_rank()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = dict(CONFIGS[args.workload])
    S, tau, chunk = cfg.pop("stride"), cfg.pop("threshold"), cfg.pop("chunk")
    w = make_workload(seed=args.seed + rank, q_full=True, **cfg)
    B, L, Hq, d = w.q.shape
    Hkv = cfg["Hkv"]
    if B != 1 or L % chunk:
        raise SystemExit("the chunked step takes batch 1 and whole chunks")
    n_chunks, cpu_tokens = L // chunk, 1024
    host = {n: torch.from_numpy(x).to(torch.bfloat16).pin_memory() for n, x in
            (("q", w.q), ("k", w.k), ("v", w.v))}
    dq, dk, dv = (host[n].to(dev) for n in ("q", "k", "v"))
    o_full = torch.empty_like(dq)
    oc = torch.empty((B, chunk, Hq, d), dtype=dq.dtype, device=dev)
    lc = torch.empty((B, Hq, chunk), dtype=torch.float32, device=dev)
    lse = [torch.empty((B, Hq, chunk), dtype=torch.float32, device=dev)
           for _ in range(n_chunks)]
    masks = [torch.empty((B, Hq, chunk // 128, (c + 1) * chunk // 128), dtype=torch.uint8,
                         device=dev) for c in range(n_chunks)]
    keeps = [torch.empty((B, c * chunk // cpu_tokens), dtype=torch.uint8, device=dev)
             for c in range(n_chunks)]
    ws = torch.empty(bsx.bsx_estimate_workspace_bytes(bsx.shape_of(dq, dk), chunk,
                                                      L - chunk, S),
                     dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    one_kernel = args.step == "chunk_kernel"
    if one_kernel:
        wsc = torch.empty(bsx.bsx_chunk_prefill_workspace_bytes(bsx.shape_of(dq, dk), chunk,
                                                                L - chunk, S),
                          dtype=torch.uint8, device=dev)

    def chunk_step(c, ev=None):
        P = c * chunk
        q, k, v = dq[:, P:P + chunk], dk[:, :P + chunk], dv[:, :P + chunk]
        o = o_full[:, P:P + chunk]
        if one_kernel:
            # the whole chunk step in one kernel; ev brackets it
            if ev:
                ev[0].record(stream)
            bsx.bsx_chunk_step(q, k, v, P, S, tau, cpu_block_tokens=cpu_tokens, mask=masks[c],
                               o=o, lse=lse[c], o_curr=oc, lse_curr=lc,
                               keep=keeps[c] if P >= cpu_tokens else None, workspace=wsc,
                               stream=stream)
            if ev:
                ev[1].record(stream)
            return
        bsx.bsx_xattn_estimate(q, k, P, S, tau, mask=masks[c], workspace=ws, stream=stream)
        if ev:
            ev[0].record(stream)
        bsx.bsx_bsa_prefill_split(q, k, v, masks[c], P, o_hist=o, lse_hist=lse[c],
                                  o_curr=oc, lse_curr=lc, stream=stream)
        if ev:
            ev[1].record(stream)
        bsx.bsx_merge_attn(o, lse[c], oc, lc, stream=stream)
        if P >= cpu_tokens:
            bsx.bsx_map_mask_to_cpu_blocks(masks[c], P, cpu_tokens, keep=keeps[c],
                                           stream=stream)

    for _ in range(args.warmup):
        for c in range(n_chunks):
            chunk_step(c)
    torch.cuda.synchronize()
    flops = sum(bsa_flops(masks[c].cpu().numpy(), c * chunk, 0, c * chunk // 128, d) +
                bsa_flops(masks[c].cpu().numpy(), c * chunk, c * chunk // 128,
                          (c + 1) * chunk // 128, d) for c in range(n_chunks))
    causal = sum(sum(c * chunk // 128 + qb + 1 for qb in range(chunk // 128))
                 for c in range(n_chunks)) * B * Hq
    density = sum(float(masks[c].cpu().numpy().astype(bool).sum())
                  for c in range(n_chunks)) / causal

    ev_step = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
               for _ in range(args.steps)]
    ev_bsa = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)]
               for _ in range(n_chunks)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall0 = time.time()
        for i in range(args.steps):
            flush.zero_()
            ev_step[i][0].record(stream)
            for c in range(n_chunks):
                chunk_step(c, ev_bsa[i][c])
            ev_step[i][1].record(stream)
        torch.cuda.synchronize()
        clk.mark(t_wall0, time.time())
    clocks = clk.summary()
    ms_step = float(np.mean([e[0].elapsed_time(e[1]) for e in ev_step]))
    bsa_ms = float(np.mean([sum(ev_bsa[i][c][0].elapsed_time(ev_bsa[i][c][1])
                                for c in range(n_chunks)) for i in range(args.steps)]))

    # end to end: chunk c's rows go up on one stream, its step runs on the
    # compute stream after them, its O and LSE come back on a third
    o_host = torch.empty(o_full.shape, dtype=o_full.dtype).pin_memory()
    lse_host = torch.empty((n_chunks, B, Hq, chunk), dtype=torch.float32).pin_memory()
    up, dn = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    n_e2e = max(3, args.steps // 2)
    ups = [torch.cuda.Event() for _ in range(n_chunks)]
    dones = [torch.cuda.Event() for _ in range(n_chunks)]
    e2e_ms = []
    for _ in range(n_e2e):
        flush.zero_()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(up)
        for c in range(n_chunks):
            rows = slice(c * chunk, (c + 1) * chunk)
            with torch.cuda.stream(up):
                for n, t in (("q", dq), ("k", dk), ("v", dv)):
                    t[:, rows].copy_(host[n][:, rows], non_blocking=True)
                ups[c].record(up)
            stream.wait_event(ups[c])
            chunk_step(c)
            dones[c].record(stream)
            dn.wait_event(dones[c])
            with torch.cuda.stream(dn):
                o_host[:, rows].copy_(o_full[:, rows], non_blocking=True)
                lse_host[c].copy_(lse[c], non_blocking=True)
        e1.record(dn)
        torch.cuda.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = o_host.numel() * o_host.element_size() + lse_host.numel() * 4

    (ms_step, ms_e2e), tokens, value = aggregate_ranks(
        [ms_step, float(np.mean(e2e_ms))], B * L, world, dev)
    hbm_peak, tc_peak, tc_sustained, peak_src = _peaks()
    if one_kernel:
        # the one kernel's algorithmic flops: the estimate's and the attention's
        flops += sum(estimate_flops(cfg, chunk, c * chunk, S) for c in range(n_chunks))
    achieved = flops / (bsa_ms / 1e3) / 1e12
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded planted-direction N(0,1) inputs)",
        "config": config_dict(args, world),
        "roofline": {"kernel": "chunk_step" if one_kernel else DOMINANT, "bound": "tensor",
                     "achieved": achieved,
                     "peak": tc_peak, "unit": "TFLOP/s", "frac": achieved / tc_peak,
                     "traffic": None, "peak_source": peak_src, "peak_sustained": tc_sustained,
                     "frac_vs_sustained": achieved / tc_sustained if tc_sustained else None,
                     "flops_per_launch": flops / n_chunks, "ms_per_launch": bsa_ms / n_chunks,
                     "launches_per_step": n_chunks},
        "kernels": ({"chunk_step_ms_per_step": bsa_ms, "rest_ms_per_step": ms_step - bsa_ms}
                    if one_kernel else
                    {"bsa_ms_per_step": bsa_ms, "rest_ms_per_step": ms_step - bsa_ms}),
        "density": density,
        "e2e": {"value": tokens / (ms_e2e / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e, "steps": n_e2e,
                "overlap": "chunk c+1's upload runs while chunk c computes; each chunk's "
                           "O/LSE read back while the next computes"},
        "gpu_launches": args.steps * (n_chunks if one_kernel else
                                      4 * n_chunks - sum(1 for c in range(n_chunks)
                                                         if c * chunk < cpu_tokens) + n_chunks),
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


SWEEP_THRESHOLDS = (0.8, 0.9, 0.95, 0.99, 1.0)
SWEEP_ALPHAS = (0.0, 2.0, 4.0)


def run_sweep(args):
    """Density sweep on the 32K / 4096-chunk shapes: for every planted
    strength alpha (0: pure N(0,1), 16 hot blocks otherwise) and threshold,
    the chunk step's mask density, the attention launch's TFLOP/s over the
    selected blocks and the estimator's GB/s and TFLOP/s.  One JSON line per
    point, device-resident inputs, L2 flushed between timed steps."""
    import torch

    import block_sparse_long_xattn_gb300 as bsx

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    hbm_peak, tc_peak, _, peak_src = _peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    base = dict(CONFIGS[DEFAULT_WORKLOAD])
    S = base.pop("stride")
    base.pop("threshold")
    for alpha in SWEEP_ALPHAS:
        c = dict(base, alpha=alpha, n_hot=16 if alpha > 0 else 0)
        w = make_workload(seed=args.seed, **c)
        B, Lq, Hq, d = w.q.shape
        P, Lk = w.q_start_pos, w.k.shape[1]
        cur, nkb = P // 128, Lk // 128
        q, k, v = (torch.from_numpy(x).to(torch.bfloat16).to(dev) for x in (w.q, w.k, w.v))
        mask = torch.empty((B, Hq, Lq // 128, nkb), dtype=torch.uint8, device=dev)
        ws = torch.empty(bsx.bsx_estimate_workspace_bytes(bsx.shape_of(q, k), Lq, P, S),
                         dtype=torch.uint8, device=dev)
        oh, oc = torch.empty_like(q), torch.empty_like(q)
        lh = torch.empty((B, Hq, Lq), dtype=torch.float32, device=dev)
        lc = torch.empty_like(lh)
        keep = torch.empty((B, P // 1024), dtype=torch.uint8, device=dev)
        est_fl = estimate_flops(c, Lq, P, S)
        est_bytes = (q.numel() + k.numel()) * q.element_size() + mask.numel()
        causal_blocks = sum(cur + qb + 1 for qb in range(Lq // 128)) * B * Hq
        for tau in SWEEP_THRESHOLDS:
            def step(ev=None):
                if ev:
                    ev[0].record(stream)
                bsx.bsx_xattn_estimate(q, k, P, S, tau, mask=mask, workspace=ws, stream=stream)
                if ev:
                    ev[1].record(stream)
                bsx.bsx_bsa_prefill_split(q, k, v, mask, P, o_hist=oh, lse_hist=lh,
                                          o_curr=oc, lse_curr=lc, stream=stream)
                if ev:
                    ev[2].record(stream)
                bsx.bsx_merge_attn(oh, lh, oc, lc, stream=stream)
                bsx.bsx_map_mask_to_cpu_blocks(mask, P, 1024, keep=keep, stream=stream)
                if ev:
                    ev[3].record(stream)

            for _ in range(args.warmup):
                step()
            torch.cuda.synchronize()
            m = mask.cpu().numpy()
            density = float(m.astype(bool).sum()) / causal_blocks
            fl = bsa_flops(m, P, 0, cur, d) + bsa_flops(m, P, cur, nkb, d)
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
                   for _ in range(args.steps)]
            with ClockSampler(0) as clk:
                t0 = time.time()
                for i in range(args.steps):
                    flush.zero_()
                    step(evs[i])
                torch.cuda.synchronize()
                clk.mark(t0, time.time())
            t = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(3)] for e in evs])
            t_est, t_bsa, t_rest = (float(x) for x in t.mean(axis=0))
            ms = t_est + t_bsa + t_rest
            bsa_tf = fl / (t_bsa / 1e3) / 1e12
            print(json.dumps({
                "sweep": DEFAULT_WORKLOAD, "alpha": alpha, "threshold": tau,
                "density": density, "ms_per_step": ms,
                "tokens_per_s_layer": B * Lq / (ms / 1e3),
                "bsa_ms": t_bsa, "bsa_tflops": bsa_tf, "bsa_frac": bsa_tf / tc_peak,
                "estimate_ms": t_est, "estimate_gbs": est_bytes / (t_est / 1e3) / 1e9,
                "estimate_hbm_frac": est_bytes / (t_est / 1e3) / 1e9 / hbm_peak,
                "estimate_tflops": est_fl / (t_est / 1e3) / 1e12,
                "estimate_tc_frac": est_fl / (t_est / 1e3) / 1e12 / tc_peak,
                "merge_map_ms": t_rest, "steps": args.steps, "warmup": args.warmup,
                "peak_source": peak_src, "clocks": clk.summary()}), flush=True)
        del q, k, v, ws, oh, oc
    if bsx.bsx_last_error() != 0:
        raise SystemExit("device error word set after the sweep")


def run_sparse(args):
    """The sparse regime: the chunk step (estimate, attention on history and
    current chunk in one launch, merge, map) on each sparse workload (the 32K
    and 128K chunk shapes with a strong planted direction; the estimator
    selects about 6-50% of the causal blocks).  One JSON line per workload:
    the mask density, the step's tokens/s and its roofline fraction, the
    attention launch's TFLOP/s over the selected blocks and its fractions,
    and the fused step (bsx_chunk_prefill, one kernel) and the chunk step as
    one kernel (bsx_chunk_step) on the same inputs with their fractions
    (estimate and attention flops over their time).
    Device-resident inputs, L2 flushed between timed steps."""
    import torch

    import block_sparse_long_xattn_gb300 as bsx
    from block_sparse_long_xattn_gb300.inputs import SPARSE_CONFIGS

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    hbm_peak, tc_peak, tc_sustained, peak_src = _peaks()
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    names = [args.workload] if args.workload in SPARSE_CONFIGS else list(SPARSE_CONFIGS)
    for name in names:
        c = dict(CONFIGS[name])
        S, tau = c.pop("stride"), c.pop("threshold")
        w = make_workload(seed=args.seed, **c)
        B, Lq, Hq, d = w.q.shape
        P, Lk = w.q_start_pos, w.k.shape[1]
        cur, nkb = P // 128, Lk // 128
        q, k, v = (torch.from_numpy(x).to(torch.bfloat16).to(dev) for x in (w.q, w.k, w.v))
        del w
        mask = torch.empty((B, Hq, Lq // 128, nkb), dtype=torch.uint8, device=dev)
        ws = torch.empty(bsx.bsx_estimate_workspace_bytes(bsx.shape_of(q, k), Lq, P, S),
                         dtype=torch.uint8, device=dev)
        oh, oc = torch.empty_like(q), torch.empty_like(q)
        lh = torch.empty((B, Hq, Lq), dtype=torch.float32, device=dev)
        lc = torch.empty_like(lh)
        keep = torch.empty((B, P // 1024), dtype=torch.uint8, device=dev)
        est_fl = estimate_flops(c, Lq, P, S)
        est_bytes = (q.numel() + k.numel()) * q.element_size() + mask.numel()
        merge_bytes = 3 * oh.numel() * oh.element_size() + 3 * lh.numel() * 4
        causal_blocks = sum(cur + qb + 1 for qb in range(Lq // 128)) * B * Hq

        def step(ev=None):
            if ev:
                ev[0].record(stream)
            bsx.bsx_xattn_estimate(q, k, P, S, tau, mask=mask, workspace=ws, stream=stream)
            if ev:
                ev[1].record(stream)
            bsx.bsx_bsa_prefill_split(q, k, v, mask, P, o_hist=oh, lse_hist=lh,
                                      o_curr=oc, lse_curr=lc, stream=stream)
            if ev:
                ev[2].record(stream)
            bsx.bsx_merge_attn(oh, lh, oc, lc, stream=stream)
            bsx.bsx_map_mask_to_cpu_blocks(mask, P, 1024, keep=keep, stream=stream)
            if ev:
                ev[3].record(stream)

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        m = mask.cpu().numpy()
        density = float(m.astype(bool).sum()) / causal_blocks
        fl = bsa_flops(m, P, 0, cur, d) + bsa_flops(m, P, cur, nkb, d)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
               for _ in range(args.steps)]
        with ClockSampler(0) as clk:
            t0 = time.time()
            for i in range(args.steps):
                flush.zero_()
                step(evs[i])
            torch.cuda.synchronize()
            clk.mark(t0, time.time())
        clocks = clk.summary()
        t = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(3)] for e in evs])
        t_est, t_bsa, t_rest = (float(x) for x in t.mean(axis=0))

        # the fused step on the same inputs: bsx_chunk_prefill, one kernel
        # (estimate, selection, attention over every key block; no merge)
        wsf = torch.empty(bsx.bsx_chunk_prefill_workspace_bytes(bsx.shape_of(q, k), Lq, P, S),
                          dtype=torch.uint8, device=dev)
        maskf = torch.empty_like(mask)

        def fused():
            bsx.bsx_chunk_prefill(q, k, v, P, S, tau, mask=maskf, o=oh, lse=lh, workspace=wsf,
                                  stream=stream)
        for _ in range(args.warmup):
            fused()
        torch.cuda.synchronize()
        fl_f = bsa_flops(maskf.cpu().numpy(), P, 0, nkb, d) + est_fl
        ef = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            ef[i][0].record(stream)
            fused()
            ef[i][1].record(stream)
        torch.cuda.synchronize()
        t_fused = float(np.mean([e[0].elapsed_time(e[1]) for e in ef]))

        # the chunk step as one kernel: bsx_chunk_step (estimate, selection
        # with the CPU-block flags, attention on history and current chunk
        # merged in each CTA)
        keepk = torch.empty((B, P // 1024), dtype=torch.uint8, device=dev) if P >= 1024 else None

        def chunk_kernel():
            bsx.bsx_chunk_step(q, k, v, P, S, tau, mask=maskf, o=oh, lse=lh, o_curr=oc,
                               lse_curr=lc, keep=keepk, workspace=wsf, stream=stream)
        for _ in range(args.warmup):
            chunk_kernel()
        torch.cuda.synchronize()
        fl_k = (bsa_flops(maskf.cpu().numpy(), P, 0, cur, d) +
                bsa_flops(maskf.cpu().numpy(), P, cur, nkb, d) + est_fl)
        ek = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            ek[i][0].record(stream)
            chunk_kernel()
            ek[i][1].record(stream)
        torch.cuda.synchronize()
        t_kernel = float(np.mean([e[0].elapsed_time(e[1]) for e in ek]))
        ms = t_est + t_bsa + t_rest
        bsa_tf = fl / (t_bsa / 1e3) / 1e12
        roof_ms = (max(est_fl / (tc_peak * 1e12), est_bytes / (hbm_peak * 1e9))
                   + fl / (tc_peak * 1e12) + (merge_bytes + m.size) / (hbm_peak * 1e9)) * 1e3
        at_clock = (MMA_FLOP_PER_CLK_SM * n_sm * clocks["sm_mhz"] * 1e6 / 1e12
                    if clocks.get("sm_mhz") else None)
        print(json.dumps({
            "sparse": name, "alpha": c["alpha"], "n_hot": c["n_hot"], "stride": S,
            "threshold": tau, "density": density, "ms_per_step": ms,
            "tokens_per_s_layer": B * Lq / (ms / 1e3), "tokens_roofline_frac": roof_ms / ms,
            "bsa_ms": t_bsa, "bsa_flops": fl, "bsa_tflops": bsa_tf,
            "bsa_frac": bsa_tf / tc_peak,
            "bsa_frac_at_clock": bsa_tf / at_clock if at_clock else None,
            "estimate_ms": t_est, "estimate_tflops": est_fl / (t_est / 1e3) / 1e12,
            "estimate_tc_frac": est_fl / (t_est / 1e3) / 1e12 / tc_peak,
            "merge_map_ms": t_rest,
            "fused_step": {"ms": t_fused, "tokens_per_s_layer": B * Lq / (t_fused / 1e3),
                           "flops": fl_f, "frac": fl_f / (t_fused / 1e3) / 1e12 / tc_peak,
                           "frac_at_clock": (fl_f / (t_fused / 1e3) / 1e12 / at_clock
                                             if at_clock else None)},
            "chunk_kernel": {"ms": t_kernel, "tokens_per_s_layer": B * Lq / (t_kernel / 1e3),
                             "flops": fl_k, "frac": fl_k / (t_kernel / 1e3) / 1e12 / tc_peak},
            "steps": args.steps, "warmup": args.warmup,
            "peak_source": peak_src, "clocks": clocks}), flush=True)
        del q, k, v, ws, wsf, oh, oc
        torch.cuda.empty_cache()
    if bsx.bsx_last_error() != 0:
        raise SystemExit("device error word set after the sparse runs")


# ---------------------------------------------------------------------------
def _oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_baseline(w, stride, tau, n_heads, keep_estimates=False):
    """Time the fp64 oracle's chunk step on a sample of q-heads and scale it to
    the whole chunk (heads are independent).  With keep_estimates, also
    return the oracle's estimate of each sampled head and the head list."""
    from oracle import xattn_oracle as O
    G = w.q.shape[2] // w.k.shape[2]
    heads = list(range(0, w.q.shape[2], G))[:n_heads]
    ests = []
    t0 = time.perf_counter()
    for h in heads:
        kv = h // G
        est, _, _, _ = O.chunk_step(w.q[:, :, h:h + 1], w.k[:, :, kv:kv + 1],
                                    w.v[:, :, kv:kv + 1], w.q_start_pos, stride, tau, 1024)
        ests.append(est)
    dt = time.perf_counter() - t0
    per_step = dt / len(heads) * w.q.shape[2]
    base = {"value": w.q.shape[0] * w.q.shape[1] / per_step, "unit": UNIT,
            "cores": _oracle_threads(), "kind": "oracle",
            "sample": f"chunk step for {len(heads)} of {w.q.shape[2]} q-heads "
                      f"({dt:.1f} s), scaled by the head count"}
    if keep_estimates:
        return base, ests, heads
    return base


def mask_rows_vs_oracle(mask_gpu, ests, heads, margin_tol=1e-4):
    """The GPU mask rows of the sampled heads against the oracle's: rows,
    rows near the threshold (some exclusive cumulative mass within 1e-4 of the
    target, relative to the row total: exempt from the bit-exact rule), and
    the other rows that differ (0 when the masks agree)."""
    rows = near = differ = 0
    for h, est in zip(heads, ests):
        g = mask_gpu[:, h].astype(bool)
        o = est.mask[:, 0]
        is_near = est.margin[:, 0] <= margin_tol
        same = (g == o).all(axis=-1)
        rows += g.shape[0] * g.shape[1]
        near += int(is_near.sum())
        differ += int((~same & ~is_near).sum())
    return {"heads": heads, "rows": rows, "near_threshold": near,
            "other_rows_differing": differ, "margin_tol": margin_tol}


def config_dict(args, world):
    """The workload description both arms print."""
    cfg = dict(CONFIGS[args.workload])
    B, Hq, Hkv, d = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["d"]
    out = {"workload": args.workload, "step": args.step, "B": B, "Hq": Hq, "Hkv": Hkv,
           "d": d, "stride": cfg["stride"], "threshold": cfg["threshold"],
           "cpu_block_tokens": 1024, "parallelism": f"replicas{world}",
           "l2": "flushed (256 MiB write) between timed steps", "seed": args.seed,
           "estimator_operands": args.estimator}
    if "chunk" in cfg and args.step in ("chunked", "chunk_kernel"):
        out.update({"seq_len": cfg["Lk"], "chunk": cfg["chunk"],
                    "chunks": cfg["Lk"] // cfg["chunk"]})
    else:
        out.update({"q_len": cfg["Lk"] - cfg["q_start_pos"], "q_start_pos": cfg["q_start_pos"],
                    "Lk": cfg["Lk"]})
    return out


def run_reference(args):
    """The fp64 oracle as the reference arm.  One step = the oracle's chunk
    step on one q-head of the workload (a bounded sample: a whole chunk of 32
    heads would take minutes); ms_per_step is that step's measured time, and
    value scales it to the whole chunk by the head count (heads are
    independent)."""
    rank, world, _ = _env_rank()
    if rank != 0:
        return
    cfg = dict(CONFIGS[args.workload])
    S, tau = cfg.pop("stride"), cfg.pop("threshold")
    cfg.pop("chunk", None)
    w = make_workload(seed=args.seed, **cfg)
    for _ in range(args.warmup):
        oracle_baseline(w, S, tau, 1)
    vals = [oracle_baseline(w, S, tau, 1) for _ in range(args.steps)]
    Hq = w.q.shape[2]
    # each sample's tokens/s was scaled by Hq; undo it for the step's own time
    ms = float(np.mean([w.q.shape[1] / v["value"] * 1e3 for v in vals])) / Hq
    value = w.q.shape[0] * w.q.shape[1] / (ms * Hq / 1e3)
    base = dict(vals[-1])
    base["value"] = value
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "step_is": f"the oracle's chunk step on 1 of {Hq} q-heads",
        "value_scaling": f"value = tokens per chunk / (ms_per_step x {Hq} q-heads)",
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded planted-direction N(0,1) inputs)",
        "config": config_dict(args, world),
        "cpu_baseline": base,
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 200 for the GPU arm, about 0.3 s at 32K; "
                         "20 for the reference arm, whose steps take seconds each)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--step", default="chunk",
                    choices=["chunk", "chunk_kernel", "fused", "offload", "prefill", "chunked"],
                    help="chunk: estimate, BSA on history and current chunk, merge, map "
                         "(the default); chunk_kernel: the same step as one kernel "
                         "(bsx_chunk_step); fused: bsx_chunk_prefill, estimate, selection "
                         "and attention over all key blocks in one kernel; offload: the pages' CPU-block-dense history; prefill: "
                         "fused on a whole-sequence workload; chunked: the chunk step on "
                         "every chunk of a whole sequence in order (64K in 16 chunks; "
                         "with chunk_kernel and a chunked workload, one kernel per chunk)")
    ap.add_argument("--estimator", default="bf16", choices=["bf16", "e4m3"],
                    help="operand type of the estimator's scores (e4m3: Q and the chunk's K "
                         "quantized each step, the history's K kept in e4m3)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-heads", type=int, default=4,
                    help="q-heads in the oracle sample of the cpu_baseline leg")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--nvtx", action="store_true",
                    help="wrap each phase of the step in an NVTX range (for a profiler's "
                         "timeline; adds host work to the timed region)")
    ap.add_argument("--sparse", action="store_true",
                    help="the sparse-regime workloads (32K and 128K chunks, 6-50%% of the "
                         "causal blocks selected), one JSON line each; with --workload "
                         "naming one of them, that one only")
    ap.add_argument("--sweep", action="store_true",
                    help="density sweep on the 32K / 4096-chunk shapes (thresholds 0.8-1.0 "
                         "on alpha 0, 2, 4): one JSON line per point")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = (50 if (args.sweep or args.sparse) else 200) \
            if args.impl == "gb300" else 20
    if args.warmup < 3 and args.impl == "gb300":
        ap.error("at least 3 warm-up steps")
    if args.step == "prefill" and args.workload == DEFAULT_WORKLOAD:
        args.workload = "llama8b-32k-prefill"
    if args.step == "chunked":
        if args.workload == DEFAULT_WORKLOAD:
            args.workload = "llama8b-64k-chunked"
        if "chunk" not in CONFIGS[args.workload]:
            ap.error("--step chunked takes a workload with a chunk size")
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    elif args.sparse:
        run_sparse(args)
    elif args.step == "chunked" or (args.step == "chunk_kernel" and
                                    "chunk" in CONFIGS[args.workload]):
        # a whole sequence chunk by chunk (chunk_kernel: one kernel per chunk)
        run_chunked(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
