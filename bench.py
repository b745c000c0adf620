"""Benchmark of the exact tiled attention forward pass on GB300.

One step = one forward pass (S = QK^T, online softmax, O = PV, LSE) over the
whole workload, i.e. one launch of the forward kernel through the C ABI.
Default workload: B=1, H=32, N=16384, d=128, bf16, causal -- the
long-context batch-1 case the throughput target is set on.  Inputs (403 MB)
exceed the 129 MB L2, so no flush is needed between steps; a workload whose
inputs fit in the L2 is timed launch by launch with the L2 overwritten (a
258 MB write, outside the timed intervals) before each one.

Prints one JSON line.  ``value`` is forward TFLOP/s (4*B*H*N^2*d, halved for
causal) with inputs resident in HBM; ``e2e`` is the same metric through the
host-buffer entry point with the host<->device copies inside the timed
region; ``roofline`` relates the kernel's CUDA-event time to the measured
dense bf16 tensor peak; ``cpu_baseline`` times the plain CPU oracle on a
bounded sample of rows.  ``--impl reference`` times the oracle alone.

Under torchrun (WORLD_SIZE > 1) every rank runs the same workload on its own
GPU (independent replicas: the forward pass has no exchange step), timing is
the max over ranks and ``value`` sums the ranks' work.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from exact_tiled_attention_fa2_gb300 import synthetic as sy  # noqa: E402

METRIC = "forward attention TFLOP/s at 1 GB300 and % of dense FP16/BF16 tensor peak"
L2_BYTES = 129e6          # GB300 L2
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = 4
KERNEL_SOURCES = ["fa2_common.cuh", "fa2_tile.cuh", "fa2_fwd_dbuf.cuh", "sm103_ptx.cuh", "fa2_internal.h", "fa2_abi.cu"]


BWD_KERNEL_SOURCES = KERNEL_SOURCES + ["fa2_bwd.cuh"]
# per backward main kernel: the sources its code comes from
BWD_SOURCES = {"fa2_bwd_kernel": BWD_KERNEL_SOURCES, "fa2_bwd64_kernel": BWD_KERNEL_SOURCES + ["fa2_bwd64.cuh"],
               "fa2_bwd256_kernel": BWD_KERNEL_SOURCES + ["fa2_bwd256.cuh"]}


def kernel_source_hash(names=None) -> str:
    h = hashlib.sha256()
    for name in names or KERNEL_SOURCES:
        with open(os.path.join(ROOT, "exact_tiled_attention_fa2_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peak(sustained: bool = True):
    """The dense bf16 tensor peak: the cuBLAS rate measured as a seconds-long
    loop under the power cap (sustained: the regime of the >= 1 s timed loop
    here) or as a burst."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d[key]), "of measured (bf16 %s, MEASURED_PEAKS.json)" % ("sustained" if sustained else "burst")
    except Exception:
        return (1700.0, "of fallback (1.7 PFLOP/s bf16 sustained)") if sustained else \
            (1900.0, "of fallback (1.9 PFLOP/s bf16 burst)")


def measured_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "of measured (copy bandwidth, MEASURED_PEAKS.json)"
    except Exception:
        return 6800.0, "of fallback (6.8 TB/s)"


def recorded_traffic(workload: int, kernel: str = "fa2_fwd_dbuf_kernel"):
    """DRAM bytes per launch of `kernel` from the committed ncu summaries, if the
    record was taken on this kernel source (records without a kernel field are
    an earlier forward kernel's and match nothing now)."""
    path = os.path.join(ROOT, "profiles", "traffic_per_launch.txt")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash(BWD_SOURCES.get(kernel, KERNEL_SOURCES))
    with open(path) as f:
        for line in f:
            parts = dict(p.split("=", 1) for p in line.split() if "=" in p)
            if (parts.get("kernel_sha") == src and parts.get("workload") == str(workload)
                    and parts.get("kernel", "") == kernel):
                try:
                    return float(parts["bytes_per_launch"])
                except (KeyError, ValueError):
                    return None
    return None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                maxes.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes), "reasons": sorted(reasons),
                "samples": len(sms)}


ORACLE_ROWS_PER_BATCH = 64


def oracle_sample(w: sy.Workload, q, k, v, target_s: float, rng, threads: int = 0):
    """Run the CPU oracle on random rows until ~target_s seconds; return (flops, seconds, rows).

    Each batch is ORACLE_ROWS_PER_BATCH uniformly random rows of one uniformly
    random (batch, head) slice -- an unbiased sample of the workload's rows
    that lets the oracle widen that slice's K and V once per batch."""
    import oracle

    BH = w.B * w.H
    done_flops, done_s, done_rows = 0.0, 0.0, 0
    while done_s < target_s:
        bh = np.full(ORACLE_ROWS_PER_BATCH, int(rng.integers(0, BH)))
        rows = rng.integers(0, w.N, size=ORACLE_ROWS_PER_BATCH)
        t0 = time.perf_counter()
        oracle.attention_rows(q, k, v, w.dtype, w.scale, w.causal, bh, rows, threads=threads)
        done_s += time.perf_counter() - t0
        keys = (rows + 1) if w.causal else np.full(rows.size, w.N)
        done_flops += float(4.0 * w.d * keys.sum())
        done_rows += rows.size
    return done_flops, done_s, done_rows


def oracle_sample_masked(w: sy.Workload, gen, q, k, v, target_s: float, rng, threads: int = 0):
    """oracle_sample for the general options (band / prefix mask, N_k != N): random rows
    through the oracle's sampled-row masked forward; flops 4*d per visible key."""
    import oracle

    BH, nq, nk = w.B * w.H, gen["seqlen_q"], gen["seqlen_k"]
    vis = sy.visible_keys(nq, nk, gen["window_left"], gen["window_right"], gen["prefix"])
    done_flops, done_s, done_rows = 0.0, 0.0, 0
    while done_s < target_s:
        bh = np.full(ORACLE_ROWS_PER_BATCH, int(rng.integers(0, BH)))
        rows = rng.integers(0, nq, size=ORACLE_ROWS_PER_BATCH)
        t0 = time.perf_counter()
        oracle.attention_rows_masked(q, k, v, w.dtype, w.scale, bh, rows, window_left=gen["window_left"],
                                     window_right=gen["window_right"], prefix_len=gen["prefix"], threads=threads)
        done_s += time.perf_counter() - t0
        done_flops += float(4.0 * w.d * vis[rows].sum())
        done_rows += rows.size
    return done_flops, done_s, done_rows


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The maximum of `value` over every rank of the default process group
    (the value itself when there is no group)."""
    if dist is None or not dist.is_initialized():
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step: float, steps: int, world_size: int, max_ms: float) -> float:
    """Whole-job TFLOP/s: every rank's steps, over the slowest rank's time."""
    return flops_per_step * steps * world_size / (max_ms / 1e3) / 1e12


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args, w, gen=None):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle

    if gen is not None and gen["varlen_seqs"]:
        print(json.dumps({"impl": "reference", "unavailable": "the CPU oracle arm samples rows of unpacked "
                          "problems only; run without --varlen-seqs"}), flush=True)
        return 0
    if gen is None:
        q, k, v = w.inputs()
        sample = lambda t, r: oracle_sample(w, q, k, v, t, r)
    else:
        q = sy.make_qkv(w.B, w.H, gen["seqlen_q"], w.d, w.dtype, w.seed(0), w.q_scale)[0]
        _, k, v = sy.make_qkv(w.B, w.H, gen["seqlen_k"], w.d, w.dtype, w.seed(0) + 1)
        sample = lambda t, r: oracle_sample_masked(w, gen, q, k, v, t, r)
    rng = np.random.default_rng(12345)
    per_step = max(0.5, min(4.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        sample(per_step / 4, rng)
    flops, secs, rows = 0.0, 0.0, 0
    for _ in range(args.steps):
        f, s, r = sample(per_step, rng)
        flops, secs, rows = flops + f, secs + s, rows + r
    value = flops / secs / 1e12
    cores = oracle.max_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": arm_config(args, w, gen, args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "%d random (head,row) rows of the workload, each step ~%.1f s of CPU work; "
                                   "flops counted 4*d per visible key" % (rows, per_step)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def step_input_bytes(w: sy.Workload, gen, backward: bool) -> int:
    """Bytes a timed step reads as input: q, k, v (backward: also o, dO and L)."""
    if gen is not None:
        fwd = gen["input_bytes"]
        rows_q = w.B * gen["seqlen_q"] * w.H
    else:
        fwd = 3 * w.B * w.H * w.N * w.d * 2
        rows_q = w.B * w.H * w.N
    return fwd + (rows_q * (2 * w.d * 2 + 4) if backward else 0)


def flush_l2(in_bytes: int, mode: str) -> bool:
    """Whether timed launches overwrite the L2 first: `mode` "on", or "auto"
    with step inputs that fit in the L2 (they would otherwise be read warm)."""
    return mode == "on" or (mode == "auto" and in_bytes <= L2_BYTES)


def l2_note(in_bytes: int, flush: bool) -> str:
    if flush:
        return ("inputs (%.0f MB) not larger than the 129 MB L2: L2 overwritten (a %.0f MB write) before each "
                "timed launch, launches timed one by one" % (in_bytes / 1e6, 2 * L2_BYTES / 1e6))
    return "inputs (%.0f MB) larger than the 129 MB L2; no flush" % (in_bytes / 1e6)


def workload_config(w: sy.Workload, n_gpus: int, gen=None, l2: str = "", launch: str = ""):
    c = {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
         "dtype": "bf16" if w.dtype == sy.BF16 else "fp16", "causal": w.causal,
         "scale": "1/sqrt(d)", "q_scale": w.q_scale,
         "l2": l2 or l2_note(step_input_bytes(w, gen, False), False),
         "parallelism": "replicas x%d" % n_gpus, "seed": w.seed(0)}
    if launch:
        c["launch"] = launch
    if gen is not None:
        c["workload"] = w.name + " " + gen["label"]
        c["causal"] = None
        c["mask"] = {k: gen[k] for k in ("window_left", "window_right", "prefix", "seqlen_k", "layout", "varlen_seqs")}
    return c


def arm_config(args, w: sy.Workload, gen, n_gpus: int):
    """The line's `config`, the same for both arms: the workload, the L2
    handling and the launch mode the kernel arm times with."""
    in_bytes = step_input_bytes(w, gen, args.backward)
    flush = flush_l2(in_bytes, args.flush_l2)
    return workload_config(w, n_gpus, gen, l2_note(in_bytes, flush), launch_mode(args.no_graph or flush))


def general_mask(args, w: sy.Workload):
    """The general-forward options as one dict, or None when none is given."""
    if (args.window_left is None and args.window_right is None and args.prefix == 0 and args.seqlen_k == 0
            and args.layout == "bhnd" and args.varlen_seqs == 0 and args.decode_rows == 0):
        return None
    if args.decode_rows and (args.varlen_seqs or args.seqlen_k or args.layout != "bhnd"):
        raise SystemExit("--decode-rows takes the workload's N as the key count; no --varlen-seqs/--seqlen-k/--layout")
    wl = -1 if args.window_left is None else args.window_left
    wr = (0 if w.causal else -1) if args.window_right is None else args.window_right
    nk = args.seqlen_k or w.N
    nq = args.decode_rows or w.N
    if args.varlen_seqs and args.seqlen_k:
        raise SystemExit("--varlen-seqs packs self-attention sequences (N_k = N_q); drop --seqlen-k")
    label = "window(%d,%d)" % (wl, wr)
    if args.prefix:
        label += " prefix%d" % args.prefix
    if nk != w.N:
        label += " Nk%d" % nk
    if args.layout != "bhnd":
        label += " " + args.layout
    if args.varlen_seqs:
        label += " varlen%d" % args.varlen_seqs
    if args.decode_rows:
        label = "decode %d row%s vs %d keys " % (nq, "s" if nq > 1 else "", nk) + label
    rows_q = w.B * nq    # per head
    # K and V rows a pass must read: the keys some query row sees (a bounded
    # window reads only its band); packed sequences count every key
    kv_rows = w.B * (nk if args.varlen_seqs else sy.union_visible_keys(nq, nk, wl, wr, args.prefix))
    inputs = (rows_q + 2 * kv_rows) * w.H * w.d * 2
    return {"window_left": wl, "window_right": wr, "prefix": args.prefix, "seqlen_k": nk, "layout": args.layout,
            "varlen_seqs": args.varlen_seqs, "decode_rows": args.decode_rows, "seqlen_q": nq, "label": label,
            "input_bytes": inputs,
            "bytes": inputs + rows_q * w.H * (w.d * 2 + 4)}


def backward_step(fa2, torch, w: sy.Workload, forward_step, q, k, v, o, lse, stream, **opts):
    """Run the forward once, then return the timed fa2_bwd_ex call for a seeded dout of o's layout."""
    import ctypes

    with torch.cuda.stream(stream):
        forward_step()
    stream.synchronize()
    g = torch.Generator(device="cpu").manual_seed(w.seed(0) + 500)
    dout = torch.empty_strided(o.shape, o.stride(), dtype=o.dtype, device=o.device)
    dout.copy_(torch.randn(o.shape, generator=g).to(o.dtype))
    like = lambda t: torch.empty_strided(t.shape, t.stride(), dtype=t.dtype, device=t.device)
    dq, dk, dv = like(q), like(k), like(v)
    p, _, _ = fa2._general_params(q, k, v, o, lse, w.scale, opts.get("window_left", -1), opts.get("window_right", -1),
                                  opts.get("prefix_len", 0), opts.get("cu_seqlens_q"), opts.get("cu_seqlens_k"),
                                  opts.get("max_seqlen_q"), opts.get("max_seqlen_k"))
    need = int(fa2.load_library().fa2_bwd_ex_workspace_bytes(ctypes.byref(p)))
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)

    def step():
        fa2.fa2_bwd_ex(q, k, v, o, lse, dout, dq, dk, dv, workspace=ws, scale=w.scale, stream=stream, **opts)
    return step


def varlen_lengths(total: int, seqs: int, seed: int) -> np.ndarray:
    """Seeded random sequence lengths (each >= 1) summing to total."""
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, total), size=seqs - 1, replace=False))
    return np.diff(np.concatenate([[0], cuts, [total]])).astype(np.int64)


def general_step(fa2, torch, w: sy.Workload, gen, dev, tdt, stream, backward=False):
    """Inputs, the timed call (fa2_fwd_ex / fa2_decode, or fa2_bwd_ex after one forward) and
    its algorithmic FLOPs (the backward: 2.5x the forward's) for the general options."""
    wl, wr, pre = gen["window_left"], gen["window_right"], gen["prefix"]
    to_dev = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(tdt).to(dev)
    if gen["varlen_seqs"]:
        T = w.B * w.N
        lens = varlen_lengths(T, gen["varlen_seqs"], w.seed(0) + 7)
        q_bits, k_bits, v_bits = sy.make_qkv(1, w.H, T, w.d, w.dtype, w.seed(0), w.q_scale)
        q, k, v = (to_dev(x[0].transpose(1, 0, 2)) for x in (q_bits, k_bits, v_bits))   # [T, H, d]
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev)
        o = torch.empty_like(q)
        lse = torch.empty((w.H, T), dtype=torch.float32, device=dev)
        vis = sum(int(sy.visible_keys(int(n), int(n), wl, wr, pre).sum()) for n in lens)
        maxlen = int(lens.max())
        gen["lengths"] = "min %d / median %d / max %d" % (lens.min(), int(np.median(lens)), maxlen)

        def step():
            fa2.fa2_fwd_ex(q, k, v, o, lse, scale=w.scale, window_left=wl, window_right=wr, prefix_len=pre,
                           cu_seqlens_q=cu, cu_seqlens_k=cu, max_seqlen_q=maxlen, stream=stream)
        flops = 4.0 * w.d * w.H * vis
        if backward:
            step = backward_step(fa2, torch, w, step, q, k, v, o, lse, stream, window_left=wl, window_right=wr,
                                 prefix_len=pre, cu_seqlens_q=cu, cu_seqlens_k=cu, max_seqlen_q=maxlen,
                                 max_seqlen_k=maxlen)
            flops *= 2.5
        return step, flops, None, None, None
    nk = gen["seqlen_k"]
    if gen["decode_rows"]:
        nq = gen["seqlen_q"]
        q_bits = sy.make_qkv(w.B, w.H, nq, w.d, w.dtype, w.seed(0), w.q_scale)[0]
        _, k_bits, v_bits = sy.make_qkv(w.B, w.H, nk, w.d, w.dtype, w.seed(0) + 1)
        q, k, v = (to_dev(x) for x in (q_bits, k_bits, v_bits))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, nq), dtype=torch.float32, device=dev)
        ws = torch.empty(fa2.fa2_decode_workspace_bytes(q, k, v, window_left=wl, window_right=wr, prefix_len=pre),
                         dtype=torch.uint8, device=dev)

        def step():
            fa2.fa2_decode(q, k, v, o, lse, workspace=ws, scale=w.scale, window_left=wl, window_right=wr,
                           prefix_len=pre, stream=stream)
        flops = 4.0 * w.d * w.B * w.H * float(sy.visible_keys(nq, nk, wl, wr, pre).sum())
        return step, flops, q_bits, k_bits, v_bits
    q_bits = sy.make_qkv(w.B, w.H, w.N, w.d, w.dtype, w.seed(0), w.q_scale)[0]
    _, k_bits, v_bits = sy.make_qkv(w.B, w.H, nk, w.d, w.dtype, w.seed(0) + 1)
    if gen["layout"] == "bnhd":   # [B, N, H, d] storage, passed as [B, H, N, d] views
        q, k, v = (to_dev(x.transpose(0, 2, 1, 3)).transpose(1, 2) for x in (q_bits, k_bits, v_bits))
        o = torch.empty((w.B, w.N, w.H, w.d), dtype=tdt, device=dev).transpose(1, 2)
    else:
        q, k, v = (to_dev(x) for x in (q_bits, k_bits, v_bits))
        o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)

    def step():
        fa2.fa2_fwd_ex(q, k, v, o, lse, scale=w.scale, window_left=wl, window_right=wr, prefix_len=pre,
                       stream=stream)
    flops = 4.0 * w.d * w.B * w.H * float(sy.visible_keys(w.N, nk, wl, wr, pre).sum())
    if backward:
        step = backward_step(fa2, torch, w, step, q, k, v, o, lse, stream, window_left=wl, window_right=wr,
                             prefix_len=pre)
        flops *= 2.5
    return step, flops, q_bits, k_bits, v_bits


def launch_mode(no_graph: bool) -> str:
    return "one CUDA graph replaying the timed launches" if not no_graph else "one launch per step from Python"


MIN_TIMED_S = 1.0       # device time the repeated K-step regions add up to, at least
MAX_REGIONS = 2000


def region_count(first_region_ms: float, min_total_s: float = MIN_TIMED_S, cap: int = MAX_REGIONS) -> int:
    """How many K-step regions to time so that they add up to min_total_s of
    device time (at least 3, at most `cap`), given the first region's time."""
    if first_region_ms <= 0:
        return cap
    n = int(np.ceil(min_total_s * 1e3 / first_region_ms))
    return max(3, min(cap, n))


def spread(region_ms):
    """Median and spread of the timed regions (each exactly K steps), in the
    order they ran."""
    first = float(region_ms[0])
    a = np.sort(np.asarray(region_ms, dtype=np.float64))
    med = float(np.median(a))
    p10, p90 = (float(x) for x in np.percentile(a, [10, 90]))
    return {"regions": int(a.size), "median_ms": med, "first_ms": first, "min_ms": float(a[0]), "max_ms": float(a[-1]),
            "p10_ms": p10, "p90_ms": p90, "spread_pct": 100.0 * (p90 - p10) / med if med > 0 else None,
            "total_s": float(a.sum()) / 1e3}


def time_regions(torch, step, stream, steps: int, flush_buf, graph, first_only: bool = False,
                 min_total_s: float = MIN_TIMED_S):
    """Time K-step regions on `stream` with CUDA events: one region, or (the
    default) as many as region_count asks for.  A graph replays the K launches
    (region time = its events); without one, each launch has its own events
    and, with a flush buffer, the L2 is overwritten before it, outside them
    (region time = the sum of the K launch times).  Returns (region times in
    ms, per-launch ms of every region)."""
    def one():
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            if graph is None:
                # launched one by one: keep the GPU busy while the host enqueues
                # them, so no launch waits on the host inside its own events
                torch.cuda._sleep(int(4e5 * steps))
            t0.record(stream)
            if graph is not None:
                graph.replay()
            else:
                for i in range(steps):
                    if flush_buf is not None:
                        flush_buf.zero_()
                    starts[i].record(stream)
                    step()
                    ends[i].record(stream)
            t1.record(stream)
        stream.synchronize()
        if graph is not None:
            ms = t0.elapsed_time(t1)
            return ms, [ms / steps] * steps
        per = [a.elapsed_time(b) for a, b in zip(starts, ends)]
        # with a flush, the overwrites between launches are not the workload's time
        return (sum(per) if flush_buf is not None else t0.elapsed_time(t1)), per
    first, per = one()
    regions, launches = [first], list(per)
    if not first_only:
        for _ in range(region_count(first, min_total_s) - 1):
            ms, per = one()
            regions.append(ms)
            launches += per
    return regions, launches


def build_parser() -> argparse.ArgumentParser:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, choices=sorted(sy.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="bounded CPU-oracle sample (s)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--heads", type=int, default=0,
                    help="override H (a smaller case of the same kernel, e.g. for an ncu capture)")
    ap.add_argument("--kernel-only", action="store_true", help="skip the end-to-end and CPU-baseline legs")
    ap.add_argument("--min-seconds", type=float, default=MIN_TIMED_S,
                    help="repeat the K-step region until the regions add up to this much device time "
                         "(at least 3 regions; 0 for a profiler run)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the timed steps one by one instead of replaying them from a CUDA graph")
    ap.add_argument("--flush-l2", choices=["auto", "on", "off"], default="auto",
                    help="overwrite the L2 before each timed launch (auto: when the inputs fit in it)")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (fa2_bwd) instead: 2.5x the forward FLOPs (five products)")
    g = ap.add_argument_group("general forward (fa2_fwd_ex); FLOPs then count 4*d per visible (query, key) pair")
    g.add_argument("--window-left", type=int, default=None, help="keys before the aligned one (-1: unbounded)")
    g.add_argument("--window-right", type=int, default=None,
                   help="keys after the aligned one (-1: unbounded; default 0 if the workload is causal)")
    g.add_argument("--prefix", type=int, default=0, help="keys every query sees (prefix-LM)")
    g.add_argument("--seqlen-k", type=int, default=0, help="N_k (default N); queries face the last N keys")
    g.add_argument("--layout", choices=["bhnd", "bnhd"], default="bhnd", help="storage order of q, k, v, o")
    g.add_argument("--varlen-seqs", type=int, default=0,
                   help="pack the B*N query tokens as this many sequences of seeded random lengths")
    g.add_argument("--decode-rows", type=int, default=0,
                   help="time fa2_decode: this many query rows (<= 8) per (b, h) against the workload's N keys")
    return ap


def main():
    ap = build_parser()
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = sy.WORKLOADS[args.workload]
    if args.heads > 0:
        w = sy.Workload(w.index, w.B, args.heads, w.N, w.d, w.dtype, w.causal, w.q_scale)
    gen = general_mask(args, w)
    if gen is not None and args.backward and gen["decode_rows"]:
        ap.error("--decode-rows times the forward pass only")
    if args.impl == "reference":
        return run_reference(args, w, gen)

    import torch

    import exact_tiled_attention_fa2_gb300 as fa2
    from exact_tiled_attention_fa2_gb300 import build as fa2_build

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    fa2_build.build() if rank == 0 else None
    if dist is not None:
        dist.barrier()
    fa2.load_library()

    q_bits, k_bits, v_bits = w.inputs()
    tdt = torch.bfloat16 if w.dtype == sy.BF16 else torch.float16
    host = [torch.from_numpy(x.view(np.int16)).view(tdt) for x in (q_bits, k_bits, v_bits)]
    dev = torch.device("cuda", local)
    q, k, v = (h.to(dev) for h in host)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)

    def step():
        fa2.fa2_fwd(q, k, v, o, lse, scale=w.scale, causal=w.causal, stream=stream)

    flops = w.flops() * (2.5 if args.backward else 1.0)
    if gen is not None:
        step, flops, q_bits, k_bits, v_bits = general_step(fa2, torch, w, gen, dev, tdt, stream, args.backward)

    if args.backward and gen is None:
        with torch.cuda.stream(stream):
            step()
        stream.synchronize()
        dout = torch.from_numpy(sy.make_qkv(w.B, w.H, w.N, w.d, w.dtype, w.seed(0) + 500)[0].view(np.int16)).view(
            tdt).to(dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
        bws = torch.empty(fa2.fa2_bwd_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8, device=dev)

        def step():  # noqa: F811 -- the backward pass replaces the forward as the timed step
            fa2.fa2_bwd(q, k, v, o, lse, dout, dq, dk, dv, bws, scale=w.scale, causal=w.causal, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    code, detail = fa2.fa2_get_device_status(stream)
    if code != fa2.FA2_OK:
        raise RuntimeError("device status %d (0x%x) after warm-up" % (code, detail))

    # inputs that fit in the L2 would be timed warm: overwrite the L2 before
    # every timed launch instead, outside the launch's own timing events
    in_bytes = step_input_bytes(w, gen, args.backward)
    flush = flush_l2(in_bytes, args.flush_l2)
    fbuf = None
    no_graph = args.no_graph or flush
    if flush:
        fbuf = torch.empty(int(2 * L2_BYTES), dtype=torch.uint8, device=dev)

    def capture():
        # K launches captured once and replayed: a region then holds exactly
        # the K kernels, without host launch gaps between them
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(args.steps):
                step()
        stream.synchronize()
        return g
    graph = None if no_graph else capture()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    # K-step regions, repeated until they add up to >= 1 s of device time;
    # the line reports the median region (every region is exactly K steps)
    with ClockSampler(local) as clocks:
        regions, kernel_ms = time_regions(torch, step, stream, args.steps, fbuf, graph, min_total_s=args.min_seconds)
    torch.cuda.synchronize(dev)
    timing = spread(regions)
    elapsed_ms = timing["median_ms"]
    code, detail = fa2.fa2_get_device_status(stream)
    if code != fa2.FA2_OK:
        raise RuntimeError("device status %d (0x%x) in timed region" % (code, detail))
    max_ms = max_over_ranks(elapsed_ms, dist, dev)
    if dist is not None:
        dist.barrier()
    unflushed = None
    if flush and rank == 0:
        # the same launches back to back from a CUDA graph, L2 not overwritten
        g2 = capture()
        r2, _ = time_regions(torch, step, stream, args.steps, None, g2, min_total_s=args.min_seconds)
        unflushed = spread(r2)
        del g2

    value = job_throughput(flops, args.steps, ws, max_ms)
    avg_launch_ms = max_ms / args.steps   # the median region's K launches (flushed: their own events)
    achieved = flops / (avg_launch_ms / 1e3) / 1e12
    # the timed loop runs >= 1 s back to back, long enough for the power cap
    # to set the clocks: the sustained peak is its denominator; the first
    # region (before the cap engages) is reported against the burst peak
    peak, peak_note = measured_peak(sustained=True)
    burst_peak, burst_note = measured_peak(sustained=False)
    first_achieved = flops * args.steps / (timing["first_ms"] / 1e3) / 1e12

    e2e = None
    cpu = None
    if rank == 0 and not args.kernel_only and gen is not None and ws == 1 and not args.no_cpu_baseline \
            and q_bits is not None:
        import oracle

        f, s, rows = oracle_sample_masked(w, gen, q_bits, k_bits, v_bits, args.cpu_seconds,
                                          np.random.default_rng(7))
        cpu = {"value": f / s / 1e12, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
               "sample": "%d random (head,row) rows of the workload in %.1f s (fp64 oracle, OpenMP); "
                         "flops counted 4*d per visible key" % (rows, s)}
    if rank == 0 and not args.kernel_only and not args.backward and gen is None:
        # end to end through the host-buffer entry point: H2D of q, k, v and D2H of o, lse each step
        qh, kh, vh = (h.pin_memory() for h in host)
        oh = torch.empty(q.shape, dtype=tdt).pin_memory()
        lh = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        wsb = torch.empty(fa2.fa2_fwd_host_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8, device=dev)
        fa2.fa2_fwd_host(qh, kh, vh, oh, lh, wsb, scale=w.scale, causal=w.causal, stream=stream)
        te = time.perf_counter()
        for _ in range(args.e2e_steps):
            fa2.fa2_fwd_host(qh, kh, vh, oh, lh, wsb, scale=w.scale, causal=w.causal, stream=stream)
        e2e_s = time.perf_counter() - te
        tb = w.B * w.H * w.N * w.d * 2
        e2e = {"value": flops * args.e2e_steps / e2e_s / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": 3 * tb, "d2h_bytes_per_step": tb + w.B * w.H * w.N * 4,
               "steps": args.e2e_steps, "ms_per_step": 1e3 * e2e_s / args.e2e_steps,
               "api": "fa2_fwd_host (pinned host buffers)"}
        del wsb
        if ws == 1 and not args.no_cpu_baseline:
            import oracle

            f, s, rows = oracle_sample(w, q_bits, k_bits, v_bits, args.cpu_seconds, np.random.default_rng(7))
            cpu = {"value": f / s / 1e12, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
                   "sample": "%d random (head,row) rows of the workload in %.1f s (fp64 oracle, OpenMP); "
                             "flops counted 4*d per visible key" % (rows, s)}

    if rank == 0:
        clk = clocks.summary()
        kname = ({64: "fa2_bwd64_kernel", 256: "fa2_bwd256_kernel"}.get(w.d, "fa2_bwd_kernel") if args.backward
                 else "fa2_fwd_dbuf_kernel")
        line = {
            "metric": METRIC if not args.backward else
            "backward attention TFLOP/s at 1 GB300 (2.5x the forward FLOPs) and % of dense FP16/BF16 tensor peak",
            "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": max_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == sy.BF16 else "fp16",
            "data": "synthetic",
            "config": arm_config(args, w, gen, ws),
            "timing": dict(timing, steps_per_region=args.steps,
                           rule="median over regions of exactly K steps, each bracketed by a synchronize and "
                                "timed with CUDA events on the launching stream; regions repeated until they add "
                                "up to >= %g s of device time; value = max over ranks of the median" % args.min_seconds),
            "pct_of_peak": 100.0 * value / ws / peak,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                         "frac": achieved / peak,
                         "traffic": recorded_traffic(args.workload, kname) if gen is None else None,
                         "peak_source": peak_note, "kernel": kname,
                         "first_region": {"achieved": first_achieved, "peak": burst_peak, "frac": first_achieved / burst_peak,
                                          "peak_source": burst_note},
                         "avg_launch_ms": avg_launch_ms,
                         "algorithmic_flops_per_launch": flops,
                         "algorithmic_bytes_per_launch": (w.algorithmic_bytes() if gen is None else gen["bytes"]) *
                                                         (2 if args.backward else 1)},
            "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                       "samples": clk["samples"]},
            "e2e": e2e, "cpu_baseline": cpu, "gpu_launches": args.steps * (3 if args.backward else 1),
            "kernel_sha": kernel_source_hash(BWD_SOURCES.get(kname, KERNEL_SOURCES)),
        }
        # the memory side of the roofline: algorithmic bytes per launch over the launch time
        hbm, hbm_note = measured_hbm()
        alg_bytes = line["roofline"]["algorithmic_bytes_per_launch"]
        gbs = alg_bytes / (avg_launch_ms / 1e3) / 1e9
        line["hbm"] = {"achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm, "peak_source": hbm_note,
                       "bytes_per_launch": alg_bytes}
        if unflushed is not None:
            line["latency"] = {"flushed_us_per_launch": 1e3 * avg_launch_ms,
                               "unflushed_us_per_launch": 1e3 * unflushed["median_ms"] / args.steps,
                               "unflushed_gbs": alg_bytes / (unflushed["median_ms"] / args.steps / 1e3) / 1e9,
                               "unflushed_regions": unflushed["regions"],
                               "note": "flushed: L2 overwritten before each launch (the value above); unflushed: "
                                       "the same launches back to back from a CUDA graph"}
        ridge = peak * 1e12 / (hbm * 1e9)   # FLOP per byte where the two measured peaks meet
        if gen is None and not args.backward and w.flops() / w.algorithmic_bytes() < ridge:
            # below the ridge point (the tiny single-tile workload): the memory side bounds the roofline
            line["roofline"] = dict(line["hbm"], bound="hbm", kernel=kname, avg_launch_ms=avg_launch_ms,
                                    algorithmic_bytes_per_launch=alg_bytes, algorithmic_flops_per_launch=flops,
                                    traffic=None)
        if gen is not None and gen["decode_rows"]:
            # HBM-bound: K and V read once dominate; roofline against the measured copy bandwidth
            hbm, hbm_note = measured_hbm()
            gbs = gen["bytes"] / (avg_launch_ms / 1e3) / 1e9
            line["roofline"] = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                                "traffic": None, "peak_source": hbm_note,
                                "kernel": ("fa2_fwd_dbuf_kernel (split-key mode)"
                                           if w.d == 128 or (w.d == 64 and gen["decode_rows"] >= 2)
                                           else "fa2_decode_kernel") + " + fa2_decode_merge_kernel",
                                "avg_launch_ms": avg_launch_ms, "algorithmic_bytes_per_launch": gen["bytes"],
                                "algorithmic_flops_per_launch": flops}
            line["gpu_launches"] = 2 * args.steps
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
