"""Benchmark of the HSTU fused attention forward on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

One step = one forward (work-list build + tensor-core kernel) over one batch of
the workload: by default bf16, causal, batch 32, jagged lengths U[256, 2048]
(max_seqlen 2048), 4 heads, head_dim 128, no rab. The metric is mask-aware useful
TFLOP/s = 4 * D * (valid (head, i, j) pairs) / time. Inputs are resident in HBM;
the timed steps rotate through input sets whose total exceeds L2 so no step
reads its inputs from the previous step's L2. Prints one JSON line (rank 0).

With N > 1 (torchrun) every rank runs its own full replica of the workload (the
forward has no exchange step); value = all ranks' work / max time over ranks.

--impl reference times the fp64 CPU oracle on the host cores over a bounded
sample of the same workload (the only reference this operator has).
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

import torch  # noqa: E402

L2_BYTES = 129 * 1024 * 1024


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            m = json.load(f)
        return dict(bf16=float(m.get("bf16_tflops")), hbm=float(m.get("hbm_gbs")),
                    bf16_sustained=float(m.get("bf16_tflops_sustained", m.get("bf16_tflops"))),
                    source="measured")
    return dict(bf16=1900.0, hbm=6800.0, bf16_sustained=1700.0, source="fallback")


def kernel_sources_sha() -> str:
    """Short hash of the CUDA sources, to tell whether a stored ncu capture still
    describes the kernel being timed."""
    import glob
    import hashlib
    csrc = os.path.join(ROOT, "hstu_dense_forward_gb300", "csrc")
    srcs = sorted(glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "*.cuh")) +
                  glob.glob(os.path.join(csrc, "*.h")))
    h = hashlib.sha256()
    for src in srcs:
        h.update(os.path.basename(src).encode())
        with open(src, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def stored_traffic(workload: str):
    """DRAM bytes per launch of the forward kernel from the committed ncu summary, or
    None when that capture was taken on different kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(workload)
    if not rec or rec.get("kernel_sources_sha256_16") != kernel_sources_sha():
        return None
    return rec.get("dram_bytes_per_launch")


def reduce_over_ranks(ms: float, ws: int, dev=None) -> float:
    """Max of a per-rank time over all ranks (identity with one rank)."""
    if ws == 1:
        return ms
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(flops_per_step: float, steps: int, ws: int, max_ms: float) -> float:
    """Whole-job throughput in TFLOP/s: every rank ran `steps` steps of its replica."""
    return flops_per_step * steps * ws / (max_ms * 1e-3) / 1e12


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def __enter__(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        if self.proc is None or self.tmp is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.tmp.flush()
        with open(self.tmp.name) as f:
            rows = [r.strip().split(", ") for r in f if r.strip()]
        os.unlink(self.tmp.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def _workload(name):
    from hstu_dense_forward_gb300 import workloads as W
    return W.WORKLOADS[name] if name in W.WORKLOADS else W.KV_WORKLOADS[name]


def _is_kv(w):
    from hstu_dense_forward_gb300 import workloads as W
    return isinstance(w, W.KVWorkload)


# The headline metric: mask-aware useful TFLOP/s (4 * D per valid pair) and its share of the
# bf16 peak, or HBM GB/s for the bandwidth-bound workloads; the time of one call.
METRIC = "HSTU fwd mask-aware TFLOPS & % of GB300 BF16 peak (rab: HBM GB/s); ms/call"

KV_KEYS = ("seq_offsets_k", "kv_cache", "page_offsets", "page_ids", "last_page_len")


def _generate(w):
    from hstu_dense_forward_gb300 import workloads as W
    return W.generate_kv(w) if _is_kv(w) else W.generate(w)


def _pairs(w, inp):
    from hstu_dense_forward_gb300 import count_pairs, count_pairs_kv
    if _is_kv(w):
        return count_pairs_kv(inp["seq_offsets"], w.num_heads_q, max_seqlen=w.max_seqlen,
                              seq_offsets_k=inp["seq_offsets_k"],
                              page_offsets=inp["page_offsets"],
                              last_page_len=inp["last_page_len"], page_size=w.page_size,
                              max_seqlen_k=w.max_seqlen_k, num_context=inp["num_context"],
                              num_targets=inp["num_targets"], causal=w.causal,
                              target_group_size=w.target_group_size)
    return count_pairs(inp["seq_offsets"], w.num_heads_q, max_seqlen=w.max_seqlen,
                       num_context=inp["num_context"], num_targets=inp["num_targets"],
                       causal=w.causal, target_group_size=w.target_group_size)


def _kv_sample(inp, nb):
    """The first nb sequences of a key-side workload as oracle arguments, with a cache
    holding only their pages (renumbered in order)."""
    so, so_k = inp["seq_offsets"].to(torch.int64), inp["seq_offsets_k"].to(torch.int64)
    args = dict(seq_offsets_k=so_k[:nb + 1])
    if inp["kv_cache"] is not None:
        po = inp["page_offsets"].to(torch.int64)
        used = inp["page_ids"][:int(po[nb])].to(torch.int64)
        args.update(kv_cache=inp["kv_cache"][used], page_offsets=po[:nb + 1],
                    page_ids=torch.arange(used.numel()), last_page_len=inp["last_page_len"][:nb])
    return (inp["q"][:int(so[nb])], inp["k"][:int(so_k[nb])], inp["v"][:int(so_k[nb])],
            so[:nb + 1], args)


def _algorithmic_bytes_kv(w, inp):
    """Key-side workload: Q read and O written once; per key/value head, every key of a
    sequence (cached history rows and new rows) read once as K and once as V."""
    el = torch.finfo(W_dtype(w)).bits // 8
    out_el = 2 if w.dtype == "fp8" else el  # FP8 inputs give bf16 out
    tq = int(inp["seq_offsets"][-1])
    keys = int((inp["seq_offsets_k"][1:] - inp["seq_offsets_k"][:-1]).sum() + inp["history"].sum())
    return (tq * w.num_heads_q * (el + out_el) + 2 * keys * w.num_heads_kv * el) * w.head_dim


def W_dtype(w):
    from hstu_dense_forward_gb300 import workloads as W
    return W.DTYPES[w.dtype]


def _algorithmic_bytes(w, inp, pairs_per_head):
    """Q, K, V read once, O written once, rab entries at valid pairs (2 bytes each)."""
    el = torch.finfo(w.torch_dtype).bits // 8
    T = int(inp["seq_offsets"][-1])
    qo = 2 * T * w.num_heads_q * w.head_dim * el
    kv = 2 * T * w.num_heads_kv * w.head_dim * el
    rab = pairs_per_head * el if w.rab else 0
    return qo + kv + rab


def time_windows(step, sets, steps, min_windows=10, min_seconds=1.0, stream=None):
    """Per-step milliseconds of repeated timed windows: each window is `steps` calls (inputs
    rotating over `sets`) between CUDA events on the launching stream, with a synchronize
    on both sides; windows repeat until at least `min_windows` ran and `min_seconds` of
    calls were timed."""
    out = []
    total = 0.0
    i = 0
    while len(out) < min_windows or total < min_seconds:
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step(sets[i % len(sets)])
            i += 1
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        out.append(ms / steps)
        total += ms * 1e-3
    return out


def _input_sets(w, inp, dev, W, out_dtype):
    set_bytes = sum(t.numel() * t.element_size() for t in
                    (inp["q"], inp["k"], inp["v"], inp["rab"], inp.get("kv_cache"))
                    if t is not None) + inp["q"].numel() * inp["q"].element_size()  # + out
    nsets = max(3, -(-3 * L2_BYTES // max(set_bytes, 1)))
    nsets = min(nsets, 8)
    sets = []
    for _ in range(nsets):
        d = W.to_device(inp, dev)
        d["out"] = torch.empty(d["q"].shape, dtype=out_dtype(d["q"].dtype), device=dev)
        sets.append(d)
    return sets, set_bytes


def _step_fn(kv_side):
    from hstu_dense_forward_gb300 import hstu_fwd

    def step(d):
        kv = {k: d[k] for k in KV_KEYS} if kv_side else {}
        if kv_side:
            kv["max_seqlen_k"] = d["max_seqlen_k"]
        hstu_fwd(d["q"], d["k"], d["v"], d["seq_offsets"], max_seqlen=d["max_seqlen"],
                 rab=d["rab"], num_context=d["num_context"], num_targets=d["num_targets"],
                 causal=d["causal"], target_group_size=d["target_group_size"], alpha=d["alpha"],
                 silu_scale=d["silu_scale"], out=d["out"], **kv)
    return step


def _roofline(w, inp, pairs, flops, ms_per_step, peaks, traffic):
    """The dominant bound of a workload: tensor (TFLOP/s) for the contractions, HBM
    (algorithmic GB/s) for rab and for key sides read from a paged cache."""
    achieved = flops / (ms_per_step * 1e-3) / 1e12
    timed = "CUDA events around each call: work-list build + forward kernel"
    if w.dtype == "fp32":
        # the CUDA-core path (FFMA): reported against the bf16 tensor peak for scale only
        return {"bound": "latency", "achieved": round(achieved, 4), "peak": peaks["bf16"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16"], 6),
                "traffic": traffic, "peak_source": peaks["source"], "timed": timed,
                "note": "fp32 CUDA-core path on a 40-token input: launch-latency bound"}
    if _is_kv(w):
        gbs = _algorithmic_bytes_kv(w, inp) / (ms_per_step * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm"], "unit": "GB/s",
                "frac": round(gbs / peaks["hbm"], 4), "traffic": traffic,
                "algorithmic_bytes": _algorithmic_bytes_kv(w, inp),
                "peak_source": peaks["source"], "tensor_tflops": round(achieved, 2),
                "timed": timed}
    if w.rab:
        ab = _algorithmic_bytes(w, inp, pairs)
        gbs = ab / (ms_per_step * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm"], "unit": "GB/s",
                "frac": round(gbs / peaks["hbm"], 4), "frac_of_8tbs": round(gbs / 8000.0, 4),
                "traffic": traffic, "algorithmic_bytes": ab, "peak_source": peaks["source"],
                "tensor_tflops": round(achieved, 2), "timed": timed}
    # an FP8 contraction: the bf16 peak times the nominal dense fp8 / bf16 ratio (4.5 / 2.25)
    tpeak = peaks["bf16"] * (2.0 if w.dtype == "fp8" else 1.0)
    return {"bound": "tensor", "achieved": round(achieved, 2), "peak": tpeak, "unit": "TFLOP/s",
            "frac": round(achieved / tpeak, 4),
            "frac_of_sustained": round(achieved / (peaks["bf16_sustained"] *
                                                   (2.0 if w.dtype == "fp8" else 1.0)), 4),
            "traffic": traffic,
            "peak_source": peaks["source"] + (" x 2 (fp8 / bf16 nominal)" if w.dtype == "fp8"
                                              else ""),
            "timed": timed}


def measure(w, args, dev, ws, peaks, clocks=False):
    """Time one workload on this rank (inputs resident in HBM, rotating sets larger than
    L2): returns the per-step times of every window and the derived numbers."""
    from hstu_dense_forward_gb300 import out_dtype, useful_flops
    from hstu_dense_forward_gb300 import workloads as W

    kv_side = _is_kv(w)
    inp = _generate(w)
    pairs = _pairs(w, inp)
    flops = useful_flops(pairs, w.head_dim)
    sets, set_bytes = _input_sets(w, inp, dev, W, out_dtype)
    step = _step_fn(kv_side)
    stream = torch.cuda.current_stream(dev)
    for i in range(args.warmup):
        step(sets[i % len(sets)])
    torch.cuda.synchronize()
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    clk = ClockSampler(dev.index if dev.index is not None else 0) if clocks else None
    if clk:
        clk.__enter__()
    try:
        win = time_windows(step, sets, args.steps, args.windows, args.min_seconds, stream)
    finally:
        if clk:
            clk.__exit__(None, None, None)
    med = reduce_over_ranks(statistics.median(win), ws, dev)
    mn = reduce_over_ranks(min(win), ws, dev)
    traffic = args.traffic if (args.traffic is not None and w.name == args.workload) else \
        stored_traffic(w.name)
    return dict(w=w, inp=inp, pairs=pairs, flops=flops, sets=sets, set_bytes=set_bytes,
                step=step, windows=win, ms_median=med, ms_min=mn,
                value=flops * ws / (med * 1e-3) / 1e12,
                roofline=_roofline(w, inp, pairs, flops, med, peaks, traffic),
                clocks=clk.summary() if clk else None)


def _config(w, inp, m, ws):
    kv_side = _is_kv(w)
    return {"workload": w.name, "batch": w.batch, "max_seqlen": w.max_seqlen,
            "heads_q": w.num_heads_q, "heads_kv": w.num_heads_kv, "head_dim": w.head_dim,
            "mask": "causal" if w.causal else "none", "rab": w.rab,
            "tokens": int(inp["seq_offsets"][-1]),
            **({"keys": int((inp["seq_offsets_k"][1:] - inp["seq_offsets_k"][:-1]).sum()
                            + inp["history"].sum()),
                "cached_keys": int(inp["history"].sum()), "page_size": w.page_size,
                "max_seqlen_k": w.max_seqlen_k} if kv_side else {}),
            "valid_pairs": m["pairs"], "useful_gflop_per_step": round(m["flops"] / 1e9, 6),
            "l2": f"rotating {len(m['sets'])} input sets of {m['set_bytes'] / 2**20:.0f} MiB "
                  "(> L2)",
            "parallelism": f"replicas x{ws}"}


# Configurations timed in the same run next to the headline one (the other four
# configurations of the workload list, then the FP8, paged-cache and head-dim-512 ones):
# parity-test cases that also get a line of numbers.
EXTRA_WORKLOADS = ("fp32_tiny", "bf16_rab_b16_s1024_h8_d64", "fp16_gqa8x2_targets_b8_s4096_d128",
                   "bf16_long_b4_s8192_h4_d256", "fp8_causal_b32_s2048_h4_d128",
                   "bf16_paged_b128_hist1k_4k_h4_d128", "bf16_causal_b8_s2048_h4_d512")


def run_ours(args):
    import numpy as np  # noqa: F401

    from hstu_dense_forward_gb300 import build as B
    from hstu_dense_forward_gb300 import out_dtype
    from hstu_dense_forward_gb300 import workloads as W

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        B.build()
    if ws > 1:
        dist.barrier()
    peaks = _peaks()
    w = _workload(args.workload)
    kv_side = _is_kv(w)
    m = measure(w, args, dev, ws, peaks, clocks=True)
    inp, flops, step = m["inp"], m["flops"], m["step"]
    ms_per_step = m["ms_median"]
    value = m["value"]
    stream = torch.cuda.current_stream(dev)

    # end to end through the public API: pinned host inputs -> device -> forward -> host,
    # every step. The copies run on their own streams, double-buffered, so that the H2D
    # copy of step i+1 and the D2H copy of step i-1 overlap the forward of step i.
    host = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    in_keys = [k for k in ("q", "k", "v", "seq_offsets", "num_context", "num_targets", "rab")
               + (KV_KEYS if kv_side else ()) if host[k] is not None]
    bufs = []
    for _ in range(2):
        dq = W.to_device(inp, dev)
        dq["out"] = torch.empty(dq["q"].shape, dtype=out_dtype(dq["q"].dtype), device=dev)
        bufs.append(dq)
    outs_h = [torch.empty(inp["q"].shape, dtype=out_dtype(inp["q"].dtype)).pin_memory()
              for _ in range(2)]
    h2d = sum(host[k].numel() * host[k].element_size() for k in in_keys)
    d2h = outs_h[0].numel() * outs_h[0].element_size()
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    ev_in, ev_fwd, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    started = [False, False]

    def e2e_step(i):
        b = i % 2
        dq = bufs[b]
        with torch.cuda.stream(s_in):
            if started[b]:
                s_in.wait_event(ev_fwd[b])  # the forward that last read this input set
            for k in in_keys:
                dq[k].copy_(host[k], non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if started[b]:
            stream.wait_event(ev_out[b])  # the D2H copy that last read this output
        step(dq)
        ev_fwd[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_fwd[b])
            outs_h[b].copy_(dq["out"], non_blocking=True)
            ev_out[b].record(s_out)
        started[b] = True

    e2e_steps = max(3, min(args.steps, 50))
    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    s_out.wait_stream(stream)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_value = flops * ws / (e2e_ms * 1e-3) / 1e12
    del bufs, outs_h, host

    # the other configurations, one GPU only (their CPU baselines are rank 0's anyway)
    extra = {}
    if ws == 1 and not args.no_workloads:
        for name in EXTRA_WORKLOADS:
            if name == w.name:
                continue
            we = _workload(name)
            me = measure(we, args, dev, ws, peaks, clocks=True)
            extra[name] = {
                "value": round(me["value"], 4), "unit": "TFLOP/s",
                "ms_per_step": round(me["ms_median"], 5), "ms_per_step_min": round(me["ms_min"], 5),
                "windows": len(me["windows"]), "steps_per_window": args.steps,
                "dtype": we.dtype, "config": _config(we, me["inp"], me, ws),
                "roofline": me["roofline"], "clocks": me["clocks"],
                "cpu_baseline": None if args.no_cpu_baseline else
                cpu_baselines(we, me["inp"], args.cpu_seconds),
            }
            del me

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baselines(w, inp, args.cpu_seconds)
    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "ms_per_step_min": round(m["ms_min"], 5), "windows": len(m["windows"]),
            "value_statistic": f"median of {len(m['windows'])} timed windows of {args.steps} "
                               f"steps (min window: {flops * ws / (m['ms_min'] * 1e-3) / 1e12:.1f}"
                               " TFLOP/s)",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic (seeded; shapes and distributions of the workload)",
            "config": _config(w, inp, m, ws),
            "gpu_launches": 2 * args.steps * len(m["windows"]),
            "roofline": m["roofline"],
            "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                    "pipeline": "pinned H2D of step i+1 and D2H of step i-1 overlap step i"},
            "clocks": m["clocks"],
            "cpu_baseline": cpu,
            "workloads": extra,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def cpu_baselines(w, inp, seconds):
    """The oracle on all host cores (the reported baseline) with its single-thread time
    beside it, each on a bounded sample of the workload."""
    allc = cpu_baseline(w, inp, seconds)
    one = cpu_baseline(w, inp, seconds / 2, nthreads=1)
    allc["single_thread"] = {"value": one["value"], "cores": 1, "sample": one["sample"]}
    return allc


def cpu_baseline(w, inp, seconds, nthreads=None):
    """The fp64 oracle on the host cores over the first sequences of the workload
    (all heads, whole rows), grown until it takes about `seconds`; sequences too long for
    that budget are sampled by rows instead."""
    import oracle

    nthreads = nthreads or os.cpu_count() or 1
    so0 = inp["seq_offsets"].to(torch.int64)
    if not _is_kv(w) and w.batch > 0:
        # whole-sequence cost of sequence 0 at the oracle's rate (about 3 GFLOP/s per thread,
        # one thread per (sequence, head) unit)
        L0 = int(so0[1] - so0[0])
        est = (L0 * L0 * w.num_heads_q * w.head_dim * 4) / (3e9 * min(nthreads, w.num_heads_q))
        if est > seconds:
            return _cpu_rows_baseline(w, inp, seconds, nthreads)
    so = inp["seq_offsets"].to(torch.int64)
    nb = 1
    best = None
    while True:
        sub = so[: nb + 1]
        T = int(sub[-1])
        args = dict(rab=None if inp["rab"] is None else inp["rab"][:nb],
                    num_context=None if inp["num_context"] is None else inp["num_context"][:nb],
                    num_targets=None if inp["num_targets"] is None else inp["num_targets"][:nb],
                    mask_type=oracle.MASK_CAUSAL if w.causal else oracle.MASK_NONE,
                    target_group_size=w.target_group_size, alpha=w.alpha_value,
                    silu_scale=w.silu_scale_value,
                    max_seqlen=w.max_seqlen_k if _is_kv(w) else w.max_seqlen)
        q, k, v = inp["q"][:T], inp["k"][:T], inp["v"][:T]
        kv = {}
        if _is_kv(w):
            q, k, v, sub, kv = _kv_sample(inp, nb)
        t0 = time.perf_counter()
        oracle.hstu_fwd(q, k, v, sub, nthreads=nthreads, **args, **kv)
        dt = time.perf_counter() - t0
        if _is_kv(w):
            hist = inp["history"][:nb]
            lk = (kv["seq_offsets_k"][1:] - kv["seq_offsets_k"][:-1]) + hist
            pairs = oracle.count_valid_kv(sub[1:] - sub[:-1], lk, w.num_heads_q,
                                          num_context=args["num_context"],
                                          num_targets=args["num_targets"],
                                          mask_type=args["mask_type"],
                                          target_group_size=w.target_group_size)
        else:
            pairs = oracle.count_valid(sub, w.num_heads_q, num_context=args["num_context"],
                                       num_targets=args["num_targets"],
                                       mask_type=args["mask_type"],
                                       target_group_size=w.target_group_size)
        best = (nb, dt, pairs)
        if dt >= seconds / 4 or nb >= w.batch:
            break
        nb = min(w.batch, max(nb + 1, int(nb * min(8.0, (seconds / 4) / max(dt, 1e-3)))))
    nb, dt, pairs = best
    tflops = 4 * w.head_dim * pairs / dt / 1e12
    return {"value": tflops, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
            "sample": f"sequences 0..{nb - 1} of {w.batch} (all {w.num_heads_q} heads, whole "
                      f"rows), fp64, {dt:.2f} s"}


def _cpu_rows_baseline(w, inp, seconds, nthreads):
    """The oracle on output rows of the first sequence (row i with every key it sees, all
    heads in turn), for sequences too long to run whole within the time budget; the row
    count grows until the run takes about `seconds` / 4."""
    import numpy as np

    import oracle
    so = inp["seq_offsets"].to(torch.int64).numpy()
    L = int(so[1] - so[0])
    mt = oracle.MASK_CAUSAL if w.causal else oracle.MASK_NONE
    nc = 0 if inp["num_context"] is None else int(inp["num_context"][0])
    nt = 0 if inp["num_targets"] is None else int(inp["num_targets"][0])
    kw = dict(rab=inp["rab"], num_context=inp["num_context"], num_targets=inp["num_targets"],
              mask_type=mt, target_group_size=w.target_group_size, alpha=w.alpha_value,
              silu_scale=w.silu_scale_value, max_seqlen=w.max_seqlen)
    n = 4
    while True:
        idx = np.linspace(0, L - 1, n).astype(np.int64)
        rows = np.stack([np.zeros(n, np.int64), np.arange(n) % w.num_heads_q, idx], axis=1)
        t0 = time.perf_counter()
        oracle.hstu_fwd_rows(inp["q"], inp["k"], inp["v"], so, rows, nthreads=nthreads, **kw)
        dt = time.perf_counter() - t0
        if dt >= seconds / 4 or n >= 4096:
            break
        n = min(4096, max(n + 1, int(n * min(8.0, (seconds / 4) / max(dt, 1e-3)))))
    pairs = sum(sum(oracle.valid(int(i), j, L, mt, nc, nt, w.target_group_size)
                    for j in range(L)) if mt != oracle.MASK_NONE else L for i in idx)
    return {"value": 4 * w.head_dim * pairs / dt / 1e12, "unit": "TFLOP/s", "cores": nthreads,
            "kind": "oracle",
            "sample": f"{n} output rows of sequence 0 (L={L}, heads in turn, every key), fp64, "
                      f"{dt:.2f} s"}


def run_full_oracle(args):
    """The oracle over the whole workload once, on all host cores and (unless
    --skip-single-thread) on one thread: wall times for the results table."""
    import oracle

    oracle.build()
    w = _workload(args.workload)
    inp = _generate(w)
    kw = dict(rab=inp["rab"], num_context=inp["num_context"], num_targets=inp["num_targets"],
              mask_type=oracle.MASK_CAUSAL if w.causal else oracle.MASK_NONE,
              target_group_size=w.target_group_size, alpha=w.alpha_value,
              silu_scale=w.silu_scale_value,
              max_seqlen=w.max_seqlen_k if _is_kv(w) else w.max_seqlen)
    if _is_kv(w):
        kw.update({k: inp[k] for k in KV_KEYS})
    cores = os.cpu_count() or 1
    res = {"workload": w.name, "cores": cores, "pairs": _pairs(w, inp),
           "useful_gflop": 4 * w.head_dim * _pairs(w, inp) / 1e9}
    for n in ([cores] if args.skip_single_thread else [cores, 1]):
        t0 = time.perf_counter()
        oracle.hstu_fwd(inp["q"], inp["k"], inp["v"], inp["seq_offsets"], nthreads=n, **kw)
        res[f"oracle_seconds_{'all_cores' if n == cores else '1_thread'}"] = round(
            time.perf_counter() - t0, 3)
    print(json.dumps(res), flush=True)


def run_reference(args):
    """The fp64 CPU oracle as the reference arm: each step is one bounded sample."""
    import oracle
    from hstu_dense_forward_gb300 import workloads as W

    ws, rank, _ = _dist()
    if rank != 0:
        return
    if args.full_oracle:
        run_full_oracle(args)
        return
    oracle.build()
    w = _workload(args.workload)
    inp = _generate(w)
    nthreads = os.cpu_count() or 1
    so = inp["seq_offsets"].to(torch.int64)
    nb = 1  # one sequence, all heads, whole rows: a bounded sample per step
    sub = so[: nb + 1]
    T = int(sub[-1])
    kw = dict(rab=None if inp["rab"] is None else inp["rab"][:nb],
              num_context=None if inp["num_context"] is None else inp["num_context"][:nb],
              num_targets=None if inp["num_targets"] is None else inp["num_targets"][:nb],
              mask_type=oracle.MASK_CAUSAL if w.causal else oracle.MASK_NONE,
              target_group_size=w.target_group_size, alpha=w.alpha_value,
              silu_scale=w.silu_scale_value,
              max_seqlen=w.max_seqlen_k if _is_kv(w) else w.max_seqlen)
    q, k, v = inp["q"][:T], inp["k"][:T], inp["v"][:T]
    if _is_kv(w):
        q, k, v, sub, kv = _kv_sample(inp, nb)
        kw.update(kv)
        lk = (kv["seq_offsets_k"][1:] - kv["seq_offsets_k"][:-1]) + inp["history"][:nb]
        pairs = oracle.count_valid_kv(sub[1:] - sub[:-1], lk, w.num_heads_q,
                                      num_context=kw["num_context"],
                                      num_targets=kw["num_targets"], mask_type=kw["mask_type"],
                                      target_group_size=w.target_group_size)
    else:
        pairs = oracle.count_valid(sub, w.num_heads_q, num_context=kw["num_context"],
                                   num_targets=kw["num_targets"], mask_type=kw["mask_type"],
                                   target_group_size=w.target_group_size)
    for _ in range(args.warmup):
        oracle.hstu_fwd(q, k, v, sub, nthreads=nthreads, **kw)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.hstu_fwd(q, k, v, sub, nthreads=nthreads, **kw)
    dt = (time.perf_counter() - t0) / args.steps
    value = 4 * w.head_dim * pairs / dt / 1e12
    sample = f"sequence 0 of {w.batch} (L={T}, all {w.num_heads_q} heads, whole rows), fp64"
    line = {"impl": "reference",
            "metric": METRIC,
            "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; shapes and distributions of the workload)",
            "config": {"workload": w.name, "sample": sample},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nthreads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="bf16_causal_b32_s2048_h4_d128")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--windows", type=int, default=10,
                    help="timed windows of --steps calls (at least; see --min-seconds)")
    ap.add_argument("--min-seconds", type=float, default=0.5,
                    help="keep timing windows until this many seconds of calls ran")
    ap.add_argument("--full-oracle", action="store_true",
                    help="with --impl reference: the oracle over the whole workload, once")
    ap.add_argument("--skip-single-thread", action="store_true",
                    help="with --full-oracle: all host cores only")
    ap.add_argument("--no-workloads", action="store_true",
                    help="time the headline workload only (no 'workloads' object)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the forward kernel from an ncu capture")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
