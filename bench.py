#!/usr/bin/env python3
"""Benchmark of the DSA indexer hot path (store + score/top-k) on GB300.

One step = one pass of the whole path over one batch of a workload, for both
cache formats: the step's new index keys are stored (RMSNorm + RoPE +
quantise + paged write) and every query of the batch is scored against its
visible keys and reduced to its top-k.

The headline is the largest single-GPU workload, the 22528-token causal
prefill (the pages' out-of-memory case). The other four workloads (tiny
prefill, batched decode, needle, long decode) are measured the same way and
reported under "configs". Every workload carries its throughput with inputs
resident, the end-to-end figure through the C ABI from pinned host buffers,
the roofline of its scorer launches and the C++ oracle's CPU baseline; the
store kernel's roofline is measured on the long decode's 1.05M-token fill and
on the long prefill's 22528 tokens. Each workload also reports the fp4 cache
on its own ("fp4"), and the long prefill and the batched decode the options
past the pages' path ("variants": the Hadamard-rotated cache, cache-slot
output, and for the batched decode the top-2048 selection).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload all|NAME]
  python bench.py --impl reference ...   # the C++ oracle on a bounded sample

Prints one JSON line. `value` is key-scores/s (sum over queries of the keys
each query is scored against, both formats) over all GPUs; L2 is flushed
(256 MB write, then 256 MB read of another buffer) between timed steps,
outside the timed events. `e2e` copies
each step's inputs from pinned host memory and its top-k back inside the
timed region. `roofline` is for the bf16 scorer of the headline workload,
timed by the library's CUDA events on the launch stream.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "indexer queries/s and key-scores/s (bf16 & fp8) + % of HBM/TC roofline"
HEADLINE = "long_prefill"
WORKLOAD_NAMES = ["tiny_prefill", "batched_decode", "long_prefill", "needle", "long_decode"]
FMT_NAMES = {0: "bf16", 1: "fp8", 2: "fp4"}
TOKEN_BYTES = {0: 256, 1: 132, 2: 68}
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
CSRC = os.path.join(ROOT, "dsa_sparse_attention_store_gb300", "csrc")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_PER_BF16 = 2.0   # nominal dense fp8 / bf16 tensor rate (4.5 / 2.25 PFLOP/s)
DESC = {
    "tiny_prefill": "1 sequence x 1024 tokens, causal prefill, k=512",
    "batched_decode": "64 sequences x 1 query, context U[2048,16384], page_size 64, permuted pages, k=512",
    "long_prefill": "1 sequence x 22528 tokens, causal prefill, k=512",
    "needle": "1 sequence x 10498 tokens, causal prefill, 5 planted needles, k=512",
    "long_decode": "8 sequences x 131072 context, 256 appended + 8 queries per sequence, k=1024",
}


def max_over_ranks(vals, device):
    """Element-wise maximum over all ranks of a list of floats (the slowest
    rank's times); one all_reduce on the process group's backend."""
    import torch
    import torch.distributed as tdist
    t = torch.tensor([float(v) for v in vals], device=device, dtype=torch.float64)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def whole_job_rate(units_per_rank_step: float, steps: int, world: int, ms: float) -> float:
    """Units per second over the whole job: every rank does the same work per
    step (weak scaling), timed by the slowest rank."""
    return world * units_per_rank_step * steps / (ms / 1e3)


def scorer_algorithmic(wl, fmt: int):
    """(bytes, flops) one scorer launch must move / do for workload wl in
    cache format fmt: every visible key read once (256 B bf16, 132 B fp8,
    68 B fp4),
    the queries (16 KB each, bf16 or two e4m3 terms) and head weights, one
    4-byte page id per page, 8 bytes per output entry; 2 * 64 * 128 flops
    per (query, visible key) pair."""
    import numpy as np
    pages = sum((int(L) + 63) // 64 for L in wl.seq_lens)
    nbytes = (int(wl.seq_lens.astype(np.int64).sum()) * TOKEN_BYTES[fmt]
              + wl.Tq * 64 * 128 * 2 + wl.Tq * 64 * 4
              + pages * 4 + wl.Tq * wl.k * 8)
    return nbytes, wl.key_scores() * 2 * 64 * 128


def store_algorithmic(tokens: int, fmt: int) -> int:
    """Bytes one store launch must move for `tokens` tokens: the 256-byte raw
    key read, the 256 (bf16), 132 (fp8) or 68 (fp4) bytes written, and the token's
    position and sequence id (8 bytes). The RoPE table row (512 B) and the
    page id are not counted: they repeat across tokens and sequences."""
    return tokens * (256 + TOKEN_BYTES[fmt] + 8)


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="all", choices=["all"] + WORKLOAD_NAMES)
    ap.add_argument("--fmt", choices=["both", "bf16", "fp8"], default="both")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-store-roofline", action="store_true")
    ap.add_argument("--no-fp4", action="store_true", help="skip the fp4-cache figures")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the Hadamard / k=2048 / slot-output figures")
    ap.add_argument("--cpu-seconds", type=float, default=6.0, help="oracle seconds per workload")
    return ap.parse_args(argv)


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return FALLBACK_PEAKS, "fallback"


def source_hash(names) -> str:
    """Hash of kernel sources (comments and blank space removed, so that a
    comment edit does not invalidate a traffic capture; any code change
    does)."""
    import re
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(CSRC, name), encoding="utf-8") as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def scorer_hash() -> str:
    return source_hash(("scorer.cuh", "topk.cu", "topk_fp8.cu", "topk_fp4.cu", "ptx.cuh", "internal.cuh"))


def store_hash() -> str:
    return source_hash(("store.cu", "internal.cuh"))


def traffic_of(key: str, hsh: str):
    """DRAM bytes per launch from the committed ncu capture, while the
    kernel's code still hashes to the captured version (else None)."""
    try:
        with open(TRAFFIC_FILE) as fh:
            ent = json.load(fh).get(key)
        if ent and ent.get("source_hash") == hsh:
            return ent["dram_bytes_per_launch"]
    except (OSError, ValueError):
        pass
    return None


def workload_config(wl, name, fmts):
    return {
        "workload": f"{name}: {DESC[name]}",
        "formats": [FMT_NAMES[f] for f in fmts],
        "global_batch": wl.Tq,
        "sequences": wl.B,
        "tokens_stored_per_step": int(wl.new_pos.shape[0]),
        "key_scores_per_step": int(wl.key_scores() * len(fmts)),
        "k": wl.k,
        "causal": wl.causal,
        "l2": "flushed between timed steps (256 MB write, then 256 MB read of another buffer; outside the timed events)",
    }


def make_workload(name):
    from synth import inputs as I
    return I.WORKLOADS[name]()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu=timestamp,{self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is not None:
            time.sleep(0.25)
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [ln.strip().split(", ") for ln in self.f.read().splitlines() if ln.strip()]
        os.unlink(self.f.name)
        return self._summary(rows)

    @staticmethod
    def _summary(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[2]))
                mx.append(float(r[3]))
                for n, v in zip(names, r[6:10]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ our arm
def build_lib():
    from dsa_sparse_attention_store_gb300 import build as B
    B.build()


def roofline_entry(kind, avg_ms, nbytes, flops, fmt, peaks, peak_src, traffic, launches):
    """The binding roofline of one kernel: HBM bytes or tensor flops, which
    ever needs more time at its peak. The fp8 scorer's contraction is
    e4m3 x e4m3 (two query terms per key), and so is the fp4 scorer's (its
    keys widened to e4m3 on chip), so their tensor peak is the fp8 one: the
    measured bf16 peak times the nominal fp8/bf16 ratio."""
    e8 = fmt in (1, 2)
    hbm = nbytes / (avg_ms / 1e3) / 1e9
    out = {"kernel": kind, "algorithmic_bytes_per_launch": nbytes, "avg_launch_ms": avg_ms,
           "launches": launches, "traffic": traffic}
    if flops:
        tc = flops / (avg_ms / 1e3) / 1e12
        tpk = peaks["bf16_tflops"] * (FP8_PER_BF16 if e8 else 1.0)
        tpk_s = peaks.get("bf16_tflops_sustained", tpk) * (FP8_PER_BF16 if e8 else 1.0)
        out["algorithmic_flops_per_launch"] = flops
        if e8:
            out["executed_tensor_flops_per_launch"] = 2 * flops
        if tc / tpk > hbm / peaks["hbm_gbs"]:
            dt = "fp8 (e4m3; measured bf16 x nominal 2)" if e8 else "bf16"
            out.update({"bound": "tensor", "achieved": tc, "peak": tpk, "unit": "TFLOP/s", "frac": tc / tpk,
                        "frac_of_sustained_peak": tc / tpk_s,
                        "peak_source": f"{peak_src} dense {dt} burst"})
            return out
    out.update({"bound": "hbm", "achieved": hbm, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": hbm / peaks["hbm_gbs"], "peak_source": f"{peak_src} HBM copy bandwidth"})
    return out


class Device:
    """A workload on the device: inputs, caches (pre-filled, not timed),
    outputs, workspaces, and pinned host copies of the step's inputs."""

    def __init__(self, wl, fmts, ctx, dev):
        import numpy as np
        import torch
        from dsa_sparse_attention_store_gb300 import page_bytes

        def t_bf16(bits):
            return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)

        self.wl, self.fmts, self.ctx = wl, fmts, ctx
        self.host = {
            "q": t_bf16(wl.q).pin_memory(),
            "head_w": torch.from_numpy(wl.head_w).pin_memory(),
            "new_k": t_bf16(wl.new_k).pin_memory(),
            "new_pos": torch.from_numpy(wl.new_pos).pin_memory(),
            "new_seq": torch.from_numpy(wl.new_seq).pin_memory(),
            "page_table": torch.from_numpy(wl.page_table).pin_memory(),
            "seq_lens": torch.from_numpy(wl.seq_lens).pin_memory(),
            "cu_q": torch.from_numpy(wl.cu_q).pin_memory(),
        }
        self.d = {k: v.to(dev) for k, v in self.host.items()}
        self.caches, self.outs, self.wss = {}, {}, {}
        self.fill = None
        if wl.fill_pos.shape[0]:
            self.fill = (t_bf16(wl.fill_k).to(dev), torch.from_numpy(wl.fill_pos).to(dev),
                         torch.from_numpy(wl.fill_seq).to(dev))
        for f in fmts:
            self.caches[f] = torch.zeros(wl.num_pages * page_bytes(f), dtype=torch.uint8, device=dev)
            self.outs[f] = (torch.empty((wl.Tq, wl.k), dtype=torch.int32, device=dev),
                            torch.empty((wl.Tq, wl.k), dtype=torch.float32, device=dev))
            self.wss[f] = torch.empty(ctx.topk_workspace_size(wl.Tq, wl.B, wl.k, f), dtype=torch.uint8,
                                      device=dev)
            if self.fill is not None:
                ctx.store(*self.fill, self.d["page_table"], self.caches[f], wl.num_pages, f)
        self.host_out = {f: (torch.empty((wl.Tq, wl.k), dtype=torch.int32).pin_memory(),
                             torch.empty((wl.Tq, wl.k), dtype=torch.float32).pin_memory()) for f in fmts}
        torch.cuda.synchronize()

    def step(self, src=None):
        src = src or self.d
        wl, ctx = self.wl, self.ctx
        for f in self.fmts:
            ctx.store(src["new_k"], src["new_pos"], src["new_seq"], src["page_table"], self.caches[f],
                      wl.num_pages, f)
            oi, os_ = self.outs[f]
            ctx.topk(src["q"], src["head_w"], self.caches[f], wl.num_pages, f, src["page_table"],
                     src["seq_lens"], src["cu_q"], wl.causal, wl.k, oi, os_, self.wss[f])

    def h2d_bytes(self):
        return sum(int(v.numel() * v.element_size()) for v in self.host.values())

    def d2h_bytes(self):
        return sum(int(a.numel() * a.element_size() + b.numel() * b.element_size())
                   for a, b in self.host_out.values())


def timed(fn, steps, flush):
    """Per-iteration milliseconds of fn() by CUDA events on the current
    stream, with an L2 flush between iterations outside the events."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for i in range(steps):
        evs[i][0].record()
        fn()
        evs[i][1].record()
        flush()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def measure_workload(name, args, ctx, dev, world, barrier, flush, peaks, peak_src):
    """Device, kernel and end-to-end figures of one workload (both formats
    per step)."""
    import torch
    fmts = {"both": [0, 1], "bf16": [0], "fp8": [1]}[args.fmt]
    wl = make_workload(name)
    dv = Device(wl, fmts, ctx, dev)
    for _ in range(args.warmup):
        dv.step()
        flush()
    st = ctx.device_status()
    if st != 0:
        raise RuntimeError(f"{name}: device status {st} after warm-up")

    ctx.profile_read()                      # resets the launch counters
    barrier()
    step_ms = timed(dv.step, args.steps, flush)
    barrier()
    launches = sum(n for _, n in ctx.profile_read().values())
    total_ms = sum(step_ms)

    # per-kernel times: the same steps again with the library's kernel events
    # on (events between kernels stop programmatic dependent launch from
    # overlapping them, so these are slightly pessimistic)
    ctx.profile_enable(True)
    for _ in range(args.steps):
        dv.step()
        flush()
    torch.cuda.synchronize()
    ctx.profile_enable(False)
    prof = ctx.profile_read()

    e2e_ms = None
    if not args.no_e2e:
        dd = {k: torch.empty_like(v) for k, v in dv.d.items()}

        def e2e_step():
            for k, v in dv.host.items():
                dd[k].copy_(v, non_blocking=True)
            dv.step(dd)
            for f in fmts:
                dv.host_out[f][0].copy_(dv.outs[f][0], non_blocking=True)
                dv.host_out[f][1].copy_(dv.outs[f][1], non_blocking=True)

        for _ in range(max(1, args.warmup)):
            e2e_step()
            flush()
        barrier()
        e2e_ms = sum(timed(e2e_step, args.steps, flush))
        barrier()
        del dd
    st = ctx.device_status()
    if st != 0:
        raise RuntimeError(f"{name}: device status {st} after the timed steps")

    if world > 1:
        total_ms, e2e_red = max_over_ranks([total_ms, e2e_ms or 0.0], dev)
        e2e_ms = e2e_red if e2e_ms is not None else None

    ks_step = wl.key_scores() * len(fmts)
    out = {
        "value": whole_job_rate(ks_step, args.steps, world, total_ms), "unit": "key-scores/s",
        "queries_per_s": whole_job_rate(wl.Tq * len(fmts), args.steps, world, total_ms),
        "ms_per_step": total_ms / args.steps,
        "step_ms_median": statistics.median(step_ms),
        "kernel_ms_per_step": {k: v[0] / args.steps for k, v in prof.items()},
        "gpu_launches": int(launches),
        "launches_per_step": launches / max(args.steps, 1),
        "config": workload_config(wl, name, fmts),
    }
    roofs = {}
    for f in fmts:
        sc_ms, sc_n = prof["score_" + FMT_NAMES[f]]
        nbytes, flops = scorer_algorithmic(wl, f)
        roofs[FMT_NAMES[f]] = roofline_entry(
            f"score_kernel ({FMT_NAMES[f]} cache)", sc_ms / max(sc_n, 1), nbytes, flops, f, peaks, peak_src,
            traffic_of(f"{name}/score/{FMT_NAMES[f]}", scorer_hash()), sc_n)
    out["roofline"] = roofs
    if getattr(wl, "needles", None):
        out["needle_report"] = needle_report(wl, dv, fmts, ctx, dev)
    if e2e_ms is not None:
        out["e2e"] = {"value": whole_job_rate(ks_step, args.steps, world, e2e_ms), "unit": "key-scores/s",
                      "h2d_bytes_per_step": dv.h2d_bytes(), "d2h_bytes_per_step": dv.d2h_bytes(),
                      "ms_per_step": e2e_ms / args.steps}
    if not args.no_fp4:
        out["fp4"] = measure_fp4(wl, name, args, ctx, dev, world, barrier, flush, peaks, peak_src)
    return out, wl, fmts, dv


def needles_selected(wl, out_idx):
    """How many needle queries selected each planted needle, from the GPU's
    own output rows (the parity tests compare those rows with the oracle)."""
    import numpy as np
    sel = np.asarray(out_idx)[np.asarray(wl.needle_queries)]
    per = [int((sel == p).any(axis=1).sum()) for p in wl.needles]
    return {"selected_per_needle": per, "selected": sum(per), "of": len(wl.needle_queries) * len(wl.needles)}


def needle_report(wl, dv, fmts, ctx, dev):
    """Whether each needle is selected: for the timed workload (head weights
    |N(0,1)|/8) from the last timed step's output, and for the same queries
    and keys with signed weights N(0,1)/8 from one untimed call per format."""
    import torch
    from synth import inputs as I
    rep = {"needle_positions": list(wl.needles), "needle_queries": len(wl.needle_queries),
           "abs_weights": {FMT_NAMES[f]: needles_selected(wl, dv.outs[f][0].cpu().numpy()) for f in fmts}}
    w = torch.from_numpy(I.needle(w_abs=False).head_w).to(dev)
    signed = {}
    for f in fmts:
        oi, os_ = torch.empty_like(dv.outs[f][0]), torch.empty_like(dv.outs[f][1])
        ctx.topk(dv.d["q"], w, dv.caches[f], wl.num_pages, f, dv.d["page_table"], dv.d["seq_lens"],
                 dv.d["cu_q"], wl.causal, wl.k, oi, os_, dv.wss[f])
        signed[FMT_NAMES[f]] = needles_selected(wl, oi.cpu().numpy())
    rep["signed_weights"] = signed
    st = ctx.device_status()
    if st != 0:
        raise RuntimeError(f"needle report: device status {st}")
    return rep


def measure_fp4(wl, name, args, ctx, dev, world, barrier, flush, peaks, peak_src):
    """The same workload on an fp4 cache alone (store + top-k per step): its
    throughput and scorer roofline. Not part of the headline step, whose
    formats are the pages' bf16 and fp8."""
    import torch
    dv = Device(wl, [2], ctx, dev)
    for _ in range(args.warmup):
        dv.step()
        flush()
    ctx.profile_read()
    barrier()
    step_ms = timed(dv.step, args.steps, flush)
    barrier()
    total_ms = sum(step_ms)
    ctx.profile_read()                      # only the profiled steps below count
    ctx.profile_enable(True)
    for _ in range(args.steps):
        dv.step()
        flush()
    torch.cuda.synchronize()
    ctx.profile_enable(False)
    prof = ctx.profile_read()
    st = ctx.device_status()
    if st != 0:
        raise RuntimeError(f"{name} fp4: device status {st}")
    if world > 1:
        (total_ms,) = max_over_ranks([total_ms], dev)
    sc_ms, sc_n = prof["score_fp4"]
    nbytes, flops = scorer_algorithmic(wl, 2)
    del dv
    return {"value": whole_job_rate(wl.key_scores(), args.steps, world, total_ms), "unit": "key-scores/s",
            "ms_per_step": total_ms / args.steps,
            "kernel_ms_per_step": {k: v[0] / args.steps for k, v in prof.items() if v[1]},
            "roofline": roofline_entry("score_kernel (fp4 cache)", sc_ms / max(sc_n, 1), nbytes, flops, 2,
                                       peaks, peak_src, traffic_of(f"{name}/score/fp4", scorer_hash()), sc_n)}


def measure_variant(wl, name, label, args, dev, world, barrier, flush, peaks, peak_src, hadamard=False,
                    slots=False, k=None):
    """One of the options past the pages' path on a workload, both formats
    per step like the headline: the Hadamard-rotated cache and queries, the
    top-2048 selection (k), or cache-slot output. Scorer rooflines of the
    variant's own kernels (fresh context, so the store writes the rotated
    keys when the rotation is on)."""
    import copy
    import torch
    from dsa_sparse_attention_store_gb300 import Context
    vwl = copy.copy(wl)
    if k is not None:
        vwl.k = k
    ctx = Context(theta=10000.0, eps=1e-6, max_pos=131072)
    try:
        ctx.set_hadamard(hadamard)
        ctx.set_slot_output(slots)
        dv = Device(vwl, [0, 1], ctx, dev)
        for _ in range(args.warmup):
            dv.step()
            flush()
        ctx.profile_read()
        barrier()
        step_ms = timed(dv.step, args.steps, flush)
        barrier()
        total_ms = sum(step_ms)
        ctx.profile_read()
        ctx.profile_enable(True)
        for _ in range(args.steps):
            dv.step()
            flush()
        torch.cuda.synchronize()
        ctx.profile_enable(False)
        prof = ctx.profile_read()
        st = ctx.device_status()
        if st != 0:
            raise RuntimeError(f"{name} {label}: device status {st}")
        if world > 1:
            (total_ms,) = max_over_ranks([total_ms], dev)
        roofs = {}
        for f in (0, 1):
            sc_ms, sc_n = prof["score_" + FMT_NAMES[f]]
            nbytes, flops = scorer_algorithmic(vwl, f)
            roofs[FMT_NAMES[f]] = roofline_entry(f"score_kernel ({FMT_NAMES[f]} cache, {label})",
                                                 sc_ms / max(sc_n, 1), nbytes, flops, f, peaks, peak_src,
                                                 None, sc_n)
        del dv
        return {"value": whole_job_rate(vwl.key_scores() * 2, args.steps, world, total_ms),
                "unit": "key-scores/s", "k": vwl.k, "ms_per_step": total_ms / args.steps, "roofline": roofs}
    finally:
        ctx.close()


def store_roofline(dv, which, args, flush, peaks, peak_src, label):
    """Roofline of the store kernel on `which` tokens of a workload ('fill'
    or 'new'), one launch per timed iteration, per format."""
    import torch
    wl, ctx = dv.wl, dv.ctx
    if which == "fill":
        toks = dv.fill
    else:
        toks = (dv.d["new_k"], dv.d["new_pos"], dv.d["new_seq"])
    T = int(toks[1].shape[0])
    res = {}
    for f in dv.fmts:
        def one():
            ctx.store(*toks, dv.d["page_table"], dv.caches[f], wl.num_pages, f)
        for _ in range(3):
            one()
            flush()
        ms = timed(one, max(args.steps, 5), flush)
        avg = sum(ms) / len(ms)
        ent = roofline_entry(f"store_kernel ({FMT_NAMES[f]} cache)", avg, store_algorithmic(T, f), 0, f, peaks,
                             peak_src, traffic_of(f"{label}/store/{FMT_NAMES[f]}", store_hash()), len(ms))
        ent["tokens_per_launch"] = T
        ent["tokens_per_s"] = T / (avg / 1e3)
        res[FMT_NAMES[f]] = ent
    torch.cuda.synchronize()
    return res


def run_ours(args, rank, world, local_rank):
    import torch

    from dsa_sparse_attention_store_gb300 import Context

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    ctx = Context(theta=10000.0, eps=1e-6, max_pos=131072)
    peaks, peak_src = load_peaks()
    l2 = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    l2r = torch.ones(256 << 20, dtype=torch.uint8, device=dev).view(torch.int64)

    def flush():
        # write a buffer larger than L2, then read another one: no input of
        # the next step is left in L2, and no dirty line of the flush is left
        # for the timed step to write back
        l2.fill_(1)
        torch.sum(l2r)

    dist = world > 1
    if dist:
        import torch.distributed as tdist

    def barrier():
        if dist:
            tdist.barrier()
        torch.cuda.synchronize()

    names = [args.workload] if args.workload != "all" else [HEADLINE] + [n for n in WORKLOAD_NAMES if n != HEADLINE]
    sampler = ClockSampler(local_rank)
    results, stores, wls = {}, {}, {}
    for name in names:
        res, wl, fmts, dv = measure_workload(name, args, ctx, dev, world, barrier, flush, peaks, peak_src)
        if not args.no_store_roofline:
            if name == "long_decode":
                stores["long_decode_fill"] = store_roofline(dv, "fill", args, flush, peaks, peak_src,
                                                            "long_decode_fill")
            if name == "long_prefill":
                stores["long_prefill"] = store_roofline(dv, "new", args, flush, peaks, peak_src, "long_prefill")
        results[name] = res
        wls[name] = (wl, fmts)
        del dv
        torch.cuda.empty_cache()
        if not args.no_variants and name in ("long_prefill", "batched_decode"):
            var = {"hadamard": measure_variant(wl, name, "Hadamard", args, dev, world, barrier, flush, peaks,
                                               peak_src, hadamard=True),
                   "slots": measure_variant(wl, name, "slot output", args, dev, world, barrier, flush, peaks,
                                            peak_src, slots=True)}
            if name == "batched_decode":
                var["k2048"] = measure_variant(wl, name, "k=2048", args, dev, world, barrier, flush, peaks,
                                               peak_src, k=2048)
            res["variants"] = var
            torch.cuda.empty_cache()
    clocks = sampler.stop()
    ctx.close()
    return results, stores, wls, clocks


# ------------------------------------------------------------------ oracle (CPU) arm
class OracleRunner:
    """The C++ oracle as it stands, on a workload's inputs: its own cache
    built once (setup), then per sample the step's store and a few query
    rows, spread over the batch."""

    def __init__(self, wl, fmts):
        from oracle import native as N
        self.N = N
        self.wl, self.fmts = wl, fmts
        self.caches = {}
        for f in fmts:
            c = N.new_cache(wl.num_pages, f)
            N.store(c, f, wl.fill_k, wl.fill_pos, wl.fill_seq, wl.page_table, wl.num_pages, wl.theta, wl.eps)
            self.caches[f] = c
        self.next_row = 0

    def sample(self, nrows: int):
        """Store the step's new keys, score nrows query rows per format;
        returns the key-scores done."""
        import numpy as np
        wl, N = self.wl, self.N
        rows = np.array([(self.next_row + i * 7919) % wl.Tq for i in range(min(nrows, wl.Tq))])
        self.next_row = (self.next_row + 1) % wl.Tq
        done = 0
        for f in self.fmts:
            N.store(self.caches[f], f, wl.new_k, wl.new_pos, wl.new_seq, wl.page_table, wl.num_pages,
                    wl.theta, wl.eps)
            N.index_topk(self.caches[f], f, wl.page_table, wl.seq_lens, wl.cu_q, wl.q, wl.head_w,
                         wl.causal, wl.k, rows=rows)
            done += int(N.visible_counts(wl.cu_q, wl.seq_lens, rows, wl.causal).sum())
        return done, len(rows)


def rows_per_sample(wl, target_pairs=2_000_000):
    """Query rows per oracle sample so that one sample is about target_pairs
    key-scores per format (at least 1 row, at most the batch)."""
    avg = max(wl.key_scores() / max(wl.Tq, 1), 1.0)
    return int(max(1, min(wl.Tq, round(target_pairs / avg))))


def cpu_baseline(wl, fmts, seconds):
    from oracle import native as N
    runner = OracleRunner(wl, fmts)
    nrows = rows_per_sample(wl)
    t0 = time.perf_counter()
    ks, n, rows = 0, 0, 0
    while time.perf_counter() - t0 < seconds or n == 0:
        k, r = runner.sample(nrows)
        ks += k
        rows += r
        n += 1
    dt = time.perf_counter() - t0
    return {"value": ks / dt, "unit": "key-scores/s", "cores": N.threads(), "kind": "oracle",
            "sample": f"C++ oracle (std::thread, {N.threads()} threads): {n} samples x (store of the step's "
                      f"{wl.new_pos.shape[0]} new tokens + top-k of {nrows} query rows) per format, "
                      f"{ks} key-scores in {dt:.1f} s"}


def run_reference(args):
    from oracle import native as N
    name = HEADLINE if args.workload == "all" else args.workload
    fmts = {"both": [0, 1], "bf16": [0], "fp8": [1]}[args.fmt]
    wl = make_workload(name)
    runner = OracleRunner(wl, fmts)
    nrows = rows_per_sample(wl, 1_000_000)
    for _ in range(args.warmup):
        runner.sample(nrows)
    times, ks = [], 0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        k, _ = runner.sample(nrows)
        times.append(time.perf_counter() - t0)
        ks += k
    tot = sum(times)
    value = ks / tot
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "key-scores/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 scores, f32 store (CPU oracle)", "data": "synthetic (seeded SplitMix64 + Box-Muller)",
        "config": workload_config(wl, name, fmts),
        "cpu_baseline": {"value": value, "unit": "key-scores/s", "cores": N.threads(), "kind": "oracle",
                         "sample": f"C++ oracle (std::thread, {N.threads()} threads); each step: store of the "
                                   f"{wl.new_pos.shape[0]} new tokens + top-k of {nrows} query rows per format"},
        "e2e": {"value": value, "unit": "key-scores/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def compose(args, world, results, stores, wls, clocks):
    """The JSON line: the headline workload's figures at the top level, the
    others under configs."""
    head = HEADLINE if HEADLINE in results else next(iter(results))
    h = results[head]
    wl, fmts = wls[head]
    roof = h["roofline"]
    first = FMT_NAMES[fmts[0]]
    out = {
        "metric": METRIC, "value": h["value"], "unit": "key-scores/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": h["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 q, bf16|e4m3 keys, fp32 accumulate",
        "data": "synthetic (seeded SplitMix64 + Box-Muller normals, shapes of the workload)",
        "config": h["config"],
        "queries_per_s": h["queries_per_s"],
        "step_ms_median": h["step_ms_median"],
        "kernel_ms_per_step": h["kernel_ms_per_step"],
        "roofline": roof[first],
        "roofline_other_format": roof.get("fp8") if first == "bf16" else None,
        "roofline_fp4": h["fp4"]["roofline"] if "fp4" in h else None,
        "variants": h.get("variants"),
        "gpu_launches": h["gpu_launches"],
        "launches_per_step": h["launches_per_step"],
        "clocks": clocks,
    }
    if "e2e" in h:
        out["e2e"] = h["e2e"]
    if "needle_report" in h:
        out["needle_report"] = h["needle_report"]
    if stores:
        out["store_roofline"] = stores
    out["configs"] = {n: r for n, r in results.items() if n != head}
    return out


def main(argv=None):
    args = parse_args(argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl")
    build_lib()
    results, stores, wls, clocks = run_ours(args, rank, world, local_rank)
    if rank == 0:
        out = compose(args, world, results, stores, wls, clocks)
        if world == 1 and not args.no_cpu_baseline:
            for name, (wl, fmts) in wls.items():
                cb = cpu_baseline(wl, fmts, args.cpu_seconds)
                if name == out["config"]["workload"].split(":")[0]:
                    out["cpu_baseline"] = cb
                else:
                    out["configs"][name]["cpu_baseline"] = cb
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as tdist
        tdist.barrier()
        tdist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
