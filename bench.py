#!/usr/bin/env python3
"""Benchmark of the DSA indexer hot path (store + score/top-k) on GB300.

One step = one pass of the whole path over one batch of the workload: the
step's new index keys are stored (RMSNorm + RoPE + quantise + paged write)
and every query of the batch is scored against its visible keys and reduced
to its top-k. The default workload is the batched decode: 64 sequences, one
query each, contexts uniform in [2048, 16384], 64-token pages with a permuted
page table, k = 512, run for both cache formats (bf16 and fp8) in each step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample

Prints one JSON line. `value` is key-scores/s (sum over queries of the keys
each query is scored against) over all GPUs; inputs are resident in HBM when
the timed region starts and L2 is flushed (256 MB write) between timed steps,
outside the timed events. `e2e` is the same metric through the C ABI with
the step's inputs copied from pinned host memory and the results copied back
inside the timed region. `roofline` is for the scorer kernel, timed by the
library's own CUDA events on the launch stream.
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
FMT_NAMES = {0: "bf16", 1: "fp8"}
TOKEN_BYTES = {0: 256, 1: 132}
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
SCORER_SRC = os.path.join(ROOT, "dsa_sparse_attention_store_gb300", "csrc", "topk.cu")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


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
    cache format fmt: every visible key read once (256 B bf16, 132 B fp8),
    the queries (16 KB each, bf16 or two e4m3 terms) and head weights, one
    4-byte page id per page, 8 bytes per output entry; 2 * 64 * 128 flops
    per (query, visible key) pair."""
    import numpy as np
    pages = sum((int(L) + 63) // 64 for L in wl.seq_lens)
    nbytes = (int(wl.seq_lens.astype(np.int64).sum()) * TOKEN_BYTES[fmt]
              + wl.Tq * 64 * 128 * 2 + wl.Tq * 64 * 4
              + pages * 4 + wl.Tq * wl.k * 8)
    return nbytes, wl.key_scores() * 2 * 64 * 128


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="batched_decode",
                    choices=["batched_decode", "tiny_prefill", "long_prefill", "needle", "long_decode"])
    ap.add_argument("--fmt", choices=["both", "bf16", "fp8"], default="both")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    return ap.parse_args()


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return FALLBACK_PEAKS, "fallback"


def scorer_hash() -> str:
    """Hash of the scorer's code (comments and blank space removed, so that
    a comment edit does not invalidate a traffic capture; any code change
    does)."""
    import re
    h = hashlib.sha256()
    for name in ("topk.cu", "ptx.cuh", "internal.cuh"):
        with open(os.path.join(os.path.dirname(SCORER_SRC), name), encoding="utf-8") as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def workload_config(wl, fmts):
    desc = {
        "batched_decode": "64 sequences x 1 query, context U[2048,16384], page_size 64, permuted pages, k=512",
        "tiny_prefill": "1 sequence x 1024 tokens, causal prefill, k=512",
        "long_prefill": "1 sequence x 22528 tokens, causal prefill, k=512",
        "needle": "1 sequence x 10498 tokens, causal prefill, 5 planted needles, k=512",
        "long_decode": "8 sequences x 131072 context, 256 appended + 8 queries per sequence, k=1024",
    }
    base = wl.name.split("_B")[0].split("_L")[0]
    return {
        "workload": f"{base}: {desc.get(base, wl.name)}",
        "formats": [FMT_NAMES[f] for f in fmts],
        "global_batch": wl.Tq,
        "sequences": wl.B,
        "tokens_stored_per_step": int(wl.new_pos.shape[0]),
        "key_scores_per_step": int(wl.key_scores() * len(fmts)),
        "k": wl.k,
        "causal": wl.causal,
        "l2": "flushed between timed steps (256 MB write, outside the timed events)",
    }


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
        self.t0 = self.t1 = None

    def mark(self, start: bool):
        if start:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

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

    def _summary(self, rows):
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


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    from dsa_sparse_attention_store_gb300 import Context, page_bytes
    from synth import inputs as I

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    fmts = {"both": [0, 1], "bf16": [0], "fp8": [1]}[args.fmt]
    wl = I.WORKLOADS[args.workload]()
    ctx = Context(theta=wl.theta, eps=wl.eps, max_pos=wl.max_pos)

    def t_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)

    host = {  # step inputs in pinned host memory (for the end-to-end leg)
        "q": t_bf16(wl.q).pin_memory(),
        "head_w": torch.from_numpy(wl.head_w).pin_memory(),
        "new_k": t_bf16(wl.new_k).pin_memory(),
        "new_pos": torch.from_numpy(wl.new_pos).pin_memory(),
        "new_seq": torch.from_numpy(wl.new_seq).pin_memory(),
        "page_table": torch.from_numpy(wl.page_table).pin_memory(),
        "seq_lens": torch.from_numpy(wl.seq_lens).pin_memory(),
        "cu_q": torch.from_numpy(wl.cu_q).pin_memory(),
    }
    d = {k: v.to(dev) for k, v in host.items()}
    caches, outs, wss = {}, {}, {}
    for f in fmts:
        caches[f] = torch.zeros(wl.num_pages * page_bytes(f), dtype=torch.uint8, device=dev)
        outs[f] = (torch.empty((wl.Tq, wl.k), dtype=torch.int32, device=dev),
                   torch.empty((wl.Tq, wl.k), dtype=torch.float32, device=dev))
        wss[f] = torch.empty(ctx.topk_workspace_size(wl.Tq, wl.B, wl.k, f), dtype=torch.uint8, device=dev)
        if wl.fill_pos.shape[0]:  # pre-filled context (setup, not timed)
            fk = t_bf16(wl.fill_k).to(dev)
            fp = torch.from_numpy(wl.fill_pos).to(dev)
            fs = torch.from_numpy(wl.fill_seq).to(dev)
            ctx.store(fk, fp, fs, d["page_table"], caches[f], wl.num_pages, f)
            del fk, fp, fs
    torch.cuda.synchronize()
    host_out = {f: (torch.empty((wl.Tq, wl.k), dtype=torch.int32).pin_memory(),
                    torch.empty((wl.Tq, wl.k), dtype=torch.float32).pin_memory()) for f in fmts}

    def step(src):
        for f in fmts:
            ctx.store(src["new_k"], src["new_pos"], src["new_seq"], src["page_table"], caches[f],
                      wl.num_pages, f)
            oi, os_ = outs[f]
            ctx.topk(src["q"], src["head_w"], caches[f], wl.num_pages, f, src["page_table"],
                     src["seq_lens"], src["cu_q"], wl.causal, wl.k, oi, os_, wss[f])

    l2 = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def flush():
        l2.fill_(1)

    dist = world > 1
    if dist:
        import torch.distributed as tdist

    def barrier():
        if dist:
            tdist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step(d)
        flush()
    st = ctx.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")

    sampler = ClockSampler(local_rank)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    ctx.profile_read()                      # resets the launch counters
    barrier()
    sampler.mark(True)
    for i in range(args.steps):
        evs[i][0].record()
        step(d)
        evs[i][1].record()
        flush()
    barrier()
    sampler.mark(False)
    launches = sum(n for _, n in ctx.profile_read().values())
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = sum(step_ms)

    # per-kernel times: the same steps again with the library's kernel events
    # on (events between kernels stop programmatic dependent launch from
    # overlapping them, so these are slightly pessimistic)
    ctx.profile_enable(True)
    for i in range(args.steps):
        step(d)
        flush()
    torch.cuda.synchronize()
    ctx.profile_enable(False)
    prof = ctx.profile_read()

    # end-to-end through the C ABI from pinned host buffers
    e2e_ms = None
    h2d = sum(int(v.numel() * v.element_size()) for v in host.values())
    d2h = sum(int(a.numel() * a.element_size() + b.numel() * b.element_size()) for a, b in host_out.values())
    if not args.no_e2e:
        dd = {k: torch.empty_like(v) for k, v in d.items()}

        def e2e_step():
            for k, v in host.items():
                dd[k].copy_(v, non_blocking=True)
            step(dd)
            for f in fmts:
                host_out[f][0].copy_(outs[f][0], non_blocking=True)
                host_out[f][1].copy_(outs[f][1], non_blocking=True)

        for _ in range(max(1, args.warmup)):
            e2e_step()
            flush()
        barrier()
        eevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)]
        for i in range(args.steps):
            eevs[i][0].record()
            e2e_step()
            eevs[i][1].record()
            flush()
        barrier()
        e2e_ms = sum(a.elapsed_time(b) for a, b in eevs)
    clocks = sampler.stop()
    st = ctx.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed steps")

    if dist:
        total_ms, e2e_red = max_over_ranks([total_ms, e2e_ms or 0.0], dev)
        e2e_ms = e2e_red if e2e_ms is not None else None

    ks_step = wl.key_scores() * len(fmts)
    value = whole_job_rate(ks_step, args.steps, world, total_ms)
    qps = whole_job_rate(wl.Tq * len(fmts), args.steps, world, total_ms)

    # roofline of the scorer, per cache format (its launches in the timed region)
    peaks, peak_src = load_peaks()
    launches_per_step = launches / max(args.steps, 1)

    def roofline(f):
        sc_ms, sc_n = prof["score_" + FMT_NAMES[f]]
        avg_ms = sc_ms / max(sc_n, 1)
        nbytes, flops_launch = scorer_algorithmic(wl, f)
        hbm = nbytes / (avg_ms / 1e3) / 1e9
        tc = flops_launch / (avg_ms / 1e3) / 1e12
        traffic = None
        try:
            with open(TRAFFIC_FILE) as fh:
                ent = json.load(fh).get(f"{args.workload}/{FMT_NAMES[f]}")
            if ent and ent.get("scorer_hash") == scorer_hash():
                traffic = ent["dram_bytes_per_launch"]
        except (OSError, ValueError):
            pass
        if tc / peaks["bf16_tflops"] > hbm / peaks["hbm_gbs"]:
            r = {"bound": "tensor", "achieved": tc, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                 "frac": tc / peaks["bf16_tflops"],
                 "peak_source": f"{peak_src} bf16 dense burst (the fp8 path's two e4m3 MMA passes take the tensor time of one bf16 pass)"}
        else:
            r = {"bound": "hbm", "achieved": hbm, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                 "frac": hbm / peaks["hbm_gbs"], "peak_source": f"{peak_src} HBM copy bandwidth"}
        r.update({"traffic": traffic, "kernel": f"score_kernel ({FMT_NAMES[f]} cache)",
                  "algorithmic_bytes_per_launch": nbytes, "algorithmic_flops_per_launch": flops_launch,
                  "avg_launch_ms": avg_ms, "launches": sc_n})
        return r

    roofs = {f: roofline(f) for f in fmts}

    out = {
        "metric": METRIC, "value": value, "unit": "key-scores/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 q, bf16|e4m3 keys, fp32 accumulate",
        "data": "synthetic (seeded SplitMix64 + Box-Muller normals, shapes of the workload)",
        "config": workload_config(wl, fmts),
        "queries_per_s": qps,
        "step_ms_median": statistics.median(step_ms),
        "kernel_ms_per_step": {k: v[0] / args.steps for k, v in prof.items()},
        "roofline": roofs[fmts[0]],
        "roofline_other_format": roofs[fmts[1]] if len(fmts) > 1 else None,
        "gpu_launches": int(launches),
        "launches_per_step": launches_per_step,
        "clocks": clocks,
    }
    if e2e_ms is not None:
        out["e2e"] = {"value": whole_job_rate(ks_step, args.steps, world, e2e_ms), "unit": "key-scores/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "ms_per_step": e2e_ms / args.steps}
    ctx.close()
    return out, wl, fmts


# ------------------------------------------------------------------ oracle (CPU) arm
def oracle_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        n = max((i.get("num_threads", 1) for i in info if i.get("user_api") == "blas"), default=None)
        if n:
            return int(n), "BLAS threads (threadpoolctl)"
    except ImportError:
        pass
    return os.cpu_count() or 1, "host cores (BLAS default thread count)"


class OracleRunner:
    """The oracle as it stands, on the workload's inputs: its own cache built
    once (setup), then per sample the step's store and a few query rows."""

    def __init__(self, wl, fmts):
        from oracle import store as S
        self.S = S
        self.wl = wl
        self.fmts = fmts
        self.caches = {}
        for f in fmts:
            c = S.new_cache(wl.num_pages, f)
            S.store(c, f, wl.fill_k, wl.fill_pos, wl.fill_seq, wl.page_table, wl.num_pages, wl.theta, wl.eps)
            self.caches[f] = c
        self.next_row = 0

    def sample(self, nrows: int):
        """Store the step's new keys, score nrows query rows per format;
        returns key-scores done."""
        from oracle import indexer as X
        wl = self.wl
        done = 0
        rows = [(self.next_row + i * 7919) % wl.Tq for i in range(nrows)]
        self.next_row = (self.next_row + 1) % wl.Tq
        for f in self.fmts:
            self.S.store(self.caches[f], f, wl.new_k, wl.new_pos, wl.new_seq, wl.page_table, wl.num_pages,
                         wl.theta, wl.eps)
            X.index_topk(self.caches[f], f, wl.page_table, wl.seq_lens, wl.cu_q, wl.q, wl.head_w,
                         wl.causal, wl.k, rows=rows)
            done += sum(X.visible_count(wl.cu_q, wl.seq_lens, r, wl.causal) for r in rows)
        return done, rows


def cpu_baseline(wl, fmts, seconds):
    runner = OracleRunner(wl, fmts)
    cores, how = oracle_threads()
    t0 = time.perf_counter()
    ks = 0
    n = 0
    while time.perf_counter() - t0 < seconds or n == 0:
        k, _ = runner.sample(2)
        ks += k
        n += 1
    dt = time.perf_counter() - t0
    return {"value": ks / dt, "unit": "key-scores/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} samples x (store of the step's {wl.new_pos.shape[0]} new tokens + top-k of 2 "
                      f"query rows) per format, {ks} key-scores in {dt:.1f} s; {how}"}


def run_reference(args, wl=None):
    import numpy as np  # noqa: F401
    from synth import inputs as I
    fmts = {"both": [0, 1], "bf16": [0], "fp8": [1]}[args.fmt]
    wl = wl or I.WORKLOADS[args.workload]()
    runner = OracleRunner(wl, fmts)
    cores, how = oracle_threads()
    for _ in range(args.warmup):
        runner.sample(2)
    times, ks = [], 0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        k, _ = runner.sample(2)
        times.append(time.perf_counter() - t0)
        ks += k
    tot = sum(times)
    value = ks / tot
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "key-scores/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 scores, f32 store (CPU oracle)", "data": "synthetic (seeded SplitMix64 + Box-Muller)",
        "config": workload_config(wl, fmts),
        "cpu_baseline": {"value": value, "unit": "key-scores/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: store of the {wl.new_pos.shape[0]} new tokens + top-k of 2 "
                                   f"query rows per format; {how}"},
        "e2e": {"value": value, "unit": "key-scores/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
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
    out, wl, fmts = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(wl, fmts, args.cpu_seconds)
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as tdist
        tdist.barrier()
        tdist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
