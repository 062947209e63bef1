"""Benchmark of the split-K paged decode attention library.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step is one fa_decode_run over the whole batch of a seeded synthetic
workload (default: batched_gqa, 16 sequences x 32 query heads / 8 kv heads,
head dim 128, 4096 keys each in 128-row pages, split-K 4). Metric: decode
attention KV HBM GB/s = minimum bytes (K + V + Q + O, each element once; the
latent row once) / device time per step; also query tokens / s and the
fraction of the measured HBM roofline. L2 is flushed (512 MiB write) before
every timed step, outside the timed interval. Rank 0 prints one JSON line.

--impl reference times the fp64 CPU oracle (the only other implementation of
this computation) on the host cores, on the same workload and metric.
Under torchrun with N > 1 every rank runs its own replica (the path has no
cross-GPU exchange); value is the bytes of all ranks / the slowest rank's time.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode attention KV HBM GB/s"
FALLBACK_HBM_GBS = 6800.0


def min_bytes(w, seq_lens) -> int:
    """K + V + Q + O bytes, each element once; the latent row once."""
    total_keys = int(sum(int(x) for x in seq_lens))
    row = w.qk_depth if w.latent else w.qk_depth + w.ov_depth
    kv = total_keys * w.num_kv_heads * row * 2
    q = w.batch * w.num_q * w.num_q_heads * w.qk_depth * 2
    o = w.batch * w.num_q * w.num_q_heads * w.ov_depth * 2
    return kv + q + o


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    """Hash of the device-code sources (the host planner's files are excluded)."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "split_paged_decode_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        if f.endswith((".cu", ".cuh", ".h")) and f not in ("fa_decode_host.cu", "stream_k_plan.h"):
            h.update(f.encode())
            h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            doc = json.load(f)
        ent = doc[workload]
        if ent.get("kernel_source_hash") != kernel_source_hash():
            return None
        return float(ent["bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        for ln in getattr(self, "lines", []):
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl"
        import torch

        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        else:
            backend = "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------
def time_oracle(inp, min_seconds: float, max_reps: int = 1000):
    """Time the fp64 oracle, as it stands, over whole passes of `inp` on every
    host core until min_seconds have elapsed. Returns (seconds per pass, passes, threads)."""
    import oracle
    from split_paged_decode_gb300.workloads import bf16_bits

    threads = oracle.hardware_threads()
    q, k = bf16_bits(inp.q), bf16_bits(inp.k_pages)
    v = None if inp.v_pages is None else bf16_bits(inp.v_pages)
    pt, lens = inp.page_table.numpy(), inp.seq_lens.numpy()
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.decode(q, k, v, pt, lens, inp.scale, ov_depth=inp.workload.ov_depth, threads=threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            return el / reps, reps, threads


def oracle_sample(w):
    """Bounded sample of a workload for the oracle: whole sequences, cut so that
    one pass stays near a second on a 16-core host."""
    from split_paged_decode_gb300.workloads import generate

    budget_macs = 4.0e9
    per_seq = (w.seq_len or (w.seq_len_lo + w.seq_len_hi) // 2) * w.num_q * w.num_q_heads * (
        w.qk_depth + w.ov_depth)
    nseq = max(1, min(w.batch, int(budget_macs // max(per_seq, 1))))
    sample = w.with_(batch=nseq)
    return sample, generate(sample), f"{nseq} of {w.batch} sequences of the {w.name} workload, all heads"


def run_reference(args, world, rank):
    from split_paged_decode_gb300.workloads import WORKLOADS

    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    sample, inp, desc = oracle_sample(w)
    nbytes = min_bytes(sample, inp.seq_lens.tolist())
    for _ in range(args.warmup):
        time_oracle(inp, 0.0, max_reps=1)
    per = []
    for _ in range(args.steps):
        s, _, threads = time_oracle(inp, 0.0, max_reps=1)
        per.append(s)
    sec = statistics.mean(per)
    gbs = nbytes / sec / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample": desc},
        "query_tokens_per_s": sample.batch * sample.num_q / sec,
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_gpu(args, world, rank, local):
    import torch

    import split_paged_decode_gb300 as spd
    from split_paged_decode_gb300.workloads import WORKLOADS, generate

    spd.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    inp = generate(w)
    nbytes = min_bytes(w, inp.seq_lens.tolist())
    stream = torch.cuda.Stream(device=dev)

    q, k = inp.q.to(dev), inp.k_pages.to(dev)
    v = None if inp.v_pages is None else inp.v_pages.to(dev)
    pt, lens = inp.page_table.to(dev), inp.seq_lens.to(dev)
    out = torch.empty((w.batch, w.num_q, w.num_q_heads, w.ov_depth), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.batch, w.num_q, w.num_q_heads), dtype=torch.float32, device=dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    h = spd.fa_decode_create(w.num_q_heads, w.num_kv_heads, w.qk_depth, w.nope_depth, w.ov_depth,
                             w.page_size, w.num_q, w.splitk)
    launches_per_step = 3 if w.splitk == 0 else 1

    def step():
        spd.fa_decode_run(h, q, k, v, pt, lens, inp.scale, out, lse, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.fill_(1)
            step()
        stream.synchronize()
        if spd.fa_decode_check(h, stream) != 0:
            raise RuntimeError("device status raised during warm-up")

        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier(world)
        torch.cuda.synchronize()
        with ClockSampler(local) as clocks:
            for i in range(args.steps):
                flush.fill_(i & 0xFF)       # 512 MiB write evicts L2 (129 MB) before each timed step
                starts[i].record(stream)
                step()
                ends[i].record(stream)
            torch.cuda.synchronize()
        barrier(world)
        times_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        if spd.fa_decode_check(h, stream) != 0:
            raise RuntimeError("device status raised during the timed steps")

        # end to end through the same C ABI call: pinned host inputs copied in,
        # the result read back, every step
        pin = lambda t: None if t is None else t.pin_memory()  # noqa: E731
        hq, hk, hv, hpt, hlens = pin(inp.q), pin(inp.k_pages), pin(inp.v_pages), pin(inp.page_table), \
            pin(inp.seq_lens)
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hpt, hlens) if t is not None)
        d2h = hout.numel() * hout.element_size() + hlse.numel() * hlse.element_size()
        e2e_steps = max(3, min(args.steps, 20))

        def e2e_step():
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            if v is not None:
                v.copy_(hv, non_blocking=True)
            pt.copy_(hpt, non_blocking=True)
            lens.copy_(hlens, non_blocking=True)
            step()
            hout.copy_(out, non_blocking=True)
            hlse.copy_(lse, non_blocking=True)

        e2e_step()
        stream.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        stream.synchronize()
        e2e_ms = e0.elapsed_time(e1) / e2e_steps

    spd.fa_decode_destroy(h)
    ms = statistics.mean(times_ms)
    ms_max = max_over_ranks(ms, world)
    e2e_ms = max_over_ranks(e2e_ms, world)
    if rank != 0:
        return
    gbs = world * nbytes / (ms_max * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    per_launch_ms = ms / launches_per_step
    achieved = nbytes / launches_per_step / (per_launch_ms * 1e-3) / 1e9
    clk = clocks.summary()
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "num_q": w.num_q, "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "qk_depth": w.qk_depth, "ov_depth": w.ov_depth,
                   "page_size": w.page_size, "splitk": w.splitk, "seq_lens": "fixed %d" % w.seq_len
                   if w.seq_len else f"uniform [{w.seq_len_lo}, {w.seq_len_hi}] seed {w.seed}",
                   "min_bytes_per_step": nbytes, "l2": "flushed before every timed step (512 MiB write)",
                   "parallelism": f"replicas x{world}"},
        "query_tokens_per_s": world * w.batch * w.num_q / (ms_max * 1e-3),
        "roofline_pct": 100.0 * gbs / world / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} (copy bandwidth, burst)",
                     "traffic": ncu_traffic(w.name)},
        "e2e": {"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"]},
    }
    if not args.no_cpu_baseline:
        sample, sinp, desc = oracle_sample(w)
        sec, reps, threads = time_oracle(sinp, args.cpu_seconds)
        line["cpu_baseline"] = {"value": min_bytes(sample, sinp.seq_lens.tolist()) / sec / 1e9, "unit": "GB/s",
                                "cores": threads, "kind": "oracle", "sample": f"{desc}; {reps} passes"}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="batched_gqa",
                    choices=["tiny", "batched_gqa", "long_context", "ragged_speculative", "mla"])
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle timing budget of cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_gpu(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
