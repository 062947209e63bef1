"""Benchmark of the split-K paged decode attention library.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step is one fa_decode_run over the whole batch of a seeded synthetic
workload (default: batched_gqa, 16 sequences x 32 query heads / 8 kv heads,
head dim 128, 4096 keys each in 128-row pages, split-K 4). Metric: decode
attention KV HBM GB/s = minimum bytes (K + V + Q + O, each element once; the
latent row once) / device time per step; also query tokens / s and the
fraction of the measured HBM roofline. L2 is flushed (512 MiB write) before
every timed step, outside the timed interval. Rank 0 prints one JSON line.

The line's headline is the chosen workload. Its `workloads` object holds the
same measurement (same steps, warm-up and flush) for every workload of the
library, taken in the same run, so that each one's GB/s and roofline
fraction sit under the same clock record (--headline-only skips them).

--impl reference times the fp64 CPU oracle (the only other implementation of
this computation) on the host cores, on the same workload and metric.
Under torchrun with N > 1 every rank runs its own replica (the path has no
cross-GPU exchange); value is the bytes of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode attention KV HBM GB/s"
FALLBACK_HBM_GBS = 6800.0
WORKLOAD_NAMES = ["tiny", "batched_gqa", "long_context", "ragged_speculative", "mla"]
# The workloads again over an fp8 (E4M3) cache with per-token K scales; the
# MLA latent rows keep their rope part in a bf16 cache of its own.
FP8_WORKLOADS = {"batched_gqa_e4m3": "batched_gqa", "long_context_e4m3": "long_context",
                 "ragged_speculative_e4m3": "ragged_speculative", "mla_e4m3": "mla"}


def workload(name: str):
    from split_paged_decode_gb300.workloads import WORKLOADS

    if name in FP8_WORKLOADS:
        base = WORKLOADS[FP8_WORKLOADS[name]]
        rope = base.qk_depth - base.nope_depth if base.latent else 0
        return base.with_(name=name, kv_dtype="e4m3", k_scale=True, rope_depth=rope)
    return WORKLOADS[name]


def min_bytes(w, seq_lens) -> int:
    """K + V + Q + O bytes, each element once; the latent row once. An E4M3
    cache counts one byte per K / V element plus its 4-byte per-token K scale
    and the bf16 rope part."""
    total_keys = int(sum(int(x) for x in seq_lens))
    row = w.qk_depth if w.latent else w.qk_depth + w.ov_depth
    if w.kv_dtype == "e4m3":
        per_key = (row - w.rope_depth) + 2 * w.rope_depth + (4 if w.k_scale else 0)
        kv = total_keys * w.num_kv_heads * per_key
    else:
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


def _code_only(text: str) -> str:
    """C/C++ source without comments and with whitespace collapsed (string
    literals are kept as they are, apart from whitespace)."""
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif text[i] == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    return " ".join("".join(out).split())


# Translation units of each kernel family (by the kernel's name in an ncu capture).
KERNEL_UNITS = (("mla_tc_decode_kernel", ("kernel_mla_tc.cu",)),
                ("simt_decode_kernel", ("kernel_simt.cu",)),
                ("tc_decode_kernel", ("kernel_tc.cu", "kernel_tc_fp8.cu")))


def kernel_units(kernel_name: str):
    for key, units in KERNEL_UNITS:
        if key in kernel_name:
            return units
    return None


def kernel_source_files(units) -> dict:
    """The sources a kernel family is built from: its translation units and
    every local header they include, transitively (name -> text)."""
    dirs = [os.path.join(ROOT, "split_paged_decode_gb300", "csrc"), os.path.join(ROOT, "include")]
    seen, stack = {}, list(units)
    while stack:
        name = stack.pop()
        if name in seen:
            continue
        path = next((os.path.join(d, name) for d in dirs if os.path.isfile(os.path.join(d, name))), None)
        if path is None:
            continue
        text = open(path, encoding="utf-8").read()
        seen[name] = text
        stack += re.findall(r'^\s*#\s*include\s+"([^"]+)"', text, flags=re.M)
    return seen


def kernel_source_hash(units) -> str:
    """Hash of a kernel family's sources (comments and whitespace do not
    count, so an edit of comments keeps the stored ncu traffic of the same
    code)."""
    seen = kernel_source_files(units)
    h = hashlib.sha256()
    for name in sorted(seen):
        h.update(name.encode())
        h.update(_code_only(seen[name]).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current sources of its kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            doc = json.load(f)
        ent = doc[workload]
        units = kernel_units(ent["kernel"])
        if units is None or ent.get("kernel_source_hash") != kernel_source_hash(units):
            return None
        return float(ent["bytes_per_launch"])
    except Exception:
        return None


def workload_config(w, nbytes: int) -> dict:
    return {"workload": w.name, "batch": w.batch, "num_q": w.num_q, "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "qk_depth": w.qk_depth, "ov_depth": w.ov_depth,
            "page_size": w.page_size, "splitk": w.splitk,
            "seq_lens": "fixed %d" % w.seq_len if w.seq_len else
            f"uniform [{w.seq_len_lo}, {w.seq_len_hi}] seed {w.seed}",
            "kv_dtype": w.kv_dtype if w.kv_dtype == "bf16" else f"{w.kv_dtype}, per-token K scale {w.k_scale}",
            "min_bytes_per_step": nbytes, "l2": "flushed before every timed step (512 MiB write)"}


# ---------------------------------------------------------------------------
# SM clocks and clock-event reasons during the timed regions
# ---------------------------------------------------------------------------
_REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
                0x80: "hw_power_brake_slowdown"}


class ClockSampler:
    """Polls the SM clock and the active clock-event reasons of one GPU from a
    background thread (NVML through ctypes, every ~2 ms; nvidia-smi at 20 ms
    if NVML cannot be loaded). Timed regions are marked with mark(); summary()
    takes the samples that fall inside them (or, if none does, all samples
    taken while the sampler ran, and says so). Reads only."""

    def __init__(self, cuda_index: int, period_s: float = 0.002):
        self.cuda_index = cuda_index
        self.period = period_s
        self.samples = []  # (perf_counter, sm_mhz, reason bits)
        self.max_mhz = None
        self.windows = []
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None

    def _nvml_handle(self):
        nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if nvml.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        handle = ctypes.c_void_p()
        ok = False
        try:
            import torch

            props = torch.cuda.get_device_properties(self.cuda_index)
            uuid = str(getattr(props, "uuid", ""))
            if uuid:
                key = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
                ok = nvml.nvmlDeviceGetHandleByUUID(key.encode(), ctypes.byref(handle)) == 0
            if not ok and hasattr(props, "pci_bus_id"):
                bus = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                              props.pci_device_id)
                ok = nvml.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(handle)) == 0
        except Exception:
            ok = False
        if not ok and nvml.nvmlDeviceGetHandleByIndex_v2(self.cuda_index, ctypes.byref(handle)) != 0:
            raise RuntimeError("no NVML handle")
        return nvml, handle

    def _poll_nvml(self, nvml, handle):
        clk = ctypes.c_uint()
        reasons = ctypes.c_ulonglong()
        get_reasons = getattr(nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            t = time.perf_counter()
            if nvml.nvmlDeviceGetClockInfo(handle, 1, ctypes.byref(clk)) == 0:  # 1: SM clock
                r = reasons.value if get_reasons(handle, ctypes.byref(reasons)) == 0 else 0
                self.samples.append((t, float(clk.value), int(r)))
            time.sleep(self.period)

    def _poll_smi(self):
        fields = ("clocks.sm,clocks.max.sm,clocks_event_reasons.sw_power_cap,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.hw_thermal_slowdown")
        self._proc = subprocess.Popen(["nvidia-smi", f"--id={self.cuda_index}", f"--query-gpu={fields}",
                                       "--format=csv,noheader,nounits", "-lms", "20"], stdout=subprocess.PIPE,
                                      stderr=subprocess.DEVNULL, text=True)
        for ln in self._proc.stdout:
            parts = [x.strip() for x in ln.split(",")]
            try:
                sm, mx = float(parts[0]), float(parts[1])
            except (ValueError, IndexError):
                continue
            self.max_mhz = mx
            bits = 0
            for bit, v in zip((0x4, 0x8, 0x20, 0x40), parts[2:6]):
                if v.lower() == "active":
                    bits |= bit
            self.samples.append((time.perf_counter(), sm, bits))

    def start(self):
        try:
            nvml, handle = self._nvml_handle()
            mx = ctypes.c_uint()
            if nvml.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self.source = "nvml"
            self._thread = threading.Thread(target=self._poll_nvml, args=(nvml, handle), daemon=True)
        except Exception:
            self.source = "nvidia-smi"
            self._thread = threading.Thread(target=self._poll_smi, daemon=True)
        self._thread.start()
        return self

    def stop(self):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def mark(self, t0: float, t1: float):
        self.windows.append((t0, t1))

    def summary(self):
        inside = [s for s in self.samples if any(a <= s[0] <= b for a, b in self.windows)]
        window = "timed"
        if len(inside) < 3:
            inside, window = list(self.samples), "whole run (too few samples inside the timed regions)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0, "source": self.source}
        bits = 0
        for s in inside:
            bits |= s[2]
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for b, n in _REASON_BITS.items() if bits & b), "samples": len(inside),
                "window": window, "source": self.source}


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
def time_oracle(inp, min_seconds: float, max_reps: int = 1000, threads: int | None = None):
    """Time the fp64 oracle, as it stands, over whole passes of `inp` on
    `threads` host threads (default: every core) until min_seconds have
    elapsed. Returns (seconds per pass, passes, threads)."""
    import oracle
    from split_paged_decode_gb300.workloads import bf16_bits

    if threads is None:
        threads = oracle.hardware_threads()
    pt, lens = inp.page_table.numpy(), inp.seq_lens.numpy()
    q = bf16_bits(inp.q)
    if inp.workload.kv_dtype == "e4m3":
        k8 = inp.k_pages.numpy()
        v8 = None if inp.v_pages is None else inp.v_pages.numpy()
        rope = None if inp.k_rope is None else bf16_bits(inp.k_rope)
        ks = None if inp.k_scale is None else inp.k_scale.numpy()

        def run():
            oracle.decode_fp8(q, k8, v8, pt, lens, inp.scale, k_rope=rope, k_scale=ks,
                              ov_depth=inp.workload.ov_depth, threads=threads)
    else:
        k = bf16_bits(inp.k_pages)
        v = None if inp.v_pages is None else bf16_bits(inp.v_pages)

        def run():
            oracle.decode(q, k, v, pt, lens, inp.scale, ov_depth=inp.workload.ov_depth, threads=threads)
    reps, t0 = 0, time.perf_counter()
    while True:
        run()
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            return el / reps, reps, threads


def oracle_sample(w, budget_macs: float = 4.0e9):
    """Bounded sample of a workload for the oracle: whole sequences, cut so that
    one pass stays near a second on a 16-core host (budget_macs multiply-adds)."""
    from split_paged_decode_gb300.workloads import generate

    per_seq = (w.seq_len or (w.seq_len_lo + w.seq_len_hi) // 2) * w.num_q * w.num_q_heads * (
        w.qk_depth + w.ov_depth)
    nseq = max(1, min(w.batch, int(budget_macs // max(per_seq, 1))))
    sample = w.with_(batch=nseq)
    return sample, generate(sample), f"{nseq} of {w.batch} sequences of the {w.name} workload, all heads"


def cpu_baseline(w, seconds: float, single_core_seconds: float) -> dict:
    """The oracle on every host core and on one, GB/s-equivalent (the same
    algorithmic bytes / oracle time)."""
    sample, sinp, desc = oracle_sample(w)
    nbytes = min_bytes(sample, sinp.seq_lens.tolist())
    sec, reps, threads = time_oracle(sinp, seconds)
    res = {"value": nbytes / sec / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
           "sample": f"{desc}; {reps} passes"}
    if single_core_seconds > 0:
        s1, inp1, desc1 = oracle_sample(w, budget_macs=1.0e9)
        sec1, reps1, _ = time_oracle(inp1, single_core_seconds, threads=1)
        res["single_core"] = {"value": min_bytes(s1, inp1.seq_lens.tolist()) / sec1 / 1e9, "unit": "GB/s",
                              "cores": 1, "sample": f"{desc1}; {reps1} passes"}
    return res


def run_reference(args, world, rank):
    from split_paged_decode_gb300.workloads import generate

    if rank != 0:
        return
    w = workload(args.workload)
    sample, inp, desc = oracle_sample(w)
    nbytes = min_bytes(sample, inp.seq_lens.tolist())
    for _ in range(args.warmup):
        time_oracle(inp, 0.0, max_reps=1)
    per = []
    threads = 1
    for _ in range(args.steps):
        s, _, threads = time_oracle(inp, 0.0, max_reps=1)
        per.append(s)
    sec = statistics.mean(per)
    gbs = nbytes / sec / 1e9
    full = generate(w) if sample.batch != w.batch else inp
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(workload_config(w, min_bytes(w, full.seq_lens.tolist())), parallelism=f"replicas x{world}"),
        "query_tokens_per_s": sample.batch * sample.num_q / sec,
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{desc}; GB/s-equivalent = that sample's algorithmic bytes / oracle time"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
class Measured:
    pass


def measure(spd, torch, w, dev, stream, steps, warmup, flush, clocks, keep=False) -> Measured:
    """Device time of `steps` decode steps of workload w, each after an L2 flush,
    with CUDA events on the launching stream."""
    from split_paged_decode_gb300.workloads import generate

    m = Measured()
    inp = generate(w)
    m.w, m.inp = w, inp
    m.nbytes = min_bytes(w, inp.seq_lens.tolist())
    q, k = inp.q.to(dev), inp.k_pages.to(dev)
    v = None if inp.v_pages is None else inp.v_pages.to(dev)
    pt, lens = inp.page_table.to(dev), inp.seq_lens.to(dev)
    out = torch.empty((w.batch, w.num_q, w.num_q_heads, w.ov_depth), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.batch, w.num_q, w.num_q_heads), dtype=torch.float32, device=dev)
    e4m3 = w.kv_dtype == "e4m3"
    if e4m3:
        ks = None if inp.k_scale is None else inp.k_scale.to(dev)
        rope = None if inp.k_rope is None else inp.k_rope.to(dev)
        h = spd.fa_decode_create_kv(w.num_q_heads, w.num_kv_heads, w.qk_depth, w.nope_depth, w.ov_depth,
                                    w.page_size, w.num_q, w.splitk, spd.FA_KV_E4M3, w.rope_depth)
    else:
        h = spd.fa_decode_create(w.num_q_heads, w.num_kv_heads, w.qk_depth, w.nope_depth, w.ov_depth,
                                 w.page_size, w.num_q, w.splitk)
    desc = spd.fa_decode_describe(h)
    m.kernel = desc.split()[1].split("=", 1)[1]
    # The per-sequence split (splitk 0) is one launch of 4-CTA clusters on the
    # tensor-core path, which the description states, for up to 4096
    # sequences; otherwise one launch per cluster size (1, 2, 4).
    m.launches_per_step = 1 if w.splitk != 0 or ("one launch" in desc and w.batch <= 4096) else 3

    def step():
        if e4m3:
            spd.fa_decode_run_kv(h, q, k, v, rope, ks, pt, lens, inp.scale, out, lse, stream=stream)
        else:
            spd.fa_decode_run(h, q, k, v, pt, lens, inp.scale, out, lse, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            flush.fill_(1)
            step()
        stream.synchronize()
        if spd.fa_decode_check(h, stream) != 0:
            raise RuntimeError(f"{w.name}: device status raised during warm-up")
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(steps):
            flush.fill_(i & 0xFF)       # 512 MiB write evicts L2 (129 MB) before each timed step
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        clocks.mark(t0, time.perf_counter())
        m.times_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        if spd.fa_decode_check(h, stream) != 0:
            raise RuntimeError(f"{w.name}: device status raised during the timed steps")
    m.ms = statistics.mean(m.times_ms)
    if keep:
        m.h, m.step = h, step
        m.dev_tensors = (q, k, v, pt, lens, out, lse)
        m.dev_scale = ks if e4m3 else None
        m.dev_rope = rope if e4m3 else None
    else:
        spd.fa_decode_destroy(h)
    return m


def host_enqueue_us(spd, torch, m, stream, calls: int = 50) -> dict:
    """Host time per enqueue of fa_decode_run and of fa_decode_run_noalloc
    (status read skipped) on the headline inputs: the CPU cost of a call,
    the device work being queued behind it."""
    w, inp = m.w, m.inp
    q, k, v, pt, lens, out, lse = m.dev_tensors
    res = {}
    # the allocation-free entry point takes a bf16 cache only
    names = ("fa_decode_run_kv",) if w.kv_dtype == "e4m3" else ("fa_decode_run", "fa_decode_run_noalloc")
    for name in names:
        ts = []
        for _ in range(calls):
            t0 = time.perf_counter()
            if name != "fa_decode_run_noalloc":
                m.step()
            else:
                spd.fa_decode_run_noalloc(w.num_q_heads, w.num_kv_heads, w.qk_depth, w.nope_depth, w.ov_depth,
                                          w.page_size, w.num_q, w.splitk, q, k, v, pt, lens, inp.scale, out, lse,
                                          stream=stream, status_slot=0, wait=False)
            ts.append((time.perf_counter() - t0) * 1e6)
            stream.synchronize()
        res[name] = statistics.median(ts)
    return res


def run_gpu(args, world, rank, local):
    import torch

    import split_paged_decode_gb300 as spd
    from split_paged_decode_gb300.workloads import WORKLOADS

    spd.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    peak, peak_kind = hbm_peak()
    w = workload(args.workload)
    clocks = ClockSampler(local).start()
    try:
        barrier(world)
        head = measure(spd, torch, w, dev, stream, args.steps, args.warmup, flush, clocks, keep=True)
        others = {}
        if not args.headline_only:
            for name in WORKLOAD_NAMES + list(FP8_WORKLOADS):
                if name != w.name:
                    others[name] = measure(spd, torch, workload(name), dev, stream, args.steps, args.warmup,
                                           flush, clocks)
        barrier(world)
    finally:
        clocks.stop()

    # end to end through the same C ABI call: pinned host inputs copied in,
    # the result read back, every step
    q, k, v, pt, lens, out, lse = head.dev_tensors
    inp = head.inp
    pin = lambda t: None if t is None else t.pin_memory()  # noqa: E731
    hq, hk, hv, hpt, hlens = pin(inp.q), pin(inp.k_pages), pin(inp.v_pages), pin(inp.page_table), \
        pin(inp.seq_lens)
    hks, ks = pin(inp.k_scale), head.dev_scale
    hrope, rope = pin(inp.k_rope), head.dev_rope
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hpt, hlens, hks, hrope) if t is not None)
    d2h = hout.numel() * hout.element_size() + hlse.numel() * hlse.element_size()
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        q.copy_(hq, non_blocking=True)
        k.copy_(hk, non_blocking=True)
        if v is not None:
            v.copy_(hv, non_blocking=True)
        pt.copy_(hpt, non_blocking=True)
        lens.copy_(hlens, non_blocking=True)
        if ks is not None:
            ks.copy_(hks, non_blocking=True)
        if rope is not None:
            rope.copy_(hrope, non_blocking=True)
        head.step()
        hout.copy_(out, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)

    with torch.cuda.stream(stream):
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
        enqueue = host_enqueue_us(spd, torch, head, stream)
    spd.fa_decode_destroy(head.h)

    ms_max = max_over_ranks(head.ms, world)
    e2e_ms = max_over_ranks(e2e_ms, world)
    if rank != 0:
        return
    nbytes = head.nbytes
    gbs = world * nbytes / (ms_max * 1e-3) / 1e9
    achieved = nbytes / head.launches_per_step / (head.ms / head.launches_per_step * 1e-3) / 1e9
    clk = clocks.summary()

    def entry(m):
        g = m.nbytes / (m.ms * 1e-3) / 1e9
        return {"kernel": m.kernel, "us_per_step": m.ms * 1e3, "gbs": g, "frac": g / peak,
                "query_tokens_per_s": m.w.batch * m.w.num_q / (m.ms * 1e-3), "launches_per_step": m.launches_per_step,
                "min_bytes_per_step": m.nbytes, "traffic": ncu_traffic(m.w.name)}

    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.kv_dtype == "bf16" else "e4m3 KV, bf16 Q/out",
        "data": "synthetic",
        "config": dict(workload_config(w, nbytes), parallelism=f"replicas x{world}"),
        "query_tokens_per_s": world * w.batch * w.num_q / (ms_max * 1e-3),
        "roofline_pct": 100.0 * gbs / world / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} (copy bandwidth, burst)",
                     "kernel": head.kernel, "traffic": ncu_traffic(w.name)},
        "e2e": {"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": head.launches_per_step * args.steps,
        "clocks": clk,
        "host_enqueue_us": enqueue,
    }
    if others:
        line["workloads"] = {name: entry(m) for name, m in [(w.name, head)] + list(others.items())}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds, args.cpu_single_core_seconds)
        if others:
            for name in ("tiny", "long_context"):
                if name in line["workloads"]:
                    cb = cpu_baseline(workload(name), 1.0, 1.0)
                    line["workloads"][name]["cpu_baseline_gbs"] = cb["value"]
                    line["workloads"][name]["cpu_baseline_cores"] = cb["cores"]
                    line["workloads"][name]["cpu_single_core_gbs"] = cb["single_core"]["value"]
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="batched_gqa", choices=WORKLOAD_NAMES + list(FP8_WORKLOADS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle timing budget of cpu_baseline")
    ap.add_argument("--cpu-single-core-seconds", type=float, default=3.0,
                    help="oracle timing budget of the single-core baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true", help="measure the chosen workload only")
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
