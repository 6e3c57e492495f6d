"""Benchmark: key-value LSD radix sort of 2^28 u32 keys with a u32 index
payload, 8-bit digits (4 passes), on one GB300 (or N independent replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--n LOG2] [--no-distributions] [--no-e2e] [--no-cpu-baseline]
                    [--no-copy-probe] [--no-small-sorts] [--no-rows]

Prints one JSON line on rank 0.  `value` is sorted keys per second with the
inputs already in HBM (inputs of 2 GiB, larger than L2, so no flush is
needed); `e2e` is the same sort through the C ABI with the keys and payloads
copied from pinned host memory and the result copied back inside the timed
region.  `roofline` reports the onesweep scatter kernel (the dominant one)
against the measured HBM copy bandwidth; `cpu_baseline` times the CPU oracle
on a bounded sample of the same workload.  `distributions` times the other
key distributions of the same workload, each also with pass skipping on
(reported apart from the ideal-bytes model, since identity passes are not
run); `small_sorts` compares stream launches with CUDA-graph replay of the
same sort from 2^10 to 2^20 keys; `row_sorts` times the row-wise fp16 sort
on the FlagTree H20 shapes with both ways of finding tile offsets, beside
torch.sort.  Under torchrun each rank sorts its own
replica (the sort has no exchange step); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Gkeys/s sorted (u32 keys & pairs, 2^28) + achieved HBM GB/s vs GB300 peak"
FALLBACK_HBM_GBS = 6800.0
DIGIT_BITS = 8
KEY_BYTES = 4
VAL_BYTES = 4


def ideal_bytes(n: int, passes: int, key_bytes: int, val_bytes: int) -> int:
    """One read of the keys for all histograms, then per pass one read and
    one write of every key and payload."""
    return n * key_bytes + passes * 2 * n * (key_bytes + val_bytes)


def sweep_bytes_per_launch(n: int, key_bytes: int, val_bytes: int) -> int:
    return 2 * n * (key_bytes + val_bytes)


def workload_name(n_log2: int) -> str:
    return (f"key-value sort, 2^{n_log2} u32 keys (uniform 32-bit, seed 0) + u32 index payload, "
            f"{DIGIT_BITS}-bit digits ({32 // DIGIT_BITS} passes)")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


SWEEP_SOURCES = ("onesweep.cuh", "sweep_u32.cu", "kernels.h", "common.cuh", "keys.cuh")


def code_only(text: str) -> str:
    """C++ source without comments and with whitespace collapsed, so that a
    change of wording in a comment does not count as a change of the kernel."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def onesweep_source_hash(read=None) -> str:
    """Hash of the code (comments stripped) the u32 scatter kernel is built
    from; `read(name)` returns a file's text (default: the working tree)."""
    if read is None:
        def read(name):
            with open(os.path.join(ROOT, "lsd_radix_sort_gb300", "csrc", name), encoding="utf-8",
                      errors="replace") as fh:
                return fh.read()
    h = hashlib.sha256()
    for f in SWEEP_SOURCES:
        h.update(code_only(read(f)).encode())
    return h.hexdigest()[:16]


def recorded_traffic(n: int):
    """DRAM bytes per onesweep launch from the committed ncu summary, scaled to
    n keys, or None when the kernel source changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "onesweep_u32_pairs_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("source_hash") != onesweep_source_hash():
        return None
    return int(d["dram_bytes_per_key"] * n)


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


E2E_REPS = 3  # repetitions of each end-to-end schedule; the best is reported


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (the job's time is its slowest replica)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def small_sort_latency(rs, torch, workloads, log2_sizes, reps: int = 200):
    """Per-sort time of small key-value sorts launched on a stream and replayed
    from a CUDA graph that captured the same call (the launch sequence of a
    sort is fixed and needs no host synchronisation, so one call captures)."""
    import numpy as np
    out = {}
    stream = torch.cuda.current_stream()
    for lg in log2_sizes:
        n = 1 << lg
        dk = torch.from_numpy(workloads.u32_uniform(n, lg).view(np.int32)).cuda()
        dv = torch.from_numpy(workloads.index_payload(n).view(np.int32)).cuda()
        ko, vo = torch.empty_like(dk), torch.empty_like(dv)
        temp = torch.empty(rs.temp_bytes(n, 4, 4, 0, 32, DIGIT_BITS), dtype=torch.uint8,
                           device="cuda")

        def sort():
            rs.radix_sort_pairs(dk, dv, ko, vo, 0, 32, DIGIT_BITS, temp=temp)

        def timed(fn):
            for _ in range(10):
                fn()
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) * 1e3 / reps
        t_stream = timed(sort)
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(3):
                sort()
        stream.wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            sort()
        t_graph = timed(g.replay)
        out[f"2^{lg}"] = {"stream_us": round(t_stream, 2), "graph_us": round(t_graph, 2),
                          "graph_saves": round(1 - t_graph / t_stream, 3)}
        del g, dk, dv, ko, vo, temp
    return out


def keys_only_configs(rs, torch, workloads, reps: int = 50):
    """The two keys-only workloads: 1,024 keys below 4,096 sorted on bits
    0-11 in three 4-bit passes, and 4,194,304 uniform u32 keys sorted in
    eight 4-bit or four 8-bit passes (seeds 0-2; the inputs fit in L2).
    Stream-launched time per sort, and the CUDA-graph replay of the same
    call, with each result checked against a stable sort on the device."""
    import numpy as np
    stream = torch.cuda.current_stream()
    cases = [("1024_keys_b4_bits0_12", 1024, 4, 12, lambda seed: workloads.u32_small(1024, seed, 12)),
             ("2^22_keys_b4", 1 << 22, 4, 32, lambda seed: workloads.u32_uniform(1 << 22, seed)),
             ("2^22_keys_b8", 1 << 22, 8, 32, lambda seed: workloads.u32_uniform(1 << 22, seed))]
    out = {}
    for name, n, bits, end, gen in cases:
        per_seed = []
        for seed in range(3):
            dk = torch.from_numpy(gen(seed).view(np.int32)).cuda()
            ko = torch.empty_like(dk)
            temp = torch.empty(rs.temp_bytes(n, 4, 0, 0, end, bits), dtype=torch.uint8,
                               device="cuda")

            def sort():
                rs.radix_sort_keys(dk, ko, 0, end, bits, temp=temp)

            def timed(fn):
                for _ in range(5):
                    fn()
                torch.cuda.synchronize()
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                for _ in range(reps):
                    fn()
                b.record(stream)
                torch.cuda.synchronize()
                return a.elapsed_time(b) * 1e3 / reps
            t_stream = timed(sort)
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                for _ in range(3):
                    sort()
            stream.wait_stream(side)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                sort()
            t_graph = timed(g.replay)
            k64 = dk.to(torch.int64) & 0xFFFFFFFF
            want = torch.sort(k64 & ((1 << end) - 1), stable=True)
            ok = bool(torch.equal(ko.to(torch.int64) & 0xFFFFFFFF, k64[want.indices]))
            per_seed.append({"seed": seed, "stream_us": round(t_stream, 2),
                             "graph_us": round(t_graph, 2), "checked": ok})
            del g, dk, ko, temp
        best = min(min(r["stream_us"], r["graph_us"]) for r in per_seed)
        out[name] = {"n": n, "digit_bits": bits, "passes": (end + bits - 1) // bits,
                     "gkeys_s_best": round(n / best / 1e3, 2), "seeds": per_seed}
    return out


def _order_key(torch, k, key_type: str, descending: bool = False):
    """int64 tensor whose signed order is the sort order of the keys (the
    order-preserving transform of the typed sorts), for result checks."""
    if key_type in ("u32", "i32", "f32"):
        u = k.view(torch.int32).to(torch.int64) & 0xFFFFFFFF
        top = u >> 31
        if key_type == "i32":
            t = u ^ 0x80000000
        elif key_type == "f32":
            t = torch.where(top == 1, u ^ 0xFFFFFFFF, u ^ 0x80000000)
        else:
            t = u
        return (0xFFFFFFFF - t) if descending else t
    x = k.view(torch.int64)
    return (x ^ -(1 << 63)) if key_type == "u64" else x  # unsigned order as signed


def _check_sorted_pairs(torch, keys_in, keys_out, vals_out, order_in, order_out) -> bool:
    """Payload indices are a permutation carrying each key, keys are in order
    and equal keys keep input order (the stable order is then fixed)."""
    idx = vals_out.view(torch.int32).to(torch.int64)
    if not torch.equal(keys_in[idx], keys_out):
        return False
    if bool((order_out[1:] < order_out[:-1]).any()):
        return False
    ties = order_out[1:] == order_out[:-1]
    if bool((ties & (idx[1:] < idx[:-1])).any()):
        return False
    return bool(torch.bincount(idx, minlength=idx.numel()).eq(1).all())


def config_sorts(rs, torch, workloads, n_log2: int, peak: float, reps: int = 10):
    """The other headline-size workloads, each timed with CUDA events over
    `reps` sorts after 3 warm-ups (inputs resident, larger than L2) and its
    result checked on the device: u32 keys only; u64 key-value sorts
    (uniform, skewed, the 0-39-bit run); typed 32-bit key-value sorts; the
    row-wise fp16/bf16 sort of (1024, 65536) ascending and descending."""
    import numpy as np
    n = 1 << n_log2
    stream = torch.cuda.current_stream()
    out = {}

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    def entry(ms, nkeys, ideal, ok, **kw):
        d = {"ms": round(ms, 4), "gkeys_s": round(nkeys / ms / 1e6, 2),
             "hbm_frac": round(ideal / (ms * 1e-3) / 1e9 / peak, 4), "checked": ok}
        d.update(kw)
        return d

    # u32 keys only: histogram read 4 B + 4 passes x (read + write) 4 B
    k32 = torch.from_numpy(workloads.u32_uniform(n, 0).view(np.int32)).cuda()
    ko = torch.empty_like(k32)
    temp = torch.empty(rs.temp_bytes(n, 4, 0, 0, 32, 8), dtype=torch.uint8, device="cuda")
    ms = timed(lambda: rs.radix_sort_keys(k32, ko, 0, 32, 8, temp=temp))
    o = _order_key(torch, ko, "u32")
    ok = not bool((o[1:] < o[:-1]).any()) and torch.equal(
        torch.sort(_order_key(torch, k32, "u32")).values, o)
    out["u32_keys"] = entry(ms, n, n * (4 + 4 * 8), ok, digit_bits=8, passes=4)
    del ko, temp

    # typed 32-bit key-value sorts on the same bit patterns (f32 includes
    # every special pattern the uniform words produce: NaNs, infinities, -0)
    vals = torch.from_numpy(workloads.index_payload(n).view(np.int32)).cuda()
    ko, vo = torch.empty_like(k32), torch.empty_like(vals)
    temp = torch.empty(rs.temp_bytes(n, 4, 4, 0, 32, 8), dtype=torch.uint8, device="cuda")
    for kt, desc in (("f32", False), ("f32", True), ("i32", False)):
        kin = k32.view(torch.float32) if kt == "f32" else k32
        kout = ko.view(torch.float32) if kt == "f32" else ko
        ms = timed(lambda: rs.radix_sort_pairs(kin, vals, kout, vo, temp=temp, key_type=kt,
                                               descending=desc))
        ok = _check_sorted_pairs(torch, k32, ko, vo, None, _order_key(torch, ko, kt, desc))
        out[f"{kt}_pairs{'_desc' if desc else ''}"] = entry(ms, n, n * (4 + 4 * 16), ok)
    del k32, ko, vo, temp

    # u64 keys + u32 payload: histogram read 8 B + P passes x (read + write) 12 B
    for name, gen, end in (("u64_pairs_uniform", workloads.u64_uniform, 64),
                           ("u64_pairs_skewed", workloads.u64_skewed, 64),
                           ("u64_pairs_bits0_39", workloads.u64_uniform, 40)):
        k64 = torch.from_numpy(gen(n, 0).view(np.int64)).cuda()
        ko, vo = torch.empty_like(k64), torch.empty_like(vals)
        temp = torch.empty(rs.temp_bytes(n, 8, 4, 0, end, 8), dtype=torch.uint8, device="cuda")
        ms = timed(lambda: rs.radix_sort_pairs(k64, vals, ko, vo, 0, end, 8, temp=temp))
        masked = ko if end == 64 else ko & ((1 << end) - 1)
        ok = _check_sorted_pairs(torch, k64, ko, vo, None,
                                 _order_key(torch, masked, "u64" if end == 64 else "i64"))
        passes = (end + 7) // 8
        out[name] = entry(ms, n, n * (8 + passes * 24), ok, passes=passes)
        del k64, ko, vo, temp
    del vals

    # row-wise 16-bit float sorts, (1024, 65536), int64 indices; minimum bytes:
    # histogram read 2 B, pass 0 read 2 / write 2 + 4 (int32 index), pass 1
    # read 2 + 4 / write 2 + 8 (int64 index)
    rows, cols = 1024, 65536
    for kind in ("f16", "bf16"):
        x = torch.from_numpy(workloads.rows16(rows, cols, kind, 0).view(np.int16)).cuda()
        x = x.view(torch.float16 if kind == "f16" else torch.bfloat16)
        v = torch.empty_like(x)
        i = torch.empty((rows, cols), dtype=torch.int64, device="cuda")
        temp = torch.empty(rs.segmented_temp_bytes(rows, cols), dtype=torch.uint8, device="cuda")
        for desc in (False, True):
            ms = timed(lambda: rs.segmented_sort(x, desc, values_out=v, indices_out=i, temp=temp))
            xi = x.view(torch.int16)
            gathered = torch.equal(torch.gather(xi, 1, i), v.view(torch.int16))
            u = xi.to(torch.int64) & 0xFFFF
            t = torch.where(u >= 0x8000, u ^ 0xFFFF, u | 0x8000)
            t = (0xFFFF - t) if desc else t
            tv = torch.gather(t, 1, i)
            ok = gathered and not bool((tv[:, 1:] < tv[:, :-1]).any()) and not bool(
                ((tv[:, 1:] == tv[:, :-1]) & (i[:, 1:] < i[:, :-1])).any())
            out[f"rows_{kind}_{rows}x{cols}{'_desc' if desc else ''}"] = entry(
                ms, rows * cols, rows * cols * 26, ok,
                hbm_frac_formula=round(rows * cols * 42 / (ms * 1e-3) / 1e9 / peak, 4))
        del x, v, i, temp
    return out


ROW_SHAPES = [(64, 64), (256, 256), (1024, 1024), (4096, 4096), (1024, 65536), (1024, 1),
              (1024, 512), (16, 131072), (8, 262144)]


def row_sorts(rs, torch, workloads, reps: int = 20):
    """Row-wise fp16 sorts on the FlagTree PR #1084 H20 shapes (ascending,
    last dimension): torch.sort, and this library with the tile offsets found
    by the look-back and precomputed before each pass."""
    import numpy as np
    out = {}
    for rows, cols in ROW_SHAPES:
        x = torch.from_numpy(workloads.rows16(rows, cols, "f16", 0).view(np.int16)).cuda()
        x = x.view(torch.float16)
        v = torch.empty_like(x)
        idx = torch.empty((rows, cols), dtype=torch.int64, device="cuda")
        temp = torch.empty(rs.segmented_temp_bytes(rows, cols), dtype=torch.uint8, device="cuda")

        def timed(fn):
            for _ in range(5):
                fn()
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(reps):
                fn()
            b.record()
            torch.cuda.synchronize()
            return a.elapsed_time(b) / reps
        entry = {"torch_sort_ms": round(timed(lambda: torch.sort(x, dim=-1)), 4)}
        for mode, name in ((False, "lookback_ms"), (True, "precomputed_ms")):
            entry[name] = round(timed(lambda: rs.segmented_sort(x, False, v, idx, temp,
                                                                tile_offsets=mode)), 4)
        out[f"{rows}x{cols}"] = entry
        del x, v, idx, temp
    return out


def host_cores() -> dict:
    """The host's logical cores and the ones this process may run on."""
    try:
        usable = len(os.sched_getaffinity(0))
    except Exception:
        usable = os.cpu_count()
    return {"logical": os.cpu_count(), "usable": usable}


def _median_time(fn, reps: int) -> float:
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        fn()
        times.append(time.perf_counter() - t0)
    return statistics.median(times)


def cpu_oracle_rate(n_sample: int, reps: int = 1):
    """Time the CPU oracle (as it stands, one thread) on a sample of the workload."""
    import oracle
    from lsd_radix_sort_gb300 import workloads
    keys = workloads.u32_uniform(n_sample, 0)
    vals = workloads.index_payload(n_sample)
    oracle.build()
    secs = _median_time(lambda: oracle.sort(keys, vals, 0, 32, DIGIT_BITS), reps)
    return n_sample / secs / 1e9, secs


def cpu_config_rates(log2: int) -> dict:
    """The oracle (one thread, as it stands) on a bounded sample of every
    configuration, and numpy's stable sort of the headline keys on one core
    (a library comparison sort, the CUDA Handbook's std::sort analogue).
    Samples: 2^log2 keys for the 2^28 workloads (2^(log2-2) for 64-bit keys),
    the small configurations whole; median of 3 runs below 2^24 keys, one
    run above.  Rates in Gkeys/s."""
    import oracle
    from lsd_radix_sort_gb300 import workloads
    oracle.build()
    out = {}

    def rate(name, n, fn, sample):
        secs = _median_time(fn, 3 if n < (1 << 24) else 1)
        out[name] = {"gkeys_s": n / secs / 1e9, "seconds": round(secs, 4), "sample": sample}

    k = workloads.u32_small(1024, 0, 12)
    rate("1024_keys_b4_bits0_12", 1024, lambda: oracle.sort(k, None, 0, 12, 4), "whole (1,024 keys)")
    for bits in (4, 8):
        k = workloads.u32_uniform(1 << 22, 0)
        rate(f"2^22_keys_b{bits}", 1 << 22, lambda: oracle.sort(k, None, 0, 32, bits),
             "whole (4,194,304 keys, seed 0)")
    n = 1 << log2
    k = workloads.u32_uniform(n, 0)
    v = workloads.index_payload(n)
    rate("u32_pairs_uniform", n, lambda: oracle.sort(k, v, 0, 32, 8), f"2^{log2} of 2^28 keys")
    rate("u32_keys_uniform", n, lambda: oracle.sort(k, None, 0, 32, 8), f"2^{log2} of 2^28 keys")
    t0 = time.perf_counter()
    np.argsort(k, kind="stable")
    secs = time.perf_counter() - t0
    out["numpy_stable_argsort_u32_1core"] = {"gkeys_s": n / secs / 1e9, "seconds": round(secs, 4),
                                             "sample": f"2^{log2} uniform u32 keys, one thread"}
    for name, gen in workloads.U32_DISTRIBUTIONS.items():
        if name == "uniform":
            continue
        kk = gen(1 << (log2 - 2), 0)
        vv = workloads.index_payload(kk.size)
        rate(f"u32_pairs_{name}", kk.size, lambda: oracle.sort(kk, vv, 0, 32, 8),
             f"2^{log2 - 2} of 2^28 keys")
    n64 = 1 << (log2 - 2)
    v64 = workloads.index_payload(n64)
    for name, gen, end in (("u64_pairs_uniform", workloads.u64_uniform, 64),
                           ("u64_pairs_skewed", workloads.u64_skewed, 64),
                           ("u64_pairs_bits0_39", workloads.u64_uniform, 40)):
        kk = gen(n64, 0)
        rate(name, n64, lambda: oracle.sort(kk, v64, 0, end, 8), f"2^{log2 - 2} of 2^28 keys")
    rows = 64
    for kind in ("f16", "bf16"):
        x = workloads.rows16(rows, 65536, kind, 0)
        rate(f"rows_{kind}_1024x65536", rows * 65536, lambda: oracle.segmented_sort16(x, False),
             f"{rows} of 1024 rows")
    return out


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle on the host cores, bounded samples."""
    if rank != 0:
        return
    n_sample = 1 << args.ref_log2
    import oracle
    from lsd_radix_sort_gb300 import workloads
    oracle.build()
    keys = workloads.u32_uniform(n_sample, 0)
    vals = workloads.index_payload(n_sample)
    for _ in range(args.warmup):
        oracle.sort(keys, vals, 0, 32, DIGIT_BITS)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.sort(keys, vals, 0, 32, DIGIT_BITS)
    dt = (time.perf_counter() - t0) / args.steps
    v = n_sample / dt / 1e9
    sample = f"2^{args.ref_log2} keys of the same uniform u32 key-value workload per step"
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "Gkeys/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u32", "data": "synthetic",
            "config": {"workload": workload_name(args.n_log2), "sample_keys": n_sample},
            "cpu_baseline": {"value": v, "unit": "Gkeys/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "Gkeys/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def time_sorts(rs, torch, dk, dv, ko, vo, temp, steps, warmup, stream, **opts):
    for _ in range(warmup):
        rs.radix_sort_pairs(dk, dv, ko, vo, 0, 32, DIGIT_BITS, temp=temp, **opts)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        rs.radix_sort_pairs(dk, dv, ko, vo, 0, 32, DIGIT_BITS, temp=temp, **opts)
    stop.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(stop) / steps


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--n", dest="n_log2", type=int, default=28)
    ap.add_argument("--ref-log2", type=int, default=24)
    ap.add_argument("--cpu-log2", type=int, default=28)
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-distributions", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-copy-probe", action="store_true")
    ap.add_argument("--no-small-sorts", action="store_true")
    ap.add_argument("--no-rows", action="store_true")
    ap.add_argument("--no-configs", action="store_true")
    ap.add_argument("--no-cpu-configs", action="store_true")
    ap.add_argument("--e2e-sets", type=int, default=2,
                    help="device buffer sets the pipelined end-to-end schedule rotates through")
    ap.add_argument("--details", default=None,
                    help="file for the bulky tables (default: bench_details.json at the "
                         "repository root)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank, world, local = dist_setup()
    details = {}  # bulky tables, written beside the run instead of printed
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import lsd_radix_sort_gb300 as rs
    from lsd_radix_sort_gb300 import build, workloads

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build.build()
    rs.load_library()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    n = 1 << args.n_log2
    passes = 32 // DIGIT_BITS

    keys = workloads.u32_uniform(n, 0)
    vals = workloads.index_payload(n)
    dk = torch.from_numpy(keys.view(np.int32)).to(dev)
    dv = torch.from_numpy(vals.view(np.int32)).to(dev)
    ko = torch.empty_like(dk)
    vo = torch.empty_like(dv)
    temp = torch.empty(rs.temp_bytes(n, 4, 4, 0, 32, DIGIT_BITS), dtype=torch.uint8, device=dev)

    # ---- device-resident timed region (with per-kernel events) ----------
    for _ in range(args.warmup):
        rs.radix_sort_pairs(dk, dv, ko, vo, 0, 32, DIGIT_BITS, temp=temp)
    torch.cuda.synchronize()
    rs.profile_read()
    rs.launch_count_reset()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    rs.profile_enable(True)
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(args.steps):
        rs.radix_sort_pairs(dk, dv, ko, vo, 0, 32, DIGIT_BITS, temp=temp)
    stop.record(stream)
    torch.cuda.synchronize()
    rs.profile_enable(False)
    barrier(world)
    clocks = sampler.stop()
    launches = rs.launch_count_reset()
    ms = start.elapsed_time(stop) / args.steps
    recs = rs.profile_read()
    status = rs.device_status(temp)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed sorts")
    ms_max = max_over_ranks(ms, world, dev)
    value = world * n / (ms_max * 1e-3) / 1e9

    per_kernel = {}
    for name, kms, units in recs:
        d = per_kernel.setdefault(name, [0, 0.0])
        d[0] += 1
        d[1] += kms
    sweep_launches, sweep_ms = per_kernel.get("onesweep", [0, 0.0])
    sweep_avg = sweep_ms / max(sweep_launches, 1)
    peak, peak_kind = load_peaks()
    achieved = sweep_bytes_per_launch(n, KEY_BYTES, VAL_BYTES) / (sweep_avg * 1e-3) / 1e9
    total_ideal = ideal_bytes(n, passes, KEY_BYTES, VAL_BYTES)
    roofline = {"bound": "hbm", "kernel": "onesweep (one scatter pass)",
                "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_source": f"{peak_kind} hbm_gbs (copy, burst)",
                "copy_probe_gbs": None,
                "traffic": recorded_traffic(n),
                "algorithmic_bytes_per_launch": sweep_bytes_per_launch(n, KEY_BYTES, VAL_BYTES),
                "avg_launch_ms": sweep_avg}
    kernels = {k: {"launches": c, "total_ms": t, "share": t / max(sum(x[1] for x in
                                                                      per_kernel.values()), 1e-9)}
               for k, (c, t) in per_kernel.items()}

    # ---- the copy probe: this build's own streaming copy on the same GPU ----
    copy_gbs = None
    if not args.no_copy_probe:
        src = torch.empty(1 << 31, dtype=torch.uint8, device=dev)  # 2 GiB, > L2
        dst = torch.empty_like(src)
        for _ in range(3):
            rs.copy_probe(dst, src)
        torch.cuda.synchronize()
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(10):
            rs.copy_probe(dst, src)
        c1.record(stream)
        torch.cuda.synchronize()
        copy_gbs = 2 * src.numel() / (c0.elapsed_time(c1) / 10 * 1e-3) / 1e9
        rs.profile_read()
        del src, dst

    # ---- end to end through host buffers ---------------------------------
    e2e = None
    if not args.no_e2e:
        # Every step copies its keys and payloads from pinned host memory,
        # sorts them through the public API, and copies the sorted keys and
        # payloads back.  Serial: one step after the other on one stream.
        # Pipelined (reported as `e2e`): device buffer sets (two by default); step i's
        # upload, sort and readback are ordered by events, so step i's
        # readback overlaps step i+1's upload and sort (the link carries both
        # directions at once); each step still moves all of its own bytes.
        # An upload into a set waits only for the sort that last read that
        # set's inputs; the sort waits for its upload and for the readback of
        # the set's previous outputs, which it overwrites.
        hk = torch.from_numpy(keys.view(np.int32)).pin_memory()
        hv = torch.from_numpy(vals.view(np.int32)).pin_memory()
        sets = []
        nsets = args.e2e_sets
        for _ in range(nsets):
            sets.append({"dk": torch.empty_like(dk), "dv": torch.empty_like(dv),
                         "ko": torch.empty_like(dk), "vo": torch.empty_like(dv),
                         "temp": torch.empty_like(temp),
                         "hko": torch.empty_like(hk).pin_memory(),
                         "hvo": torch.empty_like(hv).pin_memory()})
        up, comp, down = torch.cuda.Stream(), stream, torch.cuda.Stream()

        def serial_step():
            b = sets[0]
            b["dk"].copy_(hk, non_blocking=True)
            b["dv"].copy_(hv, non_blocking=True)
            rs.radix_sort_pairs(b["dk"], b["dv"], b["ko"], b["vo"], 0, 32, DIGIT_BITS,
                                temp=b["temp"])
            b["hko"].copy_(b["ko"], non_blocking=True)
            b["hvo"].copy_(b["vo"], non_blocking=True)

        freed = [None] * nsets     # the set's last readback is done
        consumed = [None] * nsets  # the set's last sort is done (its inputs are free)

        def pipelined_step(i):
            b = sets[i % nsets]
            with torch.cuda.stream(up):
                if consumed[i % nsets] is not None:
                    up.wait_event(consumed[i % nsets])
                b["dk"].copy_(hk, non_blocking=True)
                b["dv"].copy_(hv, non_blocking=True)
                loaded = torch.cuda.Event()
                loaded.record(up)
            comp.wait_event(loaded)
            if freed[i % nsets] is not None:
                comp.wait_event(freed[i % nsets])
            rs.radix_sort_pairs(b["dk"], b["dv"], b["ko"], b["vo"], 0, 32, DIGIT_BITS,
                                temp=b["temp"], stream=comp)
            sorted_ev = torch.cuda.Event()
            sorted_ev.record(comp)
            consumed[i % nsets] = sorted_ev
            with torch.cuda.stream(down):
                down.wait_event(sorted_ev)
                b["hko"].copy_(b["ko"], non_blocking=True)
                b["hvo"].copy_(b["vo"], non_blocking=True)
                done = torch.cuda.Event()
                done.record(down)
            freed[i % nsets] = done

        # The host link is shared with the rest of the machine: bursts of
        # 50-180 ms in which host copies run several times slower come and
        # go whatever this program does (its enqueue stays at 0.1 ms per
        # step).  Each schedule is therefore timed in E2E_REPS repetitions of
        # `steps` consecutive steps, and the best repetition's mean step time
        # is reported, every repetition beside it.
        def timed_e2e(step_fn, steps):
            for i in range(2):
                step_fn(i)
            torch.cuda.synchronize()
            reps = []
            for _ in range(E2E_REPS):
                barrier(world)
                t0 = time.perf_counter()
                for i in range(steps):
                    step_fn(i)
                torch.cuda.synchronize()
                reps.append(max_over_ranks((time.perf_counter() - t0) * 1e3 / steps, world, dev))
            return min(reps), reps

        # The host link on its own: one 1 GiB copy each way, then both at once
        # (the pipelined schedule's bound), best of three.
        def link_gbs(fn, nbytes):
            best = None
            for _ in range(3):
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                fn()
                torch.cuda.synchronize()
                dt = time.perf_counter() - t0
                best = dt if best is None else min(best, dt)
            return nbytes / best / 1e9

        def both_ways():
            with torch.cuda.stream(up):
                sets[0]["dk"].copy_(hk, non_blocking=True)
            with torch.cuda.stream(down):
                sets[0]["hko"].copy_(sets[1]["dk"], non_blocking=True)

        link = {"h2d_gbs": link_gbs(lambda: sets[0]["dk"].copy_(hk, non_blocking=True), hk.numel() * 4),
                "d2h_gbs": link_gbs(lambda: sets[0]["hko"].copy_(sets[0]["dk"], non_blocking=True),
                                    hk.numel() * 4),
                "both_ways_gbs": link_gbs(both_ways, 2 * hk.numel() * 4)}
        pipe_steps = max(args.e2e_steps, 6)
        e_serial, serial_reps = timed_e2e(lambda i: serial_step(), args.e2e_steps)
        e_pipe, pipe_reps = timed_e2e(pipelined_step, pipe_steps)
        # The last step's result, as it came back to host memory, is checked
        # whole on the device: keys in order, payloads a permutation that
        # carries each input key, equal keys in input order.
        b = sets[(pipe_steps - 1) % nsets]
        for key in ("dk", "dv", "ko", "vo", "temp"):
            for st in sets:
                st[key] = None
        hko_d, hvo_d = b["hko"].to(dev), b["hvo"].to(dev)
        ok = _check_sorted_pairs(torch, dk, hko_d, hvo_d, None, _order_key(torch, hko_d, "u32"))
        del hko_d, hvo_d
        e2e = {"value": world * n / (e_pipe * 1e-3) / 1e9, "unit": "Gkeys/s",
               "h2d_bytes_per_step": hk.numel() * 4 + hv.numel() * 4,
               "d2h_bytes_per_step": sets[0]["hko"].numel() * 4 + sets[0]["hvo"].numel() * 4,
               "ms_per_step": e_pipe, "mode": f"pipelined over {nsets} buffer sets (wall clock)",
               "timing": f"best of {E2E_REPS} repetitions of {pipe_steps} steps",
               "result_checked": ok, "result_check": "whole output, properties on the device",
               "serial_value": world * n / (e_serial * 1e-3) / 1e9,
               "host_link_gbs": {k: round(v, 1) for k, v in link.items()}}
        details["e2e"] = {"reps_ms_per_step": [round(x, 3) for x in pipe_reps],
                          "serial": {"ms_per_step": e_serial,
                                     "timing": f"best of {E2E_REPS} repetitions of "
                                               f"{args.e2e_steps} steps",
                                     "reps_ms_per_step": [round(x, 3) for x in serial_reps]}}
        del hk, hv, sets

    # ---- the other key distributions of the same workload ----------------
    dists = None
    if not args.no_distributions:
        dists = {}
        for name, gen in workloads.U32_DISTRIBUTIONS.items():
            if name == "uniform":
                dms = ms
            else:
                kk = gen(n, 0)
                dk.copy_(torch.from_numpy(kk.view(np.int32)))
                del kk
                dms = time_sorts(rs, torch, dk, dv, ko, vo, temp, max(args.steps // 2, 3), 3,
                                 stream)
            dists[name] = {"ms": round(dms, 4), "gkeys_s": round(n / (dms * 1e-3) / 1e9, 2),
                           "hbm_frac": round(total_ideal / (dms * 1e-3) / 1e9 / peak, 4)}
            if name != "uniform":
                # the same sort with pass skipping on: identity passes are not
                # run, so the ideal-bytes model above does not apply
                sms = time_sorts(rs, torch, dk, dv, ko, vo, temp, max(args.steps // 2, 3), 3,
                                 stream, pass_skipping=True)
                dists[name]["pass_skipping"] = {"ms": round(sms, 4),
                                                "passes_run": rs.passes_run(temp)}

    cfg_tab = None
    if not args.no_configs and args.n_log2 == 28:
        cfg_tab = config_sorts(rs, torch, workloads, args.n_log2, peak)
    small = None
    keys_cfg = None
    if not args.no_small_sorts:
        small_full = small_sort_latency(rs, torch, workloads, (10, 12, 13, 14, 16, 18, 20))
        details["small_sorts"] = small_full
        small = {k: [v["stream_us"], v["graph_us"]] for k, v in small_full.items()}
        keys_full = keys_only_configs(rs, torch, workloads)
        details["keys_only_configs"] = keys_full
        keys_cfg = {k: {"gkeys_s_best": v["gkeys_s_best"],
                        "checked": all(r["checked"] for r in v["seeds"])}
                    for k, v in keys_full.items()}
    rows_tab = None
    if not args.no_rows:
        rows_full = row_sorts(rs, torch, workloads)
        details["row_sorts"] = rows_full
        rows_tab = {k: [v["lookback_ms"], v["precomputed_ms"], v["torch_sort_ms"]]
                    for k, v in rows_full.items()}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, secs = cpu_oracle_rate(1 << args.cpu_log2)
        cpu = {"value": rate, "unit": "Gkeys/s", "cores": 1, "kind": "oracle",
               "sample": f"2^{args.cpu_log2} keys of the same uniform u32 key-value workload, "
                         f"one sort, {secs:.1f} s on one host thread",
               "host_cores": host_cores()}
        if not args.no_cpu_configs:
            cpu_cfg = cpu_config_rates(args.cpu_log2 - 2)
            details["cpu_baseline_configs"] = cpu_cfg
            cpu["configs_gkeys_s"] = {k: round(v["gkeys_s"], 5) for k, v in cpu_cfg.items()}

    roofline["copy_probe_gbs"] = copy_gbs
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "Gkeys/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "u32", "data": "synthetic",
                "config": {"workload": workload_name(args.n_log2), "n_keys": n,
                           "digit_bits": DIGIT_BITS, "passes": passes,
                           "l2": (f"inputs larger than L2 ({n * 8 / 2**20:.0f} MiB keys+payload vs "
                                  "129 MB L2), no flush" if n * 8 > 129e6 else
                                  f"inputs ({n * 8 / 2**20:.1f} MiB) fit in L2, no flush"),
                           "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
                "hbm": {"ideal_bytes_per_sort": total_ideal,
                        "achieved_gbs": total_ideal / (ms_max * 1e-3) / 1e9,
                        "frac_of_peak": total_ideal / (ms_max * 1e-3) / 1e9 / peak},
                "e2e": e2e, "gpu_launches": launches, "kernels": kernels,
                "roofline": roofline, "cpu_baseline": cpu, "clocks": clocks,
                "distributions": dists, "configs": cfg_tab,
                "small_sorts_us_stream_graph": small, "keys_only_configs": keys_cfg,
                "row_sorts_ms_lookback_precomputed_torch": rows_tab}
        path = os.path.abspath(args.details or os.path.join(ROOT, "bench_details.json"))
        try:
            os.makedirs(os.path.dirname(path), exist_ok=True)
            with open(path, "w") as f:
                json.dump(details, f, indent=1)
            line["details_file"] = os.path.relpath(path, ROOT)
        except OSError:
            line["details_file"] = None
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
