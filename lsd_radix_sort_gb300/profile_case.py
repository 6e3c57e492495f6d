"""Run one sort workload a fixed number of times, for profiling.

    python -m lsd_radix_sort_gb300.profile_case CASE [--log2 N] [--bits B]
                                                [--sorts K] [--warmup W]
                                                [--rows R] [--cols C]

CASE is one of
  pairs_u32   N u32 keys + u32 index payload (uniform 32-bit keys, seed 0)
  keys_u32    N u32 keys only (uniform, seed 0)
  pairs_u64   N u64 keys + u32 index payload (uniform 64-bit keys, seed 0)
  rows_f16    (R, C) fp16 rows (the standard-normal mix), ascending; by
              default (1024, 65536)
  rows_bf16   the same rows in bf16

Each sort is timed with CUDA events around every kernel the library enqueues
(on the launching stream) and the script prints one JSON line with the
average per kernel and per sort.  Under a profiler, select the launches by
kernel name and skip the warm-up sorts: every sort launches the upfront
histogram, the scan and one scatter kernel per pass, in that order.
"""
from __future__ import annotations

import argparse
import json

import numpy as np


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["pairs_u32", "keys_u32", "pairs_u64", "rows_f16",
                                     "rows_bf16"])
    ap.add_argument("--log2", type=int, default=25)
    ap.add_argument("--bits", type=int, default=8)
    ap.add_argument("--end-bit", type=int, default=None)
    ap.add_argument("--sorts", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--rows", type=int, default=1024, help="rows of the row-wise cases")
    ap.add_argument("--cols", type=int, default=65536, help="columns of the row-wise cases")
    args = ap.parse_args()

    import torch

    import lsd_radix_sort_gb300 as rs
    from lsd_radix_sort_gb300 import workloads

    rs.load_library()
    dev = torch.device("cuda", 0)
    n = 1 << args.log2
    if args.case in ("pairs_u32", "keys_u32"):
        keys = torch.from_numpy(workloads.u32_uniform(n, 0).view(np.int32)).to(dev)
        end = args.end_bit or 32
        ko = torch.empty_like(keys)
        if args.case == "pairs_u32":
            vals = torch.from_numpy(workloads.index_payload(n).view(np.int32)).to(dev)
            vo = torch.empty_like(vals)
            temp = torch.empty(rs.temp_bytes(n, 4, 4, 0, end, args.bits), dtype=torch.uint8,
                               device=dev)

            def sort():
                rs.radix_sort_pairs(keys, vals, ko, vo, 0, end, args.bits, temp=temp)
        else:
            temp = torch.empty(rs.temp_bytes(n, 4, 0, 0, end, args.bits), dtype=torch.uint8,
                               device=dev)

            def sort():
                rs.radix_sort_keys(keys, ko, 0, end, args.bits, temp=temp)
        units = n
    elif args.case == "pairs_u64":
        keys = torch.from_numpy(workloads.u64_uniform(n, 0).view(np.int64)).to(dev)
        vals = torch.from_numpy(workloads.index_payload(n).view(np.int32)).to(dev)
        end = args.end_bit or 64
        ko, vo = torch.empty_like(keys), torch.empty_like(vals)
        temp = torch.empty(rs.temp_bytes(n, 8, 4, 0, end, args.bits), dtype=torch.uint8,
                           device=dev)

        def sort():
            rs.radix_sort_pairs(keys, vals, ko, vo, 0, end, args.bits, temp=temp)
        units = n
    else:
        kind = "f16" if args.case == "rows_f16" else "bf16"
        rows, cols = args.rows, args.cols
        x = torch.from_numpy(workloads.rows16(rows, cols, kind, 0).view(np.int16)).to(dev)
        x = x.view(torch.float16 if kind == "f16" else torch.bfloat16)
        v = torch.empty_like(x)
        idx = torch.empty((rows, cols), dtype=torch.int64, device=dev)
        temp = torch.empty(rs.segmented_temp_bytes(rows, cols), dtype=torch.uint8, device=dev)

        def sort():
            rs.segmented_sort(x, False, values_out=v, indices_out=idx, temp=temp)
        units = rows * cols

    for _ in range(args.warmup):
        sort()
    torch.cuda.synchronize()
    rs.profile_read()
    rs.profile_enable(True)
    for _ in range(args.sorts):
        sort()
    torch.cuda.synchronize()
    rs.profile_enable(False)
    per = {}
    for name, ms, _ in rs.profile_read():
        d = per.setdefault(name, [0, 0.0])
        d[0] += 1
        d[1] += ms
    status = rs.device_status(temp)
    out = {"case": args.case, "keys": units, "sorts": args.sorts, "status": status,
           "per_kernel_ms": {k: round(t / c, 5) for k, (c, t) in per.items()},
           "launches_per_sort": {k: c // args.sorts for k, (c, _) in per.items()},
           "ms_per_sort_sum_of_kernels": round(sum(t for _, t in per.values()) / args.sorts, 5)}
    print(json.dumps(out), flush=True)
    if status != 0:
        raise SystemExit(f"device status {status}")


if __name__ == "__main__":
    main()
