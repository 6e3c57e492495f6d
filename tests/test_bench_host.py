"""Host-side logic of bench.py: byte accounting, the reference arm's JSON
line, and the max-over-ranks time of N replicas (two gloo ranks on CPU)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from tests.conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_ideal_bytes():
    n = 1 << 28
    # one read of the keys, then per pass a read and a write of keys+payloads
    assert bench.ideal_bytes(n, 4, 4, 4) == 68 * n
    assert bench.ideal_bytes(n, 8, 8, 4) == 200 * n          # u64 pairs, 8 passes
    assert bench.ideal_bytes(n, 5, 8, 4) == 128 * n          # u64 pairs, bits 0-39
    assert bench.ideal_bytes(4_194_304, 8, 4, 0) == 68 * 4_194_304
    assert bench.sweep_bytes_per_launch(n, 4, 4) == 16 * n


def test_context_numbers_from_the_pages():
    # day 35: 4,194,915 keys pad to 128 blocks x 129 tiles x 256 = 4,227,072;
    # a pass moves 3 x 16,908,288 B = 48.4 MiB; bitonic on 2^23 takes 23*24/2 rounds
    assert 128 * 129 * 256 == 4_227_072
    assert 4_227_072 * 4 == 16_908_288
    assert abs(3 * 16_908_288 / 2**20 - 48.4) < 0.05
    assert 23 * 24 // 2 == 276


def test_reference_arm_json_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3", "--ref-log2", "12"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "Gkeys/s"
    assert line["metric"] == bench.METRIC and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["steps"] == 2 and line["warmup"] == 3


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--ref-log2", "10"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        import bench as b
        slowest = b.max_over_ranks(1.5 + rank, world)
        b.barrier(world)
        q.put((rank, slowest))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert [v for _, v in got] == [1.5 + world - 1] * world


def test_result_checks_accept_the_oracle_and_reject_a_broken_tie():
    """The device-side result checks bench.py applies to its larger workloads
    (payload gather, order of the transformed key, ties in input order),
    run on CPU tensors: the oracle's stable sort passes, the same result
    with two tied payloads swapped fails, for every key type they cover."""
    import numpy as np
    import torch
    import oracle
    from lsd_radix_sort_gb300 import workloads
    n = 5000
    k = workloads.u32_uniform(n, 3)
    k[::7] = k[1]
    v = workloads.index_payload(n)
    for kt, desc in (("u32", False), ("f32", False), ("f32", True), ("i32", False)):
        arr = k.view(np.float32) if kt == "f32" else (k.view(np.int32) if kt == "i32" else k)
        ek, ev = oracle.sort_typed(arr, kt, v, desc)
        kin = torch.from_numpy(k.view(np.int32))
        ko = torch.from_numpy(np.ascontiguousarray(ek).view(np.int32))
        vo = torch.from_numpy(ev.view(np.int32))
        order = bench._order_key(torch, ko, kt, desc)
        assert bench._check_sorted_pairs(torch, kin, ko, vo, None, order)
        j = int(torch.nonzero(order[1:] == order[:-1])[0])
        bad = vo.clone()
        bad[j], bad[j + 1] = vo[j + 1].item(), vo[j].item()
        assert not bench._check_sorted_pairs(torch, kin, ko, bad, None, order)
    k64 = workloads.u64_skewed(n, 0)
    for end in (64, 40):
        ek, ev = oracle.sort(k64, v, 0, end, 8)
        ko = torch.from_numpy(ek.view(np.int64))
        key = ko if end == 64 else ko & ((1 << end) - 1)
        order = bench._order_key(torch, key, "u64" if end == 64 else "i64")
        assert bench._check_sorted_pairs(torch, torch.from_numpy(k64.view(np.int64)), ko,
                                         torch.from_numpy(ev.view(np.int32)), None, order)


def test_kernel_hash_ignores_comments_only():
    """The traffic record stays valid across comment edits of the kernel
    sources and is dropped when the code changes."""
    src = "int f(int x) {  // twice\n  /* the\n value */ return 2 * x;\n}\n"
    assert bench.code_only(src) == bench.code_only(src.replace("twice", "two times"))
    assert bench.code_only(src) != bench.code_only(src.replace("2 * x", "3 * x"))
    files = {name: src for name in bench.SWEEP_SOURCES}
    h = bench.onesweep_source_hash(lambda name: files[name])
    files["kernels.h"] = src.replace("// twice", "// doubled")
    assert bench.onesweep_source_hash(lambda name: files[name]) == h
    files["kernels.h"] = src.replace("return", "return 1 +")
    assert bench.onesweep_source_hash(lambda name: files[name]) != h
