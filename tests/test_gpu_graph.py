"""A sort is a fixed sequence of launches on one stream with no host
synchronisation and no allocation, so a call captures into a CUDA graph
(CUDA Handbook ch. 16, the graph version of the sort's launches) and the
graph replays it on whatever the captured buffers hold."""
import numpy as np
import pytest
import torch

import oracle
from lsd_radix_sort_gb300 import workloads

pytestmark = pytest.mark.gpu


def capture(fn):
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        fn()
    stream.wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("n", [1000, 70_001])
@pytest.mark.parametrize("skipping", [False, True])
def test_graph_replay_sorts_new_inputs(rs, n, skipping):
    dk = torch.empty(n, dtype=torch.int32, device="cuda")
    dv = torch.empty(n, dtype=torch.int32, device="cuda")
    ko, vo = torch.empty_like(dk), torch.empty_like(dv)
    temp = torch.empty(rs.temp_bytes(n, 4, 4, 0, 32, 8), dtype=torch.uint8, device="cuda")
    dk.copy_(torch.from_numpy(workloads.u32_uniform(n, 0).view(np.int32)))
    dv.copy_(torch.from_numpy(workloads.index_payload(n).view(np.int32)))
    g = capture(lambda: rs.radix_sort_pairs(dk, dv, ko, vo, 0, 32, 8, temp=temp,
                                            pass_skipping=skipping))
    for seed, dist in ((1, "uniform"), (2, "low_entropy"), (3, "all_equal"), (4, "sorted")):
        keys = workloads.U32_DISTRIBUTIONS[dist](n, seed)
        vals = workloads.index_payload(n)
        dk.copy_(torch.from_numpy(keys.view(np.int32)))
        g.replay()
        torch.cuda.synchronize()
        ek, ev = oracle.sort(keys, vals, 0, 32, 8)
        assert np.array_equal(ko.cpu().numpy().view(np.uint32), ek), dist
        assert np.array_equal(vo.cpu().numpy().view(np.uint32), ev), dist


def test_graph_replay_rows(rs):
    rows, cols = 8, 5000
    x = torch.empty((rows, cols), dtype=torch.float16, device="cuda")
    vals = torch.empty_like(x)
    idx = torch.empty((rows, cols), dtype=torch.int64, device="cuda")
    temp = torch.empty(rs.segmented_temp_bytes(rows, cols), dtype=torch.uint8, device="cuda")
    x.copy_(torch.from_numpy(workloads.rows16(rows, cols, "f16", 0).view(np.float16)))
    g = capture(lambda: rs.segmented_sort(x, True, vals, idx, temp))
    for seed in (1, 2):
        h = workloads.rows16(rows, cols, "f16", seed)
        x.copy_(torch.from_numpy(h.view(np.float16)))
        g.replay()
        torch.cuda.synchronize()
        ev, ei = oracle.segmented_sort16(h, True)
        assert np.array_equal(vals.cpu().numpy().view(np.uint16), ev)
        assert np.array_equal(idx.cpu().numpy(), ei)
