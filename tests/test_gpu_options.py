"""Per-call options, against the oracle.

Modes are options of the call that wants them (struct rs_options): two
callers in one process, on two streams, each get their own schedule, and
neither changes the other's."""
import numpy as np
import pytest
import torch

import oracle
from lsd_radix_sort_gb300 import workloads
from tests.gpu_util import assert_pairs, poisoned_like, to_dev, to_host

pytestmark = pytest.mark.gpu


def const_byte_keys(n, seed):
    """u32 keys whose bits 8..15 are constant: with pass skipping, 3 of 4 passes run."""
    return (workloads.u32_uniform(n, seed) & np.uint32(0xFFFF00FF)) | np.uint32(0x5A00)


def test_two_streams_two_modes(rs):
    n = 300_001
    ka, kb = const_byte_keys(n, 1), workloads.u32_uniform(n, 2)
    vals = workloads.index_payload(n)
    eka, eva = oracle.sort(ka, vals, 0, 32, 8)
    ekb, evb = oracle.sort(kb, vals, 0, 32, 8)
    dka, dkb, dv = to_dev(ka), to_dev(kb), to_dev(vals)
    ta = torch.empty(rs.temp_bytes(n, 4, 4, 0, 32, 8), dtype=torch.uint8, device="cuda")
    tb = torch.empty_like(ta)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    sa.wait_stream(torch.cuda.current_stream())
    sb.wait_stream(torch.cuda.current_stream())
    for _ in range(3):  # interleaved enqueues: neither call changes the other's mode
        with torch.cuda.stream(sa):
            koa, voa = poisoned_like(dka), poisoned_like(dv)
            rs.radix_sort_pairs(dka, dv, koa, voa, 0, 32, 8, temp=ta, pass_skipping=True,
                                small_sort=False)
        with torch.cuda.stream(sb):
            kob, vob = poisoned_like(dkb), poisoned_like(dv)
            rs.radix_sort_pairs(dkb, dv, kob, vob, 0, 32, 8, temp=tb)
    torch.cuda.synchronize()
    assert rs.passes_run(ta, stream=sa) == 3 and rs.passes_run(tb, stream=sb) == 4
    assert_pairs(to_host(koa, np.uint32), to_host(voa, np.uint32), eka, eva, "stream a")
    assert_pairs(to_host(kob, np.uint32), to_host(vob, np.uint32), ekb, evb, "stream b")


def test_two_streams_rows_offsets_and_lookback(rs):
    rows, cols = 40, 20_000
    h = workloads.rows16(rows, cols, "f16", seed=9)
    ev, ei = oracle.segmented_sort16(h, False)
    x = to_dev(h).view(torch.float16)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    sa.wait_stream(torch.cuda.current_stream())
    sb.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(sa):
        va, ia = rs.segmented_sort(x, False, tile_offsets=True)
    with torch.cuda.stream(sb):
        vb, ib = rs.segmented_sort(x, False)
    torch.cuda.synchronize()
    for v, i in ((va, ia), (vb, ib)):
        assert np.array_equal(to_host(v.view(torch.int16), np.uint16), ev)
        assert np.array_equal(i.cpu().numpy(), ei)
