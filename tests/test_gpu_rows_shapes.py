"""Row-wise 16-bit sorts on the shapes of the FlagTree PR #1084 H20 table
([64, 64] ... [8, 262144], last dimension), ascending and descending, with
the tile offsets found by the decoupled look-back and precomputed before
each pass: both are bit-exact with the oracle."""
import numpy as np
import pytest
import torch

import oracle
from lsd_radix_sort_gb300 import workloads

pytestmark = pytest.mark.gpu

H20_SHAPES = [(64, 64), (256, 256), (1024, 1024), (4096, 4096), (1024, 65536), (1024, 1),
              (1024, 512), (16, 131072), (8, 262144)]


@pytest.mark.parametrize("offsets_mode", [False, True], ids=["lookback", "precomputed"])
@pytest.mark.parametrize("shape", H20_SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
@pytest.mark.parametrize("descending", [False, True])
def test_h20_shapes(rs, offsets_mode, shape, descending):
    rows, cols = shape
    kind = "bf16" if rows * cols % 3 == 0 else "f16"
    h = workloads.rows16(rows, cols, kind, seed=rows + cols)
    x = torch.from_numpy(h.view(np.int16)).cuda()
    x = x.view(torch.bfloat16 if kind == "bf16" else torch.float16)
    v, i = rs.segmented_sort(x, descending, tile_offsets=offsets_mode)
    torch.cuda.synchronize()
    ev, ei = oracle.segmented_sort16(h, descending)
    assert np.array_equal(v.view(torch.int16).cpu().numpy().view(np.uint16), ev)
    assert np.array_equal(i.cpu().numpy(), ei)


def test_precomputed_in_place_and_ragged(rs):
    for rows, cols in ((3, 4097), (5, 12_345), (2, 1)):
        h = workloads.rows16(rows, cols, "f16", seed=cols)
        x = torch.from_numpy(h.view(np.int16)).cuda().view(torch.float16)
        v, i = rs.segmented_sort(x, False, values_out=x, tile_offsets=True)
        torch.cuda.synchronize()
        ev, ei = oracle.segmented_sort16(h, False)
        assert np.array_equal(v.view(torch.int16).cpu().numpy().view(np.uint16), ev)
        assert np.array_equal(i.cpu().numpy(), ei)
