"""The Python binding refuses buffers the kernels would overrun, before any
launch: outputs of the wrong size or width, scratch too small.  The shape
checks come before the device checks, so they run on CPU tensors."""
import pytest
import torch

import lsd_radix_sort_gb300 as rs


def test_keys_output_size_and_width():
    keys = torch.zeros(100, dtype=torch.int32)
    with pytest.raises(ValueError, match="out must hold 100"):
        rs.radix_sort_keys(keys, torch.zeros(99, dtype=torch.int32))
    with pytest.raises(ValueError, match="out must hold 100"):
        rs.radix_sort_keys(keys, torch.zeros(100, dtype=torch.int16))
    with pytest.raises(ValueError, match="out must hold 100"):
        rs.radix_sort_keys(torch.zeros(100, dtype=torch.int64), torch.zeros(100, dtype=torch.int32))


def test_pairs_output_sizes():
    keys = torch.zeros(64, dtype=torch.int64)
    vals = torch.zeros(64, dtype=torch.int32)
    with pytest.raises(ValueError, match="keys_out"):
        rs.radix_sort_pairs(keys, vals, torch.zeros(64, dtype=torch.int32), torch.zeros_like(vals))
    with pytest.raises(ValueError, match="values_out"):
        rs.radix_sort_pairs(keys, vals, torch.zeros_like(keys), torch.zeros(63, dtype=torch.int32))
    with pytest.raises(ValueError, match="one per key"):
        rs.radix_sort_pairs(keys, torch.zeros(65, dtype=torch.int32))


def test_segmented_output_shapes():
    x = torch.zeros(4, 10, dtype=torch.float16)
    with pytest.raises(ValueError, match="values_out"):
        rs.segmented_sort(x, values_out=torch.zeros(4, 9, dtype=torch.float16))
    with pytest.raises(ValueError, match="values_out"):
        rs.segmented_sort(x, values_out=torch.zeros(4, 10, dtype=torch.float32))
    with pytest.raises(ValueError, match="indices_out"):
        rs.segmented_sort(x, indices_out=torch.zeros(4, 10, dtype=torch.int32))
    with pytest.raises(ValueError, match="indices_out"):
        rs.segmented_sort(x, indices_out=torch.zeros(40, dtype=torch.int64))


def test_cpu_tensors_are_refused():
    keys = torch.zeros(100, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        rs.radix_sort_keys(keys)
    with pytest.raises(ValueError, match="CUDA"):
        rs.radix_sort_pairs(keys, torch.zeros(100, dtype=torch.int32))
