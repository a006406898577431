"""The guard-byte helper of the device tests, checked on the host: it sees a
write one byte before or after its view, and none inside."""

import pytest
import torch

from helpers import GUARD, Guarded


@pytest.mark.parametrize("dtype", [torch.uint8, torch.bfloat16, torch.float32, torch.int32])
def test_view_is_aligned_and_inside_writes_pass(dtype):
    g = Guarded((37, 5), dtype, "cpu", fill=0)
    assert g.t.shape == (37, 5) and g.t.data_ptr() % 256 == g.raw.data_ptr() % 256
    g.t.fill_(1)
    g.check("inside")


@pytest.mark.parametrize("offset", [-1, 0])
def test_a_write_past_either_end_is_caught(offset):
    g = Guarded(12, torch.float32, "cpu", fill=0)
    pos = GUARD + offset if offset < 0 else GUARD + g.nbytes + offset
    g.raw[pos] = 0
    with pytest.raises(AssertionError, match="guard bytes changed"):
        g.check("planted")
