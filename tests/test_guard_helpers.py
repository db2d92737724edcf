"""The guard-byte helper itself, on CPU tensors: it must see a write one byte
past either end of the tensor, and count elements a call left unwritten."""
import pytest
import torch

from guard_helpers import Guarded


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.uint8, torch.int32])
def test_guard_detects_writes_past_either_end(dtype):
    g = Guarded((3, 5, 8), dtype, "cpu")
    assert g.t.data_ptr() % 256 == g.buf.data_ptr() % 256  # same alignment as the buffer
    assert g.unwritten() == 3 * 5 * 8
    g.t.zero_()
    g.check("inside only")
    assert g.unwritten() == 0
    g.buf[g.guard - 1] = 0
    with pytest.raises(AssertionError):
        g.check("before")
    g.buf[g.guard - 1] = 0xA5
    g.buf[g.guard + g.nbytes] = 1
    with pytest.raises(AssertionError):
        g.check("after")


def test_unwritten_counts_whole_elements():
    g = Guarded((4, 4), torch.float32, "cpu")
    g.t[0].fill_(1.0)
    g.t[1, 0] = 2.0
    assert g.unwritten() == 16 - 5
