"""Guard bytes around a tensor: the stand-in for a memory checker on a pool
where none can run.  The tensor is placed inside a larger byte buffer whose
bytes before and after it hold a fixed pattern; after a call, check() finds
any write outside the tensor, and unwritten() any element the call left
holding the pattern."""
from __future__ import annotations

import numpy as np

PATTERN = 0xA5
GUARD_BYTES = 4096  # keeps the tensor 16- and 256-byte aligned inside the buffer


class Guarded:
    def __init__(self, shape, dtype, device, guard: int = GUARD_BYTES):
        import torch
        elt = torch.empty((), dtype=dtype).element_size()
        self.nbytes = int(np.prod(shape)) * elt
        assert self.nbytes > 0
        self.guard = guard
        self.buf = torch.full((guard + self.nbytes + guard,), PATTERN, dtype=torch.uint8, device=device)
        self.t = self.buf[guard:guard + self.nbytes].view(dtype).view(tuple(shape))

    def check(self, what: str = ""):
        """Assert that no byte outside the tensor changed."""
        head = self.buf[:self.guard]
        tail = self.buf[self.guard + self.nbytes:]
        bad_head = int((head != PATTERN).sum())
        bad_tail = int((tail != PATTERN).sum())
        assert bad_head == 0 and bad_tail == 0, (
            f"{what}: {bad_head} guard bytes before and {bad_tail} after the tensor were overwritten")

    def unwritten(self) -> int:
        """Elements whose bytes all still hold the pattern."""
        b = self.buf[self.guard:self.guard + self.nbytes].view(-1, self.t.element_size())
        return int((b == PATTERN).all(dim=1).sum())
