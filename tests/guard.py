"""Guard bands around device output buffers (a stand-in for a memory checker).

An output tensor is carved out of a larger byte buffer whose first and last
4 KiB hold a fixed pattern; after the call, both bands must still hold it.
A kernel that writes past either end of its output (by a row, a padded tile
or a stray index) changes the pattern and fails the check, on the GPU, with
no tool attached.
"""
import math

import torch

GUARD_BYTES = 4096
PATTERN = 0xA5


class Guarded:
    def __init__(self, shape, dtype, device, fill=None):
        itemsize = torch.empty((), dtype=dtype).element_size()
        self.nbytes = math.prod(shape) * itemsize
        self.raw = torch.full((self.nbytes + 2 * GUARD_BYTES,), PATTERN, dtype=torch.uint8, device=device)
        self.t = self.raw[GUARD_BYTES:GUARD_BYTES + self.nbytes].view(dtype).view(shape)
        if fill is not None:
            self.t.fill_(fill)

    def check(self, what="output"):
        lo = self.raw[:GUARD_BYTES]
        hi = self.raw[GUARD_BYTES + self.nbytes:]
        assert bool((lo == PATTERN).all()), f"{what}: guard band before the buffer was overwritten"
        assert bool((hi == PATTERN).all()), f"{what}: guard band after the buffer was overwritten"
