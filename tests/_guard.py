"""Guarded output buffers for the GPU parity tests.

Each output is a view into a larger device buffer: the output region starts filled with NaN
(so an element the kernel never writes fails the finiteness check in tests._parity.check),
and 4096 elements on each side hold a canary value that must survive the call (a write
outside the output's extent changes it).
"""
import math

import torch

PAD = 4096
CANARY = 1234.5  # exactly representable in bf16, fp16 and fp32


class Guarded:
    def __init__(self, shape, dtype, device="cuda"):
        n = math.prod(shape)
        self.shape = tuple(shape)
        self.buf = torch.full((n + 2 * PAD,), float("nan"), dtype=dtype, device=device)
        self.buf[:PAD] = CANARY
        self.buf[PAD + n:] = CANARY
        self.view = self.buf[PAD:PAD + n].view(self.shape)

    def assert_intact(self, what=""):
        head, tail = self.buf[:PAD], self.buf[-PAD:]
        assert bool((head == CANARY).all()) and bool((tail == CANARY).all()), \
            f"{what}: a write landed outside the output"


def guarded_outputs(out_shape, out_dtype, lse_shape, device="cuda"):
    """(out guard, lse guard); lse is fp32."""
    return Guarded(out_shape, out_dtype, device), Guarded(lse_shape, torch.float32, device)
