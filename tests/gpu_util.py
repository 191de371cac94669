"""Helpers shared by the GPU tests: guard-banded device buffers and bit views."""
import numpy as np
import torch

GUARD = 4096
SENTINEL = 0xA5


class Guarded:
    """A device tensor with GUARD bytes of a sentinel pattern before and after
    it; ``intact()`` checks that no kernel wrote outside the tensor."""

    def __init__(self, shape, dtype, device="cuda", fill_nan=True):
        self.shape = tuple(shape)
        esize = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(self.shape)) * esize
        self.raw = torch.full((GUARD + n + GUARD,), SENTINEL, dtype=torch.uint8, device=device)
        self.n = n
        body = self.raw[GUARD:GUARD + n]
        if fill_nan:
            body.fill_(0xFF)  # 0xFFFF is a NaN in bf16 and fp16
        self.t = body.view(dtype).view(self.shape)

    def intact(self) -> bool:
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.n:]
        return bool((head == SENTINEL).all().item() and (tail == SENTINEL).all().item())


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
