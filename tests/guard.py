"""Guard canaries around device outputs (test-only).

`guarded(shape, dtype)` returns an output tensor that is a view into a larger
buffer whose margins (4096 elements before and after, so the view keeps the
buffer's 256-byte alignment) hold a fixed byte pattern and whose body is
poisoned with NaN; `intact()` checks that no launch wrote outside the view.
This stands in for a memory checker: an out-of-bounds store near an output
changes a canary.
"""

import torch

MARGIN = 4096
CANARY = 0xA5


class Guarded:
    def __init__(self, shape, dtype, device="cuda"):
        n = 1
        for s in shape:
            n *= int(s)
        self.n = n
        self.buf = torch.full((n + 2 * MARGIN,), float("nan"), dtype=dtype, device=device)
        raw = self.buf.view(torch.uint8)
        esz = self.buf.element_size()
        raw[: MARGIN * esz].fill_(CANARY)
        raw[(MARGIN + n) * esz:].fill_(CANARY)
        self.tensor = self.buf[MARGIN: MARGIN + n].view(*shape) if shape else self.buf[MARGIN: MARGIN + 1].view(())

    def intact(self) -> bool:
        raw = self.buf.view(torch.uint8)
        esz = self.buf.element_size()
        head = raw[: MARGIN * esz]
        tail = raw[(MARGIN + self.n) * esz:]
        return bool((head == CANARY).all().item()) and bool((tail == CANARY).all().item())


def guarded(shape, dtype):
    return Guarded(tuple(shape), dtype)
