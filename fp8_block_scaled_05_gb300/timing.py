"""Timing helpers shared by the benchmarks."""
from __future__ import annotations

import torch


class L2Flush:
    """Evicts the GPU's L2 (129 MB on GB300) between timed launches.

    A 256 MB write replaces every cached line, so nothing the next launch
    reads is still in L2; a 256 MB read of a second buffer then replaces the
    write's dirty lines with clean ones, so the timed launch does not pay for
    writing the flush's data back to HBM (up to the whole L2, which is about
    20 us of DRAM writes).  Runs on the current stream, outside the timed
    events."""

    def __init__(self, device, nbytes: int = 256 << 20):
        self.w = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.r = torch.zeros(nbytes // 4, dtype=torch.float32, device=device)
        self.acc = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self) -> None:
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.acc)
