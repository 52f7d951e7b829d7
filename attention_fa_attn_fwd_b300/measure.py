"""L2 flush used between timed kernels (bench.py and its --case runs).

``L2Flush()`` writes a 256 MiB buffer (twice the 126 MB L2), which evicts
every line a timed kernel could reuse, and then reads a second 256 MiB
buffer, so the lines left in L2 are clean: the next timed kernel neither hits
on its own inputs nor pays for writing back the flush's dirty lines.  Both
steps are torch kernels on the current stream, issued outside the CUDA events
that bracket the timed kernel.
"""

from __future__ import annotations

import torch

FLUSH_BYTES = 256 << 20


class L2Flush:
    def __init__(self, device):
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)

    launches = 2  # torch kernels per flush (not this library's)
