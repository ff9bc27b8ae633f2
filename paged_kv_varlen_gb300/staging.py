"""One pinned host buffer and one device buffer for a step's input arrays.

A serving step hands the device several small arrays: the packed queries, the
new K/V rows, the slot mapping, cu_seqlens_q, seq_lens_k and the block tables.
Copied one by one, each costs a copy launch on the stream; packed into one
pinned staging buffer they cross in a single copy.  The device side is one
buffer too, cut into views at 256-byte aligned offsets (the kernels' TMA
descriptors and 16-byte vector loads need 16-byte aligned rows).

Host-side plumbing only: nothing here touches the attention arithmetic.
"""
from __future__ import annotations

from typing import Dict

import torch

ALIGN = 256


class StepStaging:
    """Pinned host views and device views of the arrays named in ``like``
    (name -> tensor giving shape and dtype), packed in that order.

    Fill ``host[name]`` with a step's inputs, call ``upload()`` (one
    host-to-device copy on the current stream), then pass ``dev[name]`` to the
    attention calls.
    """

    def __init__(self, like: Dict[str, torch.Tensor], device: torch.device):
        layout = {}
        off = 0
        for name, t in like.items():
            off = (off + ALIGN - 1) // ALIGN * ALIGN
            nbytes = t.numel() * t.element_size()
            layout[name] = (off, nbytes, tuple(t.shape), t.dtype)
            off += nbytes
        self.nbytes = max(off, 1)
        self.host_buffer = torch.empty(self.nbytes, dtype=torch.uint8).pin_memory()
        self.dev_buffer = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        self.host = {n: _view(self.host_buffer, *v) for n, v in layout.items()}
        self.dev = {n: _view(self.dev_buffer, *v) for n, v in layout.items()}

    def upload(self) -> None:
        """One asynchronous host-to-device copy of every packed array."""
        self.dev_buffer.copy_(self.host_buffer, non_blocking=True)


def _view(buf: torch.Tensor, off: int, nbytes: int, shape, dtype) -> torch.Tensor:
    return buf[off:off + nbytes].view(dtype).view(shape)
