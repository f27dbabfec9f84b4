"""Sentinel bands around the buffers a test hands to the library.

compute-sanitizer is not available on the GPU pool, so out-of-bounds stores
are caught by construction: every output, workspace and input buffer is
carved from a larger allocation with BAND bytes of a seeded byte pattern
before and after it.  ``check()`` verifies, after the calls, that the
bands are unchanged (nothing was written past either end) and that every
input still holds its original bytes (nothing was written into an input).
Outputs start filled with 0xFF bytes, which read as NaN in every float
dtype, so an element the kernels never write fails the parity comparison.

The tensor inside a guarded buffer starts ``BAND`` bytes after an
allocation that the caching allocator aligns to 512 bytes, so it keeps the
16-byte alignment the staged kernels need; ``misalign`` shifts it.
"""
from __future__ import annotations

import math
from typing import List, Tuple

import numpy as np
import torch

BAND = 256


def _pattern(n: int, seed: int) -> torch.Tensor:
    rng = np.random.default_rng(seed)
    return torch.from_numpy(rng.integers(0, 256, size=n, dtype=np.uint8))


class Guarded:
    """A set of guarded device (or host) buffers and their expected bands."""

    def __init__(self, device="cuda"):
        self.device = torch.device(device)
        self._bufs: List[Tuple[str, torch.Tensor, int, int, torch.Tensor, torch.Tensor]] = []
        self._inputs: List[Tuple[str, torch.Tensor, torch.Tensor]] = []
        self._seed = 1234

    def _raw(self, name: str, nbytes: int, misalign: int, fill: int, pin: bool = False) -> torch.Tensor:
        total = BAND + misalign + nbytes + BAND
        if self.device.type == "cpu":
            raw = torch.empty(total, dtype=torch.uint8, pin_memory=pin)
        else:
            raw = torch.empty(total, dtype=torch.uint8, device=self.device)
        self._seed += 1
        off = BAND + misalign
        pat = _pattern(off + BAND, self._seed)
        head, tail = pat[:off].clone(), pat[off:].clone()
        raw[:off].copy_(head)
        raw[off + nbytes:].copy_(tail)
        body = raw[off:off + nbytes]
        body.fill_(fill)
        self._bufs.append((name, raw, off, nbytes, head, tail))
        return body

    def empty(self, shape, dtype: torch.dtype, name: str, misalign: int = 0, pin: bool = False) -> torch.Tensor:
        """An output tensor of ``shape``, every byte 0xFF (NaN in float dtypes)."""
        es = torch.empty((), dtype=dtype).element_size()
        n = int(math.prod(shape)) * es
        body = self._raw(name, n, misalign, 0xFF, pin)
        return body.view(dtype).view(shape) if n else torch.empty(shape, dtype=dtype, device=body.device)

    def workspace(self, nbytes: int, name: str = "workspace", misalign: int = 0) -> torch.Tensor:
        """A uint8 workspace of ``nbytes`` whose contents on entry are the 0xFF fill."""
        return self._raw(name, nbytes, misalign, 0xFF)

    def copy_in(self, t: torch.Tensor, name: str, misalign: int = 0, pin: bool = False) -> torch.Tensor:
        """A guarded copy of input ``t`` (any device) that must stay unchanged."""
        out = self.empty(tuple(t.shape), t.dtype, name, misalign, pin)
        out.copy_(t)
        self._inputs.append((name, out, t.detach().to("cpu").clone()))
        return out

    def check(self) -> None:
        """Raises AssertionError if a band changed or an input was written."""
        if self.device.type == "cuda":
            torch.cuda.synchronize(self.device)
        bad = []
        for name, raw, off, n, before, after in self._bufs:
            head, tail = raw[:off].cpu(), raw[off + n:].cpu()
            if not torch.equal(head, before):
                i = int(torch.nonzero(head != before)[-1])
                bad.append(f"{name}: byte {i - off} (before the buffer) changed")
            if not torch.equal(tail, after):
                i = int(torch.nonzero(tail != after)[0])
                bad.append(f"{name}: byte {i} past its end changed")
        for name, t, ref in self._inputs:
            got = t.cpu().contiguous().reshape(-1).view(torch.uint8)
            if not torch.equal(got, ref.contiguous().reshape(-1).view(torch.uint8)):
                bad.append(f"input {name} was modified")
        assert not bad, "guard bands: " + "; ".join(bad)
