"""Symmetric-slot workspaces for one GEMV + all-reduce (or all-reduce) shape.

A workspace allocates one handle whose user region holds, at the same offsets
in every rank's slot, ``copies`` instances of W_r (so that a timing loop can
rotate through more bytes than L2 holds), x_r and y, and stages host data into
and out of the slots with PyTorch copies.  The computation itself is the
library call (``run``); PyTorch only moves bytes.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (DeviceView, gemv_all_reduce, one_shot_all_reduce, symm_alloc, symm_free,
               symm_rendezvous)

ALIGN = 256


def _up(v: int, a: int = ALIGN) -> int:
    return (v + a - 1) // a * a


def pad_bytes_for(N: int, min_rows: int = 8) -> int:
    """Signal pad that holds flags and counters for ceil(N / min_rows) tiles."""
    tiles = max(1, -(-N // min_rows))
    tiles = -(-tiles // 32) * 32
    return max(4096, 256 + 2 * _up(4 * tiles, 128) + 256)


class GemvWorkspace:
    def __init__(self, R: int, N: int, K: int, B: int, copies: int = 1, device: int | None = None):
        if K % R:
            raise ValueError("K must be a multiple of R")
        self.R, self.N, self.K, self.B, self.Kr = R, N, K, B, K // R
        self.copies = copies
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        self.w_bytes = N * self.Kr * 2
        self.x_bytes = B * self.Kr * 2
        self.y_bytes = B * N * 2
        off = 0
        self.w_off = []
        for _ in range(copies):
            self.w_off.append(off)
            off += _up(max(self.w_bytes, 1))
        self.x_off = off
        off += _up(max(self.x_bytes, 1))
        self.y_off = off
        off += _up(max(self.y_bytes, 1))
        self.slot_bytes = off
        # room for up to 8 partial arrays per rank (stream-K parts, K-splits)
        self.scratch_bytes = _up(max(8 * 4 * B * N, 1))
        self.pad_bytes = pad_bytes_for(N)
        with torch.cuda.device(self.device):
            self.h = symm_alloc(R, self.slot_bytes, self.scratch_bytes, self.pad_bytes)
        self.slots, self.pads, self.stride = symm_rendezvous(self.h)
        self.base = self.slots[0]

    # ------------------------------------------------------------- views
    def view(self, rank: int, offset: int, nbytes: int) -> torch.Tensor:
        return torch.as_tensor(DeviceView(self.slots[rank] + offset, (nbytes,)), device=self.device)

    def w_view(self, rank: int, copy: int = 0) -> torch.Tensor:
        return self.view(rank, self.w_off[copy], self.w_bytes)

    def x_view(self, rank: int) -> torch.Tensor:
        return self.view(rank, self.x_off, self.x_bytes)

    def y_view(self, rank: int) -> torch.Tensor:
        return self.view(rank, self.y_off, self.y_bytes)

    # ----------------------------------------------------------- staging
    @staticmethod
    def _bytes(a: np.ndarray) -> torch.Tensor:
        return torch.from_numpy(np.ascontiguousarray(a)).view(torch.uint8).reshape(-1)

    def load_W(self, W: np.ndarray, copy: int = 0) -> None:
        assert W.shape == (self.R, self.N, self.Kr) and W.dtype == np.uint16
        if self.w_bytes == 0:
            return
        for r in range(self.R):
            self.w_view(r, copy).copy_(self._bytes(W[r]))

    def load_x(self, x: np.ndarray) -> None:
        assert x.shape == (self.R, self.B, self.Kr) and x.dtype == np.uint16
        if self.x_bytes == 0:
            return
        for r in range(self.R):
            self.x_view(r).copy_(self._bytes(x[r]))

    def fill_y(self, byte: int) -> None:
        for r in range(self.R):
            self.y_view(r).fill_(byte)

    def read_y(self) -> np.ndarray:
        """(R, B, N) bf16 words from every rank's output slot."""
        torch.cuda.synchronize(self.device)
        out = np.empty((self.R, self.B, self.N), dtype=np.uint16)
        for r in range(self.R):
            out[r] = self.y_view(r).cpu().numpy().view(np.uint16).reshape(self.B, self.N)
        return out

    # --------------------------------------------------------------- run
    def W_ptr(self, copy: int = 0) -> int:
        return self.base + self.w_off[copy]

    def x_ptr(self) -> int:
        return self.base + self.x_off

    def y_ptr(self) -> int:
        return self.base + self.y_off

    def run(self, stream=None, copy: int = 0) -> None:
        gemv_all_reduce(self.h, self.W_ptr(copy), self.x_ptr(), self.y_ptr(), self.R, self.N, self.K,
                        self.B, stream)

    def close(self) -> None:
        if self.h is not None:
            symm_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class AllReduceWorkspace:
    """R slots holding `copies` input arrays of n bf16 and one output array
    (or, in place, each input array is its own output)."""

    def __init__(self, R: int, n: int, device: int | None = None, separate_out: bool = True, copies: int = 1):
        self.R, self.n, self.copies = R, n, copies
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        self.bytes = n * 2
        per = _up(max(self.bytes, 1))
        # copy c: input at in_offs[c], output at out_offs[c] (its own region, or
        # the input itself in place) -- rotating both keeps writes out of L2 too
        self.in_offs = [c * per for c in range(copies)]
        self.in_off = self.in_offs[0]
        self.separate_out = separate_out
        self.out_offs = [(copies + c) * per for c in range(copies)] if separate_out else list(self.in_offs)
        self.out_off = self.out_offs[0]
        self.slot_bytes = (2 * copies if separate_out else copies) * per
        with torch.cuda.device(self.device):
            self.h = symm_alloc(R, self.slot_bytes, 0, 4096)
        self.slots, self.pads, self.stride = symm_rendezvous(self.h)
        self.base = self.slots[0]

    def _out(self, copy: int) -> int:
        return self.out_offs[copy]

    def view(self, rank: int, offset: int, nbytes: int) -> torch.Tensor:
        return torch.as_tensor(DeviceView(self.slots[rank] + offset, (nbytes,)), device=self.device)

    def in_view(self, rank: int, copy: int = 0) -> torch.Tensor:
        return self.view(rank, self.in_offs[copy], self.bytes)

    def out_view(self, rank: int, copy: int = 0) -> torch.Tensor:
        return self.view(rank, self._out(copy), self.bytes)

    def load_in(self, inp: np.ndarray, copy: int = 0) -> None:
        assert inp.shape == (self.R, self.n) and inp.dtype == np.uint16
        if self.bytes == 0:
            return
        for r in range(self.R):
            self.in_view(r, copy).copy_(torch.from_numpy(np.ascontiguousarray(inp[r])).view(torch.uint8))

    def read_out(self, copy: int = 0) -> np.ndarray:
        torch.cuda.synchronize(self.device)
        out = np.empty((self.R, self.n), dtype=np.uint16)
        for r in range(self.R):
            out[r] = self.out_view(r, copy).cpu().numpy().view(np.uint16)
        return out

    def run(self, stream=None, copy: int = 0) -> None:
        one_shot_all_reduce(self.h, self.base + self.in_offs[copy], self.base + self._out(copy), self.R, self.n,
                            stream)

    def close(self) -> None:
        if self.h is not None:
            symm_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
