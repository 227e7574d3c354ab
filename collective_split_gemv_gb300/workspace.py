"""Symmetric-slot workspaces for one GEMV + all-reduce (or all-reduce) shape.

A workspace allocates one handle whose user region holds, at the same offsets
in every rank's slot, ``copies`` instances of W_r (so that a timing loop can
rotate through more bytes than L2 holds), x_r and y, and stages host data into
and out of the slots with PyTorch copies.  With ``packed`` the instances of
W_r are packed weights (``symm_pack_w``), made from one row-major staging
copy.  The computation itself is the library call (``run``); PyTorch only
moves bytes.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (DeviceView, all_reduce_bias_rmsnorm, gemv_all_reduce, gemv_all_reduce_bias_rmsnorm,
               gemv_reduce_scatter, multi_root_tile_reduce, one_shot_all_reduce, reduce_scatter, symm_alloc,
               symm_free, symm_pack_w, symm_packed_w_bytes, symm_rendezvous, two_shot_all_reduce)

ALIGN = 256


def _up(v: int, a: int = ALIGN) -> int:
    return (v + a - 1) // a * a


def pad_bytes_for(N: int, min_rows: int = 8) -> int:
    """Signal pad that holds flags and counters for ceil(N / min_rows) tiles."""
    tiles = max(1, -(-N // min_rows))
    tiles = -(-tiles // 32) * 32
    return max(4096, 256 + 2 * _up(4 * tiles, 128) + 256)


class GemvWorkspace:
    def __init__(self, R: int, N: int, K: int, B: int, copies: int = 1, device: int | None = None,
                 packed: bool = False):
        if K % R:
            raise ValueError("K must be a multiple of R")
        self.R, self.N, self.K, self.B, self.Kr = R, N, K, B, K // R
        self.copies = copies
        self.packed = packed
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        self.w_bytes = N * self.Kr * 2
        self.wp_bytes = symm_packed_w_bytes(R, N, K) if packed else 0
        self.x_bytes = B * self.Kr * 2
        self.y_bytes = B * N * 2
        off = 0
        # row-major W_r: the instances, or (packed) the one staging copy
        self.w_off = []
        for _ in range(1 if packed else copies):
            self.w_off.append(off)
            off += _up(max(self.w_bytes, 1))
        self.wp_off = []
        for _ in range(copies if packed else 0):
            self.wp_off.append(off)
            off += _up(self.wp_bytes)
        self.x_off = off
        off += _up(max(self.x_bytes, 1))
        self.y_off = off
        off += _up(max(self.y_bytes, 1))
        # bias and gamma of the bias + RMSNorm form (N bf16 each)
        self.bias_off = off
        off += _up(max(N * 2, 1))
        self.gamma_off = off
        off += _up(max(N * 2, 1))
        self.slot_bytes = off
        # room for up to 8 partial arrays per rank (stream-K parts, K-splits),
        # plus the fp32 z of the bias + RMSNorm form
        self.scratch_bytes = _up(max(9 * 4 * B * N, 1))
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
        """W (R, N, K/R) bf16 words into instance `copy` (packed: through the
        staging copy, then symm_pack_w on the current stream)."""
        assert W.shape == (self.R, self.N, self.Kr) and W.dtype == np.uint16
        if self.w_bytes > 0:
            for r in range(self.R):
                self.w_view(r, 0 if self.packed else copy).copy_(self._bytes(W[r]))
        if self.packed:
            self.pack(copy)

    def pack(self, copy: int = 0, stream=None) -> None:
        """Packs the row-major staging copy into packed instance `copy`."""
        symm_pack_w(self.h, self.base + self.w_off[0], self.base + self.wp_off[copy], self.R, self.N, self.K,
                    torch.cuda.current_stream(self.device) if stream is None else stream)

    def load_x(self, x: np.ndarray) -> None:
        assert x.shape == (self.R, self.B, self.Kr) and x.dtype == np.uint16
        if self.x_bytes == 0:
            return
        for r in range(self.R):
            self.x_view(r).copy_(self._bytes(x[r]))

    def load_vectors(self, bias: np.ndarray | None, gamma: np.ndarray | None) -> None:
        """bias / gamma (N bf16 words each) into slot 0 (None leaves it unused)."""
        for vec, off in ((bias, self.bias_off), (gamma, self.gamma_off)):
            if vec is not None:
                assert vec.shape == (self.N,) and vec.dtype == np.uint16
                self.view(0, off, self.N * 2).copy_(self._bytes(vec))

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
        """Instance `copy` of W_r as the fused calls take it (packed or row-major)."""
        return self.base + (self.wp_off[copy] if self.packed else self.w_off[copy])

    def W_rowmajor_ptr(self) -> int:
        """The row-major W_r (packed workspaces: the staging copy)."""
        return self.base + self.w_off[0]

    def x_ptr(self) -> int:
        return self.base + self.x_off

    def y_ptr(self) -> int:
        return self.base + self.y_off

    def read_y_rs(self) -> np.ndarray:
        """(R, B/R, N) bf16 words: each rank's rows of a reduce-scatter."""
        torch.cuda.synchronize(self.device)
        Bs = self.B // self.R
        out = np.empty((self.R, Bs, self.N), dtype=np.uint16)
        for r in range(self.R):
            out[r] = self.view(r, self.y_off, Bs * self.N * 2).cpu().numpy().view(np.uint16).reshape(Bs, self.N)
        return out

    def run(self, stream=None, copy: int = 0, mode: str = "all_reduce", eps: float = 1e-6,
            bias: bool = True, gamma: bool = True) -> None:
        """One library call: ``all_reduce`` (gemv_all_reduce), ``reduce_scatter``
        (gemv_reduce_scatter) or ``bias_rmsnorm`` (gemv_all_reduce_bias_rmsnorm
        with the loaded bias / gamma, or NULL for either when False)."""
        if mode == "all_reduce":
            gemv_all_reduce(self.h, self.W_ptr(copy), self.x_ptr(), self.y_ptr(), self.R, self.N, self.K,
                            self.B, stream)
        elif mode == "reduce_scatter":
            gemv_reduce_scatter(self.h, self.W_ptr(copy), self.x_ptr(), self.y_ptr(), self.R, self.N, self.K,
                                self.B, stream)
        elif mode == "bias_rmsnorm":
            gemv_all_reduce_bias_rmsnorm(self.h, self.W_ptr(copy), self.x_ptr(),
                                         self.base + self.bias_off if bias else None,
                                         self.base + self.gamma_off if gamma else None, self.y_ptr(),
                                         self.R, self.N, self.K, self.B, eps, stream)
        else:
            raise ValueError(f"unknown mode {mode!r}")

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

    def read_out(self, copy: int = 0, count: int | None = None) -> np.ndarray:
        """(R, count) bf16 words of every rank's output (count defaults to n;
        n // R for a reduce-scatter)."""
        torch.cuda.synchronize(self.device)
        count = self.n if count is None else count
        out = np.empty((self.R, count), dtype=np.uint16)
        for r in range(self.R):
            out[r] = self.view(r, self._out(copy), count * 2).cpu().numpy().view(np.uint16)
        return out

    def run(self, stream=None, copy: int = 0, op: str = "one_shot") -> None:
        """One library call: ``one_shot``, ``two_shot`` or ``reduce_scatter``
        (output: the first n/R elements of each rank's out)."""
        fn = {"one_shot": one_shot_all_reduce, "two_shot": two_shot_all_reduce,
              "reduce_scatter": reduce_scatter}[op]
        fn(self.h, self.base + self.in_offs[copy], self.base + self._out(copy), self.R, self.n, stream)

    def close(self) -> None:
        if self.h is not None:
            symm_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class RmsNormWorkspace:
    """R slots holding `copies` inputs of rows x H bf16, one output per copy,
    and the bias / gamma vectors (H bf16) for all_reduce_bias_rmsnorm."""

    def __init__(self, R: int, rows: int, H: int, copies: int = 1, in_place: bool = False,
                 device: int | None = None):
        self.R, self.rows, self.H, self.copies = R, rows, H, copies
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        self.bytes = rows * H * 2
        per = _up(max(self.bytes, 1))
        self.in_offs = [c * per for c in range(copies)]
        self.out_offs = list(self.in_offs) if in_place else [(copies + c) * per for c in range(copies)]
        off = (copies if in_place else 2 * copies) * per
        self.bias_off = off
        self.gamma_off = off + _up(H * 2)
        self.slot_bytes = self.gamma_off + _up(H * 2)
        with torch.cuda.device(self.device):
            self.h = symm_alloc(R, self.slot_bytes, 0, 4096)
        self.slots, self.pads, self.stride = symm_rendezvous(self.h)
        self.base = self.slots[0]

    def view(self, rank: int, offset: int, nbytes: int) -> torch.Tensor:
        return torch.as_tensor(DeviceView(self.slots[rank] + offset, (nbytes,)), device=self.device)

    def load(self, inp: np.ndarray, bias: np.ndarray | None, gamma: np.ndarray | None, copy: int = 0) -> None:
        assert inp.shape == (self.R, self.rows, self.H) and inp.dtype == np.uint16
        for r in range(self.R):
            self.view(r, self.in_offs[copy], self.bytes).copy_(
                torch.from_numpy(np.ascontiguousarray(inp[r])).view(torch.uint8).reshape(-1))
        for vec, off in ((bias, self.bias_off), (gamma, self.gamma_off)):
            if vec is not None:
                self.view(0, off, self.H * 2).copy_(torch.from_numpy(np.ascontiguousarray(vec)).view(torch.uint8))

    def read_out(self, copy: int = 0) -> np.ndarray:
        torch.cuda.synchronize(self.device)
        out = np.empty((self.R, self.rows, self.H), dtype=np.uint16)
        for r in range(self.R):
            out[r] = self.view(r, self.out_offs[copy], self.bytes).cpu().numpy().view(np.uint16).reshape(
                self.rows, self.H)
        return out

    def run(self, stream=None, copy: int = 0, eps: float = 1e-6, bias: bool = True, gamma: bool = True) -> None:
        all_reduce_bias_rmsnorm(self.h, self.base + self.in_offs[copy], self.base + self.bias_off if bias else None,
                                self.base + self.gamma_off if gamma else None, self.base + self.out_offs[copy],
                                self.R, self.rows, self.H, eps, stream)

    def close(self) -> None:
        if self.h is not None:
            symm_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class TileWorkspace:
    """R slots, each holding `copies` full row-major input tensors of
    slot_rows x slot_cols bf16 (leading dimension slot_cols) and one output
    tensor of out_rows x out_cols (leading dimension out_cols) per copy, for
    tile_reduce / multi_root_tile_reduce."""

    def __init__(self, R: int, slot_rows: int, slot_cols: int, out_rows: int, out_cols: int, copies: int = 1,
                 device: int | None = None):
        self.R, self.slot_rows, self.slot_cols = R, slot_rows, slot_cols
        self.out_rows, self.out_cols, self.copies = out_rows, out_cols, copies
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        self.in_bytes = slot_rows * slot_cols * 2
        self.out_bytes = out_rows * out_cols * 2
        pin, pout = _up(max(self.in_bytes, 1)), _up(max(self.out_bytes, 1))
        self.in_offs = [c * pin for c in range(copies)]
        self.out_offs = [copies * pin + c * pout for c in range(copies)]
        self.slot_bytes = copies * (pin + pout)
        with torch.cuda.device(self.device):
            self.h = symm_alloc(R, self.slot_bytes, 0, 4096)
        self.slots, self.pads, self.stride = symm_rendezvous(self.h)
        self.base = self.slots[0]

    def view(self, rank: int, offset: int, nbytes: int) -> torch.Tensor:
        return torch.as_tensor(DeviceView(self.slots[rank] + offset, (nbytes,)), device=self.device)

    def load_in(self, full: np.ndarray, copy: int = 0) -> None:
        """full: (R, slot_rows, slot_cols) bf16 words."""
        assert full.shape == (self.R, self.slot_rows, self.slot_cols) and full.dtype == np.uint16
        for r in range(self.R):
            self.view(r, self.in_offs[copy], self.in_bytes).copy_(
                torch.from_numpy(np.ascontiguousarray(full[r])).view(torch.uint8).reshape(-1))

    def fill_out(self, words: np.ndarray, copy: int = 0) -> None:
        """words: (R, out_rows, out_cols) bf16 words written before the call."""
        for r in range(self.R):
            self.view(r, self.out_offs[copy], self.out_bytes).copy_(
                torch.from_numpy(np.ascontiguousarray(words[r])).view(torch.uint8).reshape(-1))

    def read_out(self, copy: int = 0) -> np.ndarray:
        torch.cuda.synchronize(self.device)
        out = np.empty((self.R, self.out_rows, self.out_cols), dtype=np.uint16)
        for r in range(self.R):
            out[r] = self.view(r, self.out_offs[copy], self.out_bytes).cpu().numpy().view(np.uint16).reshape(
                self.out_rows, self.out_cols)
        return out

    def run(self, tiles, roots, rows: int, cols: int, out_at=(0, 0), stream=None, copy: int = 0) -> None:
        """tiles: [(row0, col0)] of each input tile in the slot's tensor;
        the output tile starts at out_at of the output tensor."""
        ins = [self.base + self.in_offs[copy] + (a * self.slot_cols + b) * 2 for a, b in tiles]
        out = self.base + self.out_offs[copy] + (out_at[0] * self.out_cols + out_at[1]) * 2
        multi_root_tile_reduce(self.h, ins, out, roots, rows, cols, self.slot_cols, self.out_cols, stream)

    def close(self) -> None:
        if self.h is not None:
            symm_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
