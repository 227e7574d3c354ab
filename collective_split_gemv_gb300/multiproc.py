"""Multi-process handles: R processes, one rank each, sharing symmetric slots.

``mp_alloc`` is the rendezvous of the "PyTorch Symmetric Memory" docs for
this library: every process allocates its own slot (``symm_mp_alloc``, a CUDA
virtual-memory allocation exported as a POSIX file descriptor), the
descriptors are exchanged over Unix-domain sockets (``exchange_fds``, a
descriptor can only travel between processes that way), every process maps
its peers' slots (``symm_mp_import``), and ``symm_rendezvous`` then returns
the R slot pointers -- the same layout in every process, rank r's slot at
base + r * stride.

The process group (any ``torch.distributed`` backend, ``gloo`` on the CPU is
enough) only orders the steps with barriers; no tensor goes through it.
"""
from __future__ import annotations

import os
import socket
import struct

from . import symm_free, symm_mp_alloc, symm_mp_import, symm_rendezvous


def exchange_fds(rank: int, world: int, my_fd: int, sock_dir: str, barrier) -> dict:
    """Sends `my_fd` to every other rank and receives theirs.  Each rank
    listens on ``<sock_dir>/slot<rank>.sock``; ``barrier()`` (a process-group
    barrier) separates listening from connecting and the exchange from what
    follows.  Returns {peer rank: received descriptor}; the caller closes
    them (and `my_fd`) when it no longer needs them."""
    path = os.path.join(sock_dir, f"slot{rank}.sock")
    if os.path.exists(path):
        os.unlink(path)
    srv = socket.socket(socket.AF_UNIX, socket.SOCK_STREAM)
    try:
        srv.bind(path)
        srv.listen(max(1, world))
        barrier()                                   # every rank listens
        for q in range(world):
            if q == rank:
                continue
            with socket.socket(socket.AF_UNIX, socket.SOCK_STREAM) as c:
                c.connect(os.path.join(sock_dir, f"slot{q}.sock"))
                socket.send_fds(c, [struct.pack("<i", rank)], [my_fd])
        got = {}
        try:
            for _ in range(world - 1):
                conn, _ = srv.accept()
                with conn:
                    msg, fds, _, _ = socket.recv_fds(conn, 4, 1)
                    if len(msg) != 4 or len(fds) != 1:
                        for f in fds:
                            os.close(f)
                        raise RuntimeError("malformed descriptor message")
                    peer = struct.unpack("<i", msg)[0]
                    if peer in got or not 0 <= peer < world or peer == rank:
                        os.close(fds[0])
                        raise RuntimeError(f"unexpected descriptor from rank {peer}")
                    got[peer] = fds[0]
            barrier()                               # every rank has every descriptor
        except BaseException:
            for f in got.values():                  # none of them reaches the caller
                os.close(f)
            raise
        return got
    finally:
        srv.close()
        if os.path.exists(path):
            os.unlink(path)


def mp_alloc(R: int, rank: int, slot_bytes: int, scratch_bytes: int, signal_pad_bytes: int, sock_dir: str,
             barrier):
    """Multi-process handle of rank `rank`: own slot allocated, peers'
    slots mapped.  -> (handle, slot pointers, pad pointers, stride)."""
    h, fd = symm_mp_alloc(R, rank, slot_bytes, scratch_bytes, signal_pad_bytes)
    try:
        fds = exchange_fds(rank, R, fd, sock_dir, barrier)
        try:
            for peer, pfd in sorted(fds.items()):
                symm_mp_import(h, peer, pfd)
        finally:
            for pfd in fds.values():
                os.close(pfd)
    except BaseException:
        symm_free(h)
        raise
    finally:
        os.close(fd)
    slots, pads, stride = symm_rendezvous(h)
    return h, slots, pads, stride
