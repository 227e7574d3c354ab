"""The descriptor exchange of multi-process handles, on the CPU: gloo ranks
(separate processes) send one another the write end of a pipe through
multiproc.exchange_fds; each rank writes its name into every descriptor it
received, and every rank then finds all its peers' names in its own pipe --
so each received descriptor is the sender's object, not a copy or a number."""
from __future__ import annotations

import os
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import os, sys
    sys.path.insert(0, {root!r})
    import torch.distributed as dist
    from collective_split_gemv_gb300.multiproc import exchange_fds
    rank, world, tmp = int(sys.argv[1]), int(sys.argv[2]), sys.argv[3]
    dist.init_process_group("gloo", init_method="file://" + tmp + "/pg", rank=rank, world_size=world)
    rd, wr = os.pipe()
    got = exchange_fds(rank, world, wr, tmp, dist.barrier)
    assert sorted(got) == [q for q in range(world) if q != rank], got
    for peer, fd in got.items():
        os.write(fd, b"<%d>" % rank)
        os.close(fd)
    dist.barrier()
    os.close(wr)
    os.set_blocking(rd, False)
    data = os.read(rd, 4096)
    want = sorted(b"<%d>" % q for q in range(world) if q != rank)
    assert sorted(data.replace(b"><", b">|<").split(b"|")) == want, data
    dist.barrier()
    print("ok", rank)
""")


@pytest.mark.parametrize("world", [2, 3])
def test_descriptors_travel_between_processes(world, tmp_path):
    code = CHILD.format(root=ROOT)
    procs = [subprocess.Popen([sys.executable, "-c", code, str(r), str(world), str(tmp_path)],
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True) for r in range(world)]
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=120)
        except subprocess.TimeoutExpired:
            for q in procs:
                q.kill()
            raise
        outs.append((p.returncode, out, err))
    for r, (rc, out, err) in enumerate(outs):
        assert rc == 0 and f"ok {r}" in out, (r, rc, out, err[-2000:])


def test_a_descriptor_from_an_unexpected_rank_is_refused(tmp_path):
    """Rank 0 of 2 exchanges with a fake peer that claims to be rank 0 too:
    exchange_fds raises, and neither the descriptor it received nor any other
    stays open in this process."""
    import socket
    import struct
    import threading

    from collective_split_gemv_gb300.multiproc import exchange_fds

    peer_sock = socket.socket(socket.AF_UNIX, socket.SOCK_STREAM)
    peer_sock.bind(str(tmp_path / "slot1.sock"))
    peer_sock.listen(1)
    rd, wr = os.pipe()
    fake_rd, fake_wr = os.pipe()

    def fake_peer():
        conn, _ = peer_sock.accept()                # rank 0 sends its descriptor
        with conn:
            _, fds, _, _ = socket.recv_fds(conn, 4, 1)
            for f in fds:
                os.close(f)
        with socket.socket(socket.AF_UNIX, socket.SOCK_STREAM) as c:
            c.connect(str(tmp_path / "slot0.sock"))
            socket.send_fds(c, [struct.pack("<i", 0)], [fake_wr])   # the wrong rank

    t = threading.Thread(target=fake_peer)
    before = set(os.listdir("/proc/self/fd"))
    started = []

    def barrier():
        if not started:
            started.append(1)
            t.start()

    with pytest.raises(RuntimeError, match="unexpected descriptor"):
        exchange_fds(0, 2, wr, str(tmp_path), barrier)
    t.join(timeout=30)
    peer_sock.close()
    assert set(os.listdir("/proc/self/fd")) <= before | {str(fake_rd), str(fake_wr), str(rd), str(wr)}
    for f in (rd, wr, fake_rd, fake_wr):
        os.close(f)
