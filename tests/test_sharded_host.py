"""Host side of the sharded paths on the CPU: the expert and vocabulary partitions, and the
exchange steps (all-to-all of counts and rows, all-gather of partials) run by two and three gloo
ranks on CPU tensors, checked against the rows and partials each rank must end up with."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from serve_invariant_moe_gb300 import sharded


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_expert_ranges():
    assert sharded.expert_ranges(256, 8) == [(32 * r, 32 * r + 32) for r in range(8)]
    assert sharded.expert_ranges(8, 1) == [(0, 8)]
    with pytest.raises(ValueError):
        sharded.expert_ranges(10, 4)


def test_vocab_shards_cut_at_chunk_boundaries():
    V = 151552                      # 592 chunks of 256
    P, sh = sharded.vocab_shards(V, 8)
    assert P == 74 and sh[0] == (0, 74 * 256) and sh[-1] == (7 * 74 * 256, V)
    for world in (1, 2, 3, 5, 7, 8, 600, 700):
        P, sh = sharded.vocab_shards(V, world)
        assert len(sh) == world
        assert sh[0][0] == 0 and max(v1 for _, v1 in sh) == V
        for (a0, a1), (b0, b1) in zip(sh[:-1], sh[1:]):
            assert a1 == b0 or (a1 == V and b0 == V)          # contiguous, empty shards at the end
        for v0, v1 in sh:
            assert v0 % 256 == 0 and (v1 % 256 == 0 or v1 == V) and v1 - v0 <= P * 256
    # a vocabulary that is not a multiple of the chunk: the last chunk is partial
    P, sh = sharded.vocab_shards(1000, 3)
    assert P == 2 and sh == [(0, 512), (512, 1000), (1000, 1000)]


def test_send_counts_view():
    counts = torch.arange(12, dtype=torch.int32)
    m = sharded.ep_send_counts(counts, 3)
    assert m.shape == (3, 4) and m[1].tolist() == [4, 5, 6, 7]
    with pytest.raises(ValueError):
        sharded.ep_send_counts(counts, 5)


def _rank_data(rank, world, E, H):
    """What rank `rank` holds before the exchange: per-expert row counts and its expert-sorted rows,
    each row tagged (source rank, expert, index within the expert) in its first three columns."""
    g = torch.Generator().manual_seed(100 + rank)
    counts = torch.randint(0, 4, (E,), generator=g, dtype=torch.int32)
    if rank == 0:
        counts[:E // world] = 0             # rank 0 sends nothing to rank 0's experts
    rows = []
    for e in range(E):
        for i in range(int(counts[e])):
            r = torch.zeros(H)
            r[0], r[1], r[2] = rank, e, i
            rows.append(r)
    xp = torch.stack(rows) if rows else torch.zeros((0, H))
    return counts, xp


def _exchange_worker(rank, world, port, E, H, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    coll = sharded.Collectives()
    counts, xp = _rank_data(rank, world, E, H)
    send_counts = sharded.ep_send_counts(counts, world)
    recv_counts = coll.exchange_counts(send_counts)
    send_splits, recv_splits = send_counts.sum(1).tolist(), recv_counts.sum(1).tolist()
    recv = coll.exchange_rows(xp, send_splits, recv_splits)
    # every owner returns its rows with column 3 marked, in the order received
    y_send = recv.clone()
    y_send[:, 3] = 1000 + rank
    back = coll.exchange_rows(y_send, recv_splits, send_splits)
    # vocabulary partials: rank r's [T, P, 2] block holds its rank in every entry
    T, P = 3, 5
    part = torch.full((T, P, 2), float(rank))
    gathered = coll.gather(part)
    out[rank] = dict(recv_counts=recv_counts.clone(), recv=recv.clone(), back=back.clone(), xp=xp.clone(),
                     gathered=gathered.clone())
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_gloo_exchange_of_rows_counts_and_partials(world):
    E, H = 6 * world, 8
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.start_processes(_exchange_worker, args=(world, port, E, H, out), nprocs=world, start_method="spawn", join=True)
    ranges = sharded.expert_ranges(E, world)
    data = [_rank_data(r, world, E, H) for r in range(world)]
    for d, (e0, e1) in enumerate(ranges):
        res = out[d]
        # counts: row s = what source s routed to each of d's experts
        want_counts = torch.stack([data[s][0][e0:e1] for s in range(world)])
        assert torch.equal(res["recv_counts"], want_counts)
        # rows: source-major, within a source expert by expert in the source's own order
        want = [(s, e, i) for s in range(world) for e in range(e0, e1) for i in range(int(data[s][0][e]))]
        got = [tuple(int(v) for v in row[:3]) for row in res["recv"]]
        assert got == want
    for s in range(world):
        res = out[s]
        # the reverse exchange brings every row back to the position it left from, marked by its owner
        assert torch.equal(res["back"][:, :3], res["xp"][:, :3])
        owner = [next(d for d, (e0, e1) in enumerate(ranges) if e0 <= int(e) < e1) for e in res["xp"][:, 1]]
        assert res["back"][:, 3].tolist() == [1000.0 + d for d in owner]
        # all-gather: block r from rank r, in rank order, on every rank
        assert [float(res["gathered"][r, 0, 0, 0]) for r in range(world)] == [float(r) for r in range(world)]
