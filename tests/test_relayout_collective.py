"""The seq->head regrouping IS the Ulysses all-to-all: run the collective on CPU
ranks (gloo, all_to_all_single) and compare every rank's result with the
oracle's local relayout.  This pins the oracle's index formula to a library
collective, and exercises the multi-rank form of the path without a GPU.

Pages: long-context-attention issue "关于数据分割和合并" (the all-to-all works
like a transpose: every rank ends with the full sequence for a subset of the
heads, and a second all-to-all brings the heads back) and transformers PR 31525
(sequence shards [b, s/p, n, h] enter the all-to-all).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, shards, queue):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        N = world
        x = torch.from_numpy(shards[rank].astype(np.int32))          # [b][s/N][h][d]
        b, sl, h, d = x.shape
        hl = h // N
        # seq -> head: send head group g to rank g, receive every rank's rows of my group
        send = x.reshape(b, sl, N, hl, d).permute(2, 0, 1, 3, 4).contiguous()
        recv = torch.empty_like(send)                                  # [src][b][s/N][hl][d]
        dist.all_to_all_single(recv, send)
        group = recv.permute(1, 0, 2, 3, 4).reshape(b, N * sl, hl, d)  # [b][s][hl][d]
        # head -> seq: the inverse exchange
        send2 = group.reshape(b, N, sl, hl, d).permute(1, 0, 2, 3, 4).contiguous()
        recv2 = torch.empty_like(send2)                                # [src group][b][s/N][hl][d]
        dist.all_to_all_single(recv2, send2)
        back = recv2.permute(1, 2, 0, 3, 4).reshape(b, sl, h, d)
        queue.put((rank, group.numpy(), back.numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,b,s,h,d", [(2, 1, 8, 4, 4), (4, 2, 16, 8, 2)])
def test_all_to_all_equals_oracle_relayout(orc, world, b, s, h, d):
    rng = np.random.default_rng(world)
    shards = rng.integers(0, 65536, size=(world, b, s // world, h, d)).astype(np.uint16)
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, shards, queue))
             for r in range(world)]
    for p in procs:
        p.start()
    results = {}
    for _ in range(world):
        rank, group, back = queue.get(timeout=120)
        results[rank] = (group, back)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    ref = orc.seq2head(shards, world, b, s, h, d)                   # [N][b][s][h/N][d]
    for r in range(world):
        group, back = results[r]
        assert np.array_equal(group.astype(np.uint16), ref[r]), f"rank {r} seq->head"
        assert np.array_equal(back.astype(np.uint16), shards[r]), f"rank {r} head->seq"
