"""The data-parallel decode split over two ranks (gloo on CPU, no GPU): each
rank builds its own shard of sequences with the benchmark's per-rank seeding,
runs the oracle's decode step (insert, q-quant, paged logits, top-k) on its
shard alone, and rank 0 checks that every shard's top-k equals what one
process computes over both shards' sequences as a single batch.  So a rank
needs no other rank's data: the split is self-contained, and the only
collective the benchmark uses is for timing."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SIZES = dict(B=3, lo=2100, hi=4500)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _decode_topk(oracle, wl, p):
    cache = wl.poisoned_cache(p.num_blocks)
    oracle.quant_insert(p.k, p.slots, cache)
    qv, qs = oracle.quant_q(p.q)
    ld = p.block_table.shape[1] * 64
    lg, _ = oracle.paged_mqa_logits(qv, qs, p.B, p.next_n, p.H, cache, p.block_table,
                                    p.context_lens, p.weights, ld)
    st, en = p.row_windows()
    return oracle.topk_rows(np.nan_to_num(lg, nan=-np.inf), st, en, p.topk)


def _merged(wl, shards):
    """One batch holding every shard's sequences: pages renumbered into one
    cache, rows concatenated in rank order."""
    mb = max(p.block_table.shape[1] for p in shards)
    bts, ks, slots, qs, ws, lens = [], [], [], [], [], []
    base = 0
    for p in shards:
        bt = np.full((p.B, mb), -1, np.int32)
        bt[:, :p.block_table.shape[1]] = np.where(p.block_table >= 0, p.block_table + base, -1)
        bts.append(bt)
        ks.append(p.k)
        slots.append(p.slots + base * 64)
        qs.append(p.q)
        ws.append(p.weights)
        lens.append(p.context_lens)
        base += p.num_blocks
    lens = np.concatenate(lens)
    offs = np.zeros(len(lens) + 1, np.int64)
    offs[1:] = np.cumsum(lens.astype(np.int64))
    p0 = shards[0]
    return wl.DecodeProblem("merged", len(lens), p0.next_n, p0.H, 64, lens, np.concatenate(bts),
                            base, np.concatenate(ks), offs, np.concatenate(slots),
                            np.concatenate(qs), np.concatenate(ws), p0.topk)


def _rank_main(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    try:
        import bench
        import oracle
        from sparse_attention_indexer_quant_gb300 import workloads as wl
        dist.init_process_group("gloo", rank=rank, world_size=world)
        p = bench.make_workload("batched_decode", rank, **SIZES)
        top = _decode_topk(oracle, wl, p)
        got = [None] * world
        dist.all_gather_object(got, (p, top))
        if rank == 0:
            shards = [g[0] for g in got]
            whole = _decode_topk(oracle, wl, _merged(wl, shards))
            r0 = 0
            for s, (ps, ts) in enumerate(got):
                assert not np.array_equal(ps.k[:64], got[1 - s][0].k[:64]), "shards must differ"
                assert np.array_equal(whole[r0:r0 + ps.rows], ts), f"shard {s} differs"
                r0 += ps.rows
        dist.barrier()
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, repr(e)))


def test_two_rank_decode_shards_are_self_contained(oracle):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    res = dict(q.get(timeout=300) for _ in procs)
    for pr in procs:
        pr.join(timeout=60)
    assert res == {0: "ok", 1: "ok"}, res
