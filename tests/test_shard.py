"""Partition of a batch of queries across ranks (sparse_paged_attention_gb300.shard), on the CPU.

* every query lands in exactly one shard, sequences stay whole, query blocks are dealt round-robin;
* a batch of independent workloads (workloads.concat_batch) computes, per query, what each part
  computes alone (the oracle, bit for bit);
* two gloo ranks each compute only their shard; rank 0 gathers the shards and gets the whole
  batch's output bit for bit, with no exchange on the data path (the gather is the test's check).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from oracle_io import oracle_args
import oracle
from sparse_paged_attention_gb300.shard import shard_tokens
from workloads import build, concat_batch


def _part(seed):
    # 24 prefill queries near position 300, 4 heads, head_dim 64, window 16, top-k 24 (ratio 4)
    return build(f"part{seed}", seq_positions=[np.arange(290, 314)], num_heads=4, head_dim=64,
                 window=16, topk=24, ratio=4, page_size=16, seed=seed)


def _oracle(w, toks=None):
    a = oracle_args(w)
    if toks is not None:
        for k in ("q_bits", "positions", "seq_ids", "topk_idx"):
            a[k] = a[k][toks]
    out, lse, _, err = oracle.sparse_paged_attention(**a)
    assert not err
    return out, lse


@pytest.mark.parametrize("by", ["sequence", "query_block"])
@pytest.mark.parametrize("world", [1, 2, 3, 5])
def test_every_query_in_exactly_one_shard(by, world):
    sot = np.repeat(np.arange(7), [3, 1, 4, 1, 5, 9, 2])
    parts = [shard_tokens(len(sot), sot, r, world, by=by, block=4) for r in range(world)]
    allidx = np.concatenate(parts)
    assert np.array_equal(np.sort(allidx), np.arange(len(sot)))
    for p in parts:
        assert np.all(np.diff(p) > 0)
        if by == "sequence" and len(p):
            seqs = np.unique(sot[p])
            assert np.array_equal(np.sort(p), np.nonzero(np.isin(sot, seqs))[0])   # whole sequences
    if by == "query_block":
        for r, p in enumerate(parts):
            assert np.all((p // 4) % world == r)


def test_shard_rejects_bad_arguments():
    with pytest.raises(ValueError):
        shard_tokens(10, None, 2, 2)
    with pytest.raises(ValueError):
        shard_tokens(10, None, 0, 1, by="heads")
    with pytest.raises(ValueError):
        shard_tokens(10, None, 0, 2, by="query_block", block=0)


def test_batch_computes_what_each_part_computes_alone():
    parts = [_part(s) for s in range(3)]
    batch = concat_batch(parts)
    out_b, lse_b = _oracle(batch)
    T = parts[0].num_tokens
    for s, w in enumerate(parts):
        out_p, lse_p = _oracle(w)
        assert np.array_equal(out_b[s * T:(s + 1) * T], out_p)
        assert np.array_equal(lse_b[s * T:(s + 1) * T], lse_p)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, by, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    batch = concat_batch([_part(s) for s in range(2)])
    idx = shard_tokens(batch.num_tokens, batch.seq_ids(), rank, world, by=by, block=8)
    out, lse = _oracle(batch, idx)
    # the check only: every rank's shard (indices and outputs) to rank 0
    got = [None] * world
    dist.all_gather_object(got, (idx, out, lse))
    if rank == 0:
        full_out, full_lse = _oracle(batch)
        asm_out = np.zeros_like(full_out)
        asm_lse = np.zeros_like(full_lse)
        seen = np.zeros(batch.num_tokens, dtype=int)
        for i, o, l in got:
            asm_out[i], asm_lse[i] = o, l
            seen[i] += 1
        q.put((bool(np.all(seen == 1)), bool(np.array_equal(asm_out, full_out)),
               bool(np.array_equal(asm_lse, full_lse))))
    dist.destroy_process_group()


@pytest.mark.parametrize("by", ["sequence", "query_block"])
def test_two_ranks_union_of_shards_is_the_batch(by):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, by, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    assert q.get(timeout=10) == (True, True, True)
