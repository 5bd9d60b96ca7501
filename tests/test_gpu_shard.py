"""Sharding on one GPU: what a rank computes for its shard is what the whole batch computes for
those queries.

Prefill sums every output element in one fixed order, whatever CTA takes the query, so a batch of
independent sequences (workloads.concat_batch) equals each sequence computed alone, and the union
of query-block shards (sparse_paged_attention_gb300.shard) equals the whole call, bit for bit.
Decode picks its split-K plan from the batch size, so shards of a decode batch are compared with
the oracle at the contract tolerance instead.
"""
import numpy as np
import pytest
import torch

import sparse_paged_attention_gb300 as spa
from oracle_io import run_oracle
from sparse_paged_attention_gb300.shard import shard_tokens
from workloads import build, concat_batch

pytestmark = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _pools(w, dev):
    g = lambda t: None if t is None else t.to(dev)
    win = spa.PagedPool(g(w.win.kv), g(w.win.block_table))
    cmp = None if w.cmp is None else spa.PagedPool(g(w.cmp.kv), g(w.cmp.block_table))
    return win, cmp


def _call(w, dev, idx=None, decode=False):
    """The attention of the queries `idx` of workload w (all by default), pools whole."""
    sel = (lambda t: t) if idx is None else (lambda t: t[torch.from_numpy(idx)])
    win, cmp = _pools(w, dev)
    q = sel(w.q).contiguous().to(dev)
    pos = sel(w.positions).contiguous().to(dev)
    tk = sel(w.topk_idx).contiguous().to(dev) if w.topk > 0 else None
    sot = torch.from_numpy(w.seq_ids().astype(np.int32))
    sot = sel(sot).contiguous().to(dev)
    fn = spa.sparse_attn_paged_decode if decode else spa.sparse_attn_paged_prefill
    out = fn(q, win, cmp, tk, pos, window=w.window, ratio=w.ratio, scale=w.scale,
             seq_of_token=sot, num_seqs=w.num_seqs)
    assert spa.sparse_attn_paged_check_errors() == 0
    return out


def _prefill_part(seed):
    # 320 queries per sequence, 16 heads, head_dim 128: more items than SMs, rows by tensor maps
    return build(f"shard_prefill_{seed}", seq_positions=[np.arange(700, 1020)], num_heads=16,
                 head_dim=128, window=64, topk=96, ratio=4, page_size=32, seed=seed)


def test_batch_of_sequences_equals_each_sequence_alone():
    dev = _dev()
    parts = [_prefill_part(s) for s in range(3)]
    batch = concat_batch(parts)
    out_b = _call(batch, dev).view(torch.int16).cpu()
    T = parts[0].num_tokens
    for s, w in enumerate(parts):
        out_p = _call(w, dev).view(torch.int16).cpu()
        assert torch.equal(out_b[s * T:(s + 1) * T], out_p), f"sequence {s}"


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("by", ["sequence", "query_block"])
def test_union_of_shards_is_the_batch(by, world):
    dev = _dev()
    batch = concat_batch([_prefill_part(s) for s in range(3)])
    full = _call(batch, dev).view(torch.int16).cpu()
    assembled = torch.zeros_like(full)
    seen = np.zeros(batch.num_tokens, dtype=int)
    for r in range(world):
        idx = shard_tokens(batch.num_tokens, batch.seq_ids(), r, world, by=by, block=64)
        if len(idx) == 0:
            continue
        assembled[torch.from_numpy(idx)] = _call(batch, dev, idx).view(torch.int16).cpu()
        seen[idx] += 1
    assert np.all(seen == 1)
    assert torch.equal(assembled, full)


def test_decode_shards_match_the_oracle():
    dev = _dev()
    parts = [build(f"shard_decode_{s}", seq_positions=[np.array([4095])] * 4, num_heads=64,
                   head_dim=512, window=128, topk=512, ratio=4, page_size=64, decode=True,
                   seed=s) for s in range(2)]
    batch = concat_batch(parts)
    ref, _, _, _ = run_oracle(batch)
    for r in range(2):
        idx = shard_tokens(batch.num_tokens, batch.seq_ids(), r, 2, by="sequence")
        out = _call(batch, dev, idx, decode=True).float().cpu().numpy().astype(np.float64)
        e = np.abs(out - ref[idx])
        assert np.isfinite(out).all() and e.max() <= 2e-2 and e.mean() <= 2e-3, (r, e.max())
