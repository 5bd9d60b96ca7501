"""Adapters from a seeded workload to the oracle's plain-numpy arguments (test helper)."""
import numpy as np

import oracle
from workloads import Workload, bf16_bits


def pool_np(pool, fp8):
    if pool is None:
        return None
    if fp8:
        return pool.kv.numpy()
    return bf16_bits(pool.kv)


def oracle_args(w: Workload):
    a = dict(
        q_bits=bf16_bits(w.q),
        positions=w.positions.numpy(),
        seq_ids=w.seq_ids(),
        win_kv=pool_np(w.win, w.fp8),
        win_bt=w.win.block_table.numpy(),
        cmp_kv=pool_np(w.cmp, w.fp8),
        cmp_bt=None if w.cmp is None else w.cmp.block_table.numpy(),
        topk_idx=w.topk_idx.numpy(),
        window=w.window, ratio=w.ratio, page_size=w.page_size, scale=w.scale, fp8=w.fp8,
    )
    if w.fp8:
        a.update(win_k_scale=w.win.k_scale.numpy(), win_v_scale=w.win.v_scale.numpy())
        if w.cmp is not None:
            a.update(cmp_k_scale=w.cmp.k_scale.numpy(), cmp_v_scale=w.cmp.v_scale.numpy())
    return a


def run_oracle(w: Workload, tokens=None):
    return oracle.sparse_paged_attention(**oracle_args(w), tokens=tokens)


def oracle_columns(w: Workload):
    a = oracle_args(w)
    return oracle.resolve_columns(
        a["positions"], a["seq_ids"], a["win_bt"], a["win_kv"].shape[0],
        a["cmp_bt"] if a["cmp_bt"] is not None else np.zeros((1, 1), np.int64),
        a["cmp_kv"].shape[0] if a["cmp_kv"] is not None else 0,
        a["topk_idx"], window=w.window, ratio=w.ratio, page_size=w.page_size)
