"""The seeded workload generator (CPU): determinism and the structure the pages' workloads have."""
import numpy as np
import torch

from workloads import build, make, pool_rows_referenced


def test_seeded_and_deterministic():
    a, b = make("tiny_r4"), make("tiny_r4")
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    assert torch.equal(a.topk_idx, b.topk_idx)
    assert torch.equal(a.win.kv.view(torch.int16), b.win.kv.view(torch.int16))


def test_tiny_structure():
    w = make("tiny_r4")
    assert tuple(w.q.shape) == (16, 8, 64)
    assert w.positions.tolist() == list(range(240, 256))
    tk = w.topk_idx.numpy()
    for t, p in enumerate(range(240, 256)):
        js = tk[t][tk[t] >= 0]
        assert len(js) == 32 and len(set(js.tolist())) == 32
        assert np.all(4 * js + 3 <= p)
    # block tables: a permutation of the pages (oversize 1)
    assert sorted(w.win.block_table[0].tolist()) == list(range(16))


def test_prefill_topk_padding_counts():
    w = build("p", seq_positions=[np.arange(0, 64)], num_heads=2, head_dim=64, window=8, topk=5,
              ratio=4, page_size=8, seed=1)
    tk = w.topk_idx.numpy()
    for i in range(64):
        assert np.count_nonzero(tk[i] >= 0) == min(5, (i + 1) // 4)
    assert pool_rows_referenced(w) == sum(min(i + 1, 8) + min(5, (i + 1) // 4) for i in range(64))


def test_unreferenced_pages_are_poisoned():
    w = make("decode_b1_r4")
    used = set(w.win.block_table[0, 510:512].tolist())
    kv = w.win.kv.float()
    for blk in range(w.win.num_blocks):
        assert bool(torch.isnan(kv[blk]).all()) == (blk not in used)


def test_indexer_inputs_structure():
    from workloads import indexer_inputs
    x = indexer_inputs([np.arange(100, 140), np.array([70])], 2, page_size=16, seed=3)
    a = indexer_inputs([np.arange(100, 140), np.array([70])], 2, page_size=16, seed=3)
    assert torch.equal(x.key_pool, a.key_pool) and torch.equal(x.q.view(torch.int16),
                                                                a.q.view(torch.int16))
    assert x.num_cols == 70 and x.seq_of_token.tolist() == [0] * 40 + [1]
    bt = x.block_table.numpy()
    used = bt[bt >= 0]
    assert len(set(used.tolist())) == len(used)                   # no page shared
    nb = x.key_pool.shape[0]
    spare = np.setdiff1d(np.arange(nb), used)
    scales = x.key_pool[:, :, 16].numpy()
    assert (scales[spare] == -1).all()                            # NaN scales: poisoned rows
    by = scales[used].view(np.uint8)
    assert by.min() >= 121 and by.max() <= 127


def test_indexer_candidates_are_causal_and_distinct():
    from workloads import indexer_inputs
    x = indexer_inputs([np.arange(50, 60)], 1, page_size=8, seed=4, cand_count=80)
    c = x.cand.numpy()
    for t, p in enumerate(range(50, 60)):
        js = c[t][c[t] >= 0]
        assert len(js) == min(80, p + 1) and len(set(js.tolist())) == len(js)
        assert (js <= p).all() and (c[t][len(js):] == -1).all()
    y = indexer_inputs([np.arange(50, 60)], 1, page_size=8, seed=4, cand_count=80,
                       cand_fill="anywhere")
    c = y.cand.numpy()
    assert ((c > np.arange(50, 60)[:, None])).any() and (c == -1).any()


def test_gated_pool_views():
    from workloads import gated_pool_inputs
    for view, stride in (("dense", (700, 100, 1)), ("row_pad", (756, 108, 1)),
                         ("every_other_row", (1400, 200, 1)), ("odd_offset", (700, 100, 1))):
        buf, kv, _, gate = gated_pool_inputs(3, 7, 100, seed=5, view=view)
        assert tuple(kv.shape) == (3, 7, 100) and kv.stride() == stride, view
        assert kv.data_ptr() - buf.data_ptr() == (4 if view == "odd_offset" else 0)
        assert gate.shape == kv.shape
