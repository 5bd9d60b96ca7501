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
