"""Pins of the indexer-logits oracle (oracle/indexer.py).

The fp4_e8m0_b32 decoding is pinned to hand-worked values from the OCP MX definitions
(tests/golden/e2m1_codes.json, tests/golden/indexer_row.json) and to torch's bf16 type (every
finite (code, scale) product is a bf16 value, as FreeToken PR 634 states).  The logit formula is a
reading; its arithmetic is pinned by closed forms (a unit query reads one key element, a negated
one its ReLU-clipped negative), by linearity in the weights, by a head permutation, by the
candidate/full identity and by causality.  ``test_pins_catch_*`` plant plausible slips.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import indexer as oi
from workloads import bf16_bits, indexer_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _row():
    g = _golden("indexer_row.json")
    return np.array(g["words"], dtype=np.int64).astype(np.int32), \
        {int(k): v for k, v in g["nonzero_or_signed"].items()}


# ---------------------------------------------------------------------------------------------
# format
# ---------------------------------------------------------------------------------------------
def test_e2m1_codes_match_the_hand_worked_table():
    g = _golden("e2m1_codes.json")["codes"]
    codes = np.array([int(k, 16) for k in g])
    want = np.array(list(g.values()), dtype=np.float64)
    got = oi.e2m1_to_f64(codes)
    assert np.array_equal(got, want) and np.array_equal(np.signbit(got), np.signbit(want))


def test_e8m0_scales():
    got = oi.e8m0_to_f64([0, 1, 126, 127, 128, 254, 255])
    assert got[:6].tolist() == [2.0 ** -127, 2.0 ** -126, 0.5, 1.0, 2.0, 2.0 ** 127]
    assert np.isnan(got[6])


def test_hand_worked_row():
    words, expect = _row()
    k = oi.unpack_rows(words)
    assert k.shape == (128,)
    for i in range(128):
        want = expect.get(i, 0.0)
        assert k[i] == want and np.signbit(k[i]) == np.signbit(want), (i, k[i], want)


def test_every_finite_code_scale_pair_is_a_bf16_value():
    """The page's check: every code byte against every scale byte dequantises to bf16 bits.  Here:
    each product is exactly a bf16 value (torch's bf16 conversion leaves it unchanged) for every
    scale byte whose products stay inside the bf16 range: 1 .. 252 (6 * 2^126 passes the largest
    bf16 value; 0xFF is NaN)."""
    rows = np.zeros((4, 68), dtype=np.uint8)
    rows[:, :64] = np.arange(256, dtype=np.uint8).reshape(4, 64)     # all 256 code bytes
    for s in range(1, 253):
        rows[:, 64:68] = s
        k = oi.unpack_rows(rows.view(np.int32))
        back = torch.from_numpy(k).to(torch.bfloat16).double().numpy()
        assert np.array_equal(back, k), s


def test_unpack_keeps_the_nan_scale():
    row = np.zeros(68, dtype=np.uint8)
    row[64:68] = [0xFF, 127, 127, 127]
    k = oi.unpack_rows(row.view(np.int32))
    assert np.isnan(k[:32]).all() and (k[32:] == 0).all()


# ---------------------------------------------------------------------------------------------
# logits
# ---------------------------------------------------------------------------------------------
def _one_row_pool(words):
    pool = np.zeros((1, 1, 17), dtype=np.int32)
    pool[0, 0] = words
    return pool, np.zeros((1, 1), dtype=np.int64)


def _unit_query(d, sign=1.0, heads=1):
    q = torch.zeros(1, heads, 128)
    q[0, 0, d] = sign
    return bf16_bits(q.to(torch.bfloat16))


@pytest.mark.parametrize("d", [0, 1, 30, 32, 33, 66, 67, 127, 5])
def test_unit_query_reads_one_key_element(d):
    words, expect = _row()
    pool, bt = _one_row_pool(words)
    want = expect.get(d, 0.0)
    for sign in (1.0, -1.0):
        lg, err = oi.indexer_logits(_unit_query(d, sign), np.ones((1, 1)), pool, bt, [0], [0],
                                    ratio=1, num_cols=1)
        assert not err and lg[0, 0] == max(0.0, sign * want), (d, sign, lg[0, 0])


def test_weights_act_linearly_and_heads_commute():
    x = indexer_inputs([np.arange(60, 90)], 2, num_heads=8, page_size=8, seed=3)
    args = (x.key_pool.numpy(), x.block_table.numpy(), x.positions.numpy(), x.seq_ids())
    kw = dict(ratio=2, num_cols=x.num_cols)
    w = x.weights.numpy().astype(np.float64)
    a, _ = oi.indexer_logits(bf16_bits(x.q), w, *args, **kw)
    b, _ = oi.indexer_logits(bf16_bits(x.q), 2 * w, *args, **kw)
    fin = np.isfinite(a)
    assert np.allclose(b[fin], 2 * a[fin], rtol=1e-13, atol=1e-12)
    w2 = np.random.default_rng(0).standard_normal(w.shape)
    c, _ = oi.indexer_logits(bf16_bits(x.q), w2, *args, **kw)
    s, _ = oi.indexer_logits(bf16_bits(x.q), w + w2, *args, **kw)
    assert np.allclose(s[fin], a[fin] + c[fin], rtol=1e-12, atol=1e-11)
    perm = np.random.default_rng(1).permutation(8)
    p, _ = oi.indexer_logits(bf16_bits(x.q)[:, perm], w[:, perm], *args, **kw)
    assert np.allclose(p[fin], a[fin], rtol=1e-13, atol=1e-12)


def test_causality_and_full_mode_columns():
    x = indexer_inputs([np.array([0, 1, 2, 7, 40])], 4, num_heads=4, page_size=4, seed=4,
                       num_cols=12)
    lg, err = oi.indexer_logits(bf16_bits(x.q), x.weights.numpy(), x.key_pool.numpy(),
                                x.block_table.numpy(), x.positions.numpy(), x.seq_ids(),
                                ratio=4, num_cols=12)
    assert not err
    for n, p in enumerate([0, 1, 2, 7, 40]):
        valid = (p + 1) // 4
        assert np.isfinite(lg[n, :min(valid, 10)]).all()     # the pool holds 10 entries
        assert np.isneginf(lg[n, valid:]).all()


def test_candidate_mode_gathers_full_mode():
    x = indexer_inputs([np.arange(300, 340)], 2, num_heads=6, page_size=16, seed=5,
                       cand_count=64, cand_fill="anywhere")
    args = (bf16_bits(x.q), x.weights.numpy(), x.key_pool.numpy(), x.block_table.numpy(),
            x.positions.numpy(), x.seq_ids())
    full, _ = oi.indexer_logits(*args, ratio=2, num_cols=340 // 2)
    cand, err = oi.indexer_logits(*args, ratio=2, num_cols=64, cand=x.cand.numpy())
    assert not err
    c = x.cand.numpy()
    for t in range(c.shape[0]):
        for i, j in enumerate(c[t]):
            causal = j >= 0 and 2 * j + 1 <= int(x.positions[t])
            if causal:
                assert cand[t, i] == full[t, j]
            else:
                assert np.isneginf(cand[t, i])


def test_brute_force_tiny():
    x = indexer_inputs([np.array([5, 9])], 1, num_heads=2, page_size=3, seed=6)
    lg, _ = oi.indexer_logits(bf16_bits(x.q), x.weights.numpy(), x.key_pool.numpy(),
                              x.block_table.numpy(), x.positions.numpy(), x.seq_ids(), ratio=1,
                              num_cols=x.num_cols)
    q = x.q.double().numpy()
    w = x.weights.double().numpy()
    flat = x.key_pool.numpy().reshape(-1, 17)
    bt = x.block_table.numpy()
    for t, p in enumerate([5, 9]):
        for j in range(x.num_cols):
            if j > p:
                assert np.isneginf(lg[t, j])
                continue
            row = int(bt[0, j // 3]) * 3 + j % 3
            by = flat[row].view(np.uint8)
            key = []
            for e in range(128):
                nib = (int(by[e // 2]) >> (4 * (e % 2))) & 0xF
                mag = [0, 0.5, 1, 1.5, 2, 3, 4, 6][nib & 7]
                key.append((-mag if nib & 8 else mag) * 2.0 ** (int(by[64 + e // 32]) - 127))
            total = 0.0
            for h in range(2):
                dot = sum(float(q[t, h, e]) * key[e] for e in range(128))
                total += float(w[t, h]) * max(0.0, dot)
            assert abs(lg[t, j] - total) <= 1e-12 * max(1.0, abs(total)), (t, j)


def test_bad_block_is_an_error():
    x = indexer_inputs([np.arange(0, 64)], 1, num_heads=2, page_size=8, seed=7)
    bt = x.block_table.numpy().copy()
    bt[0, 2] = x.key_pool.shape[0] + 5
    lg, err = oi.indexer_logits(bf16_bits(x.q), x.weights.numpy(), x.key_pool.numpy(), bt,
                                x.positions.numpy(), x.seq_ids(), ratio=1, num_cols=64)
    assert err and np.isneginf(lg[63, 16:24]).all() and np.isfinite(lg[63, :16]).all()


# ---------------------------------------------------------------------------------------------
# planted slips
# ---------------------------------------------------------------------------------------------
PINS = [test_hand_worked_row, test_e2m1_codes_match_the_hand_worked_table,
        lambda: [test_unit_query_reads_one_key_element(d) for d in (0, 1, 30, 32, 66, 67, 127)],
        test_causality_and_full_mode_columns, test_brute_force_tiny]


def _some_pin_fails():
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            return True
    return False


def test_pins_catch_swapped_nibbles(monkeypatch):
    real = oi.unpack_rows

    def wrong(words):
        k = real(words)
        out = k.copy()
        out[..., 0::2], out[..., 1::2] = k[..., 1::2], k[..., 0::2]
        return out
    monkeypatch.setattr(oi, "unpack_rows", wrong)
    assert _some_pin_fails()


def test_pins_catch_a_scale_block_of_16(monkeypatch):
    def wrong(words):                                  # scale g applied to elements 16g.. (mod 4)
        w = np.ascontiguousarray(np.asarray(words, dtype=np.int32))
        by = w.view(np.uint8).reshape(*w.shape[:-1], 68)
        codes = np.empty((*w.shape[:-1], 128), dtype=np.int64)
        codes[..., 0::2] = by[..., :64] & 0xF
        codes[..., 1::2] = by[..., :64] >> 4
        sc = oi.e8m0_to_f64(by[..., 64:68])
        return oi.e2m1_to_f64(codes) * sc[..., (np.arange(128) // 16) % 4]
    monkeypatch.setattr(oi, "unpack_rows", wrong)
    assert _some_pin_fails()


def test_pins_catch_a_dropped_relu(monkeypatch):
    monkeypatch.setattr(oi.np, "maximum", lambda a, b: a)
    try:
        assert _some_pin_fails()
    finally:
        monkeypatch.undo()


def test_pins_catch_an_ignored_sign_bit(monkeypatch):
    real = oi.e2m1_to_f64
    monkeypatch.setattr(oi, "e2m1_to_f64", lambda c: np.abs(real(c)))
    assert _some_pin_fails()


def test_pins_catch_off_by_one_causality(monkeypatch):
    real = oi.indexer_logits

    def wrong(*a, ratio, **kw):
        pos = np.asarray(a[4]) + 1                     # one token more than causal
        a = a[:4] + (pos,) + a[5:]
        return real(*a, ratio=ratio, **kw)
    monkeypatch.setattr(oi, "indexer_logits", wrong)
    assert _some_pin_fails()


# ---------------------------------------------------------------------------------------------
# top-k selection
# ---------------------------------------------------------------------------------------------
def _brute_topk(row, ids, k):
    scored = [(float(v), int(j)) for v, j in zip(row, ids) if np.isfinite(v)]
    best = sorted(scored, key=lambda vj: (-vj[0], vj[1]))[:k]
    return [j for _, j in best] + [-1] * (k - len(best))


def test_topk_matches_a_brute_force_sort():
    rng = np.random.default_rng(20)
    lg = rng.integers(-4, 5, size=(30, 50)).astype(np.float64)     # many ties
    lg[rng.random(lg.shape) < 0.3] = -np.inf
    for k in (1, 7, 50, 64):
        got = oi.topk_entries(lg, k)
        for t in range(30):
            assert got[t].tolist() == _brute_topk(lg[t], range(50), k), (k, t)


def test_topk_candidate_ids_and_order_invariance():
    rng = np.random.default_rng(21)
    ids = np.stack([rng.permutation(1000)[:40] for _ in range(5)])
    lg = np.round(rng.standard_normal((5, 40)), 1)
    got = oi.topk_entries(lg, 12, cand=ids)
    for t in range(5):
        assert got[t].tolist() == _brute_topk(lg[t], ids[t], 12)
        perm = rng.permutation(40)
        again = oi.topk_entries(lg[t:t + 1, perm], 12, cand=ids[t:t + 1, perm])
        assert np.array_equal(again[0], got[t])


def test_topk_of_indexer_logits_feeds_the_attention():
    """The indexer's top-k lists are valid attention top-k lists: distinct, causal entries, -1
    only at the tail."""
    x = indexer_inputs([np.arange(0, 200)], 4, num_heads=4, page_size=8, seed=22)
    lg, _ = oi.indexer_logits(bf16_bits(x.q), x.weights.numpy(), x.key_pool.numpy(),
                              x.block_table.numpy(), x.positions.numpy(), x.seq_ids(), ratio=4,
                              num_cols=x.num_cols)
    tk = oi.topk_entries(lg, 16)
    for t, p in enumerate(range(200)):
        valid = (p + 1) // 4
        row = tk[t]
        n = int((row >= 0).sum())
        assert n == min(16, valid) and (row[n:] == -1).all()
        assert len(set(row[:n].tolist())) == n and (4 * row[:n] + 3 <= p).all()
        assert np.all(np.diff(lg[t, row[:n]]) <= 0)


def test_pins_catch_ties_to_the_larger_index(monkeypatch):
    real_lexsort = np.lexsort
    monkeypatch.setattr(oi.np, "lexsort", lambda keys: real_lexsort((-keys[0], keys[1])))
    try:
        with pytest.raises(AssertionError):
            test_topk_matches_a_brute_force_sort()
    finally:
        monkeypatch.undo()
