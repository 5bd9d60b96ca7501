"""Checks that pin the float64 oracle to things other than itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with what the mathematics
or a hand-worked fixture fixes.  They look the oracle's functions up at call time, so that
``test_oracle_mutations.py`` can plant a mistake in the oracle and show that some pin catches it.
"""
import json
import os

import numpy as np
import scipy.special
import torch

import oracle.sparse_attention as O
from workloads import build, bf16_bits

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _same_f64(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    both_nan = np.isnan(a) & np.isnan(b)
    eq = (a == b) & (np.signbit(a) == np.signbit(b))
    return bool(np.all(both_nan | eq))


# --- number formats -----------------------------------------------------------------------

def pin_bf16_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert _same_f64(O.bf16_to_f64(bits), ref), "bf16 decode differs from torch's bf16 -> f64"


def pin_e4m3_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = O.e4m3_to_f64(codes)
    assert _same_f64(mine, lib), "e4m3 decode differs from torch float8_e4m3fn -> f64"
    g = _golden("e4m3_codes.json")["codes"]
    for k, v in g.items():
        val = O.e4m3_to_f64(np.array([int(k, 16)], np.uint8))[0]
        want = float("nan") if v == "nan" else float(v)
        assert _same_f64(val, want), f"code {k}: {val} != {want}"
    finite = mine[np.isfinite(mine)]
    assert finite.max() == 448.0 and finite.max() / 256 == 1.75
    assert np.count_nonzero(np.isnan(mine)) == 2


# --- column resolution --------------------------------------------------------------------

def pin_resolve_golden():
    g = _golden("resolve_small.json")
    cols, err = O.resolve_columns(
        np.array(g["positions"]), np.array(g["seq_ids"]), np.array(g["win_block_table"]),
        g["win_num_blocks"], np.array(g["cmp_block_table"]), g["cmp_num_blocks"],
        np.array(g["topk_idx"]), window=g["window"], ratio=g["ratio"],
        page_size=g["page_size"])
    assert cols.tolist() == g["expected_cols"], cols.tolist()
    assert err == g["expected_error"]
    # a block id beyond the pool is an input error, and that column is dropped
    bad = np.array(g["win_block_table"])
    bad[0, 2] = g["win_num_blocks"]
    cols2, err2 = O.resolve_columns(
        np.array(g["positions"]), np.array(g["seq_ids"]), bad, g["win_num_blocks"],
        np.array(g["cmp_block_table"]), g["cmp_num_blocks"], np.array(g["topk_idx"]),
        window=g["window"], ratio=g["ratio"], page_size=g["page_size"])
    assert err2 and cols2[0, 2] == -1 and cols2[0, :2].tolist() == [4, 5]


def _dense_history(pool_kv, table_row, n_pages):
    """Logical history of one sequence, copied page by page out of the pool (forward mapping:
    logical page lp lives in physical block table_row[lp])."""
    return np.concatenate([pool_kv[table_row[lp]] for lp in range(n_pages)], axis=0)


def _small_workload(seed, ratio=4, window=6, topk=5, fill="anywhere", fp8=False, heads=3,
                    dim=16, seqs=None, page_size=4):
    if seqs is None:
        seqs = [np.array([0, 3, 9, 17, 30]), np.array([11, 12, 25])]
    return build("pin", seq_positions=seqs, num_heads=heads, head_dim=dim, window=window,
                 topk=topk, ratio=ratio, page_size=page_size, seed=seed, topk_fill=fill,
                 fp8=fp8, decode=False)


def pin_resolve_logical_content():
    """Every resolved row must hold the token (or compressed entry) the definition names, and the
    number of columns must be min(p+1, W) + #{j >= 0 with r*j + r - 1 <= p}."""
    for seed in range(4):
        w = _small_workload(seed)
        sid = w.seq_of_token.numpy()
        pos = w.positions.numpy()
        tk = w.topk_idx.numpy()
        ps = w.page_size
        # tag every pool row with its own physical id, then read tags in logical order
        wtag = np.arange(w.win.num_blocks * ps).reshape(w.win.num_blocks, ps)
        ctag = np.arange(w.cmp.num_blocks * ps).reshape(w.cmp.num_blocks, ps)
        cols, err = O.resolve_columns(pos, sid, w.win.block_table.numpy(), w.win.num_blocks,
                                      w.cmp.block_table.numpy(), w.cmp.num_blocks, tk,
                                      window=w.window, ratio=w.ratio, page_size=ps)
        assert not err
        for t in range(len(pos)):
            b, p = int(sid[t]), int(pos[t])
            wb = w.win.block_table.numpy()[b]
            whist = _dense_history(wtag, wb, int(np.count_nonzero(wb >= 0)))
            cb = w.cmp.block_table.numpy()[b]
            chist = _dense_history(ctag, cb, int(np.count_nonzero(cb >= 0)))
            want_win = [int(whist[tok]) for tok in range(p - w.window + 1, p + 1) if tok >= 0]
            got_win = [int(c) for c in cols[t, :w.window] if c >= 0]
            assert got_win == want_win, (t, got_win, want_win)
            causal = [int(j) for j in tk[t]
                      if j >= 0 and max(range(w.ratio * j, w.ratio * j + w.ratio)) <= p]
            want_cmp = [(1 << 30) | int(chist[j]) for j in causal]
            got_cmp = [int(c) for c in cols[t, w.window:] if c >= 0]
            assert got_cmp == want_cmp, (t, got_cmp, want_cmp)
            assert np.count_nonzero(cols[t] >= 0) == min(p + 1, w.window) + len(causal)


# --- attention ----------------------------------------------------------------------------

def _workload_arrays(w):
    from oracle_io import oracle_args
    return oracle_args(w)


def pin_dense_bruteforce(fp8=False):
    """Dense masked attention over the whole logical history of each sequence: the mask is column
    membership written as set membership, the softmax is scipy's.  Must match to 1e-12."""
    for seed in range(3):
        w = _small_workload(seed, fp8=fp8)
        a = _workload_arrays(w)
        out, lse, _, err = O.sparse_paged_attention(**a)
        assert not err
        sid = w.seq_of_token.numpy()
        pos = w.positions.numpy()
        tk = w.topk_idx.numpy()
        q = bf16_bits(w.q)
        ps = w.page_size

        def dense(pool, b):
            """Whole logical history of sequence b, page by page, decoded by torch."""
            bt = pool.block_table.numpy()[b]
            pages = [int(bt[lp]) for lp in range(int(np.count_nonzero(bt >= 0)))]
            if fp8:
                codes = np.concatenate([pool.kv[pg].numpy() for pg in pages])
                vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
                rows = np.concatenate([pg * ps + np.arange(ps) for pg in pages])
                ks = pool.k_scale.numpy().astype(np.float64)[rows]
                vs = pool.v_scale.numpy().astype(np.float64)[rows]
                return vals[:, 0, :] * ks[:, None], vals[:, 1, :] * vs[:, None]
            kv = torch.cat([pool.kv[pg] for pg in pages]).double().numpy()
            return kv[:, 0, :], kv[:, 1, :]

        for t in range(len(pos)):
            b, p = int(sid[t]), int(pos[t])
            kw, vw = dense(w.win, b)
            kc, vc = dense(w.cmp, b)
            K = np.concatenate([kw, kc])
            V = np.concatenate([vw, vc])
            win_set = set(range(max(0, p - w.window + 1), p + 1))
            cmp_set = {int(j) for j in tk[t]
                       if j >= 0 and all(tok <= p for tok in range(w.ratio * j, w.ratio * (j + 1)))}
            mask = np.array([i in win_set for i in range(len(kw))]
                            + [j in cmp_set for j in range(len(kc))])
            qf = torch.from_numpy(q[t].view(np.int16)).view(torch.bfloat16).double().numpy()
            s = w.scale * np.einsum("hd,cd->hc", qf, K)
            s = np.where(mask[None, :], s, -np.inf)
            p_ = scipy.special.softmax(s, axis=1)
            want = np.einsum("hc,cd->hd", p_, np.where(mask[:, None], V, 0.0))
            want_lse = scipy.special.logsumexp(s, axis=1)
            np.testing.assert_allclose(out[t], want, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[t], want_lse, rtol=0, atol=1e-12)


def pin_ratio0_sdpa():
    """With r = 0 the method is sliding-window causal attention: compare with torch's
    scaled_dot_product_attention (float64, explicit band mask) on the dense history."""
    pos = np.arange(0, 40)
    w = build("pin_r0", seq_positions=[pos], num_heads=4, head_dim=32, window=7, topk=0,
              ratio=0, page_size=8, seed=5)
    out, lse, _, err = O.sparse_paged_attention(**_workload_arrays(w))
    assert not err
    bt = w.win.block_table.numpy()[0]
    hist = torch.cat([w.win.kv[int(bt[lp])] for lp in range(5)]).double()  # [40, 2, D]
    k = hist[:, 0, :].unsqueeze(0).expand(4, -1, -1)
    v = hist[:, 1, :].unsqueeze(0).expand(4, -1, -1)
    q = w.q.double().transpose(0, 1)                                      # [H, T, D]
    i = torch.arange(40).view(-1, 1)
    j = torch.arange(40).view(1, -1)
    band = (j <= i) & (j > i - 7)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=band,
                                                           scale=w.scale)
    np.testing.assert_allclose(out, ref.transpose(0, 1).numpy(), rtol=0, atol=1e-12)


def pin_two_column_golden():
    g = _golden("attn_two_columns.json")
    q = np.array(g["q"], np.float64)
    k = np.array(g["k_rows"], np.float64)
    v = np.array(g["v_rows"], np.float64)
    out, lse = O.attend(q, k, v, g["scale"])
    np.testing.assert_allclose(out, g["expected_out"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, g["expected_lse"], rtol=0, atol=1e-14)
    # the same case through the paged path: bf16 pool, ratio 0, page size 2, window 2
    kv = np.zeros((1, 2, 2, 2), np.float32)
    kv[0, :, 0, :] = k
    kv[0, :, 1, :] = v
    kv_bits = torch.from_numpy(kv).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    qb = torch.tensor(q, dtype=torch.bfloat16).view(1, 1, 2).view(torch.int16).numpy()
    out2, lse2, cols, _ = O.sparse_paged_attention(
        qb.view(np.uint16), np.array([1]), np.array([0]), kv_bits, np.array([[0]]), None, None,
        np.zeros((1, 0), np.int32), window=2, ratio=0, page_size=2, scale=g["scale"])
    assert cols.tolist() == [[0, 1]]
    np.testing.assert_allclose(out2[0], g["expected_out"], rtol=0, atol=1e-14)


def pin_closed_forms():
    # query at position 0 sees exactly one column (token 0): out is that V row, exactly
    w = build("pin_first", seq_positions=[np.arange(0, 6)], num_heads=5, head_dim=16, window=4,
              topk=3, ratio=4, page_size=4, seed=11)
    out, lse, cols, _ = O.sparse_paged_attention(**_workload_arrays(w))
    v0 = w.win.kv[int(w.win.block_table[0, 0]), 0, 1].double().numpy()
    assert np.count_nonzero(cols[0] >= 0) == 1
    assert np.array_equal(out[0], np.broadcast_to(v0, out[0].shape))
    # equal K rows: every weight equal, out = mean of V over the columns
    rng = np.random.default_rng(3)
    q = rng.standard_normal((4, 8))
    k = np.tile(rng.standard_normal(8), (9, 1))
    v = rng.standard_normal((9, 8))
    o, l = O.attend(q, k, v, 0.7)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(0), o.shape), rtol=0, atol=1e-12)
    # no columns: zero output, lse -inf
    o, l = O.attend(q, np.zeros((0, 8)), np.zeros((0, 8)), 0.7)
    assert np.all(o == 0) and np.all(np.isneginf(l))


def pin_split_merge():
    """Merging split-K partials by log-sum-exp equals the single pass (f64, 1e-12), for any
    split of the column list, empty splits included."""
    rng = np.random.default_rng(7)
    for trial in range(20):
        C = int(rng.integers(1, 60))
        q = rng.standard_normal((6, 16))
        k = rng.standard_normal((C, 16)) * 2
        v = rng.standard_normal((C, 16))
        whole, whole_lse = O.attend(q, k, v, 0.5)
        cuts = np.sort(rng.integers(0, C + 1, size=int(rng.integers(0, 6))))
        bounds = [0, *cuts.tolist(), C]
        parts = O.decode_split_k(q, k, v, 0.5, bounds)
        out, lse = O.merge_partials(parts)
        np.testing.assert_allclose(out, whole, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, whole_lse, rtol=0, atol=1e-12)


def pin_permutation_invariance():
    """Relabelling physical pages (moving the data with them) leaves the output unchanged, and so
    does reordering each top-k list."""
    w = _small_workload(21, fill="sample")
    a = _workload_arrays(w)
    out, lse, _, _ = O.sparse_paged_attention(**a)
    rng = np.random.default_rng(1)
    perm = rng.permutation(a["win_kv"].shape[0])
    kv2 = np.empty_like(a["win_kv"])
    kv2[perm] = a["win_kv"]
    bt2 = np.where(a["win_bt"] >= 0, perm[np.maximum(a["win_bt"], 0)], -1)
    b = dict(a, win_kv=kv2, win_bt=bt2)
    out2, _, _, _ = O.sparse_paged_attention(**b)
    assert np.array_equal(out, out2)
    tk = a["topk_idx"].copy()
    for t in range(tk.shape[0]):
        tk[t] = tk[t][rng.permutation(tk.shape[1])]
    out3, lse3, _, _ = O.sparse_paged_attention(**dict(a, topk_idx=tk))
    np.testing.assert_allclose(out3, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse3, lse, rtol=0, atol=1e-12)


def pin_fp8_scale_folding():
    """FreeToken clone PR 3, part 1: the per-row scale is constant along the reduction, so
    (q . code) * s_k == q . (code * s_k) and (p * s_v) . code == p . (code * s_v)."""
    rng = np.random.default_rng(9)
    codes = rng.integers(0, 256, size=(12, 32), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3A
    vals = O.e4m3_to_f64(codes)
    sk = rng.uniform(1e-3, 1e-1, size=12)
    q = rng.standard_normal(32)
    lhs = (vals @ q) * sk
    rhs = (vals * sk[:, None]) @ q
    np.testing.assert_allclose(lhs, rhs, rtol=1e-13, atol=0)
    p = rng.uniform(0, 1, size=12)
    np.testing.assert_allclose((p * sk) @ vals, p @ (vals * sk[:, None]), rtol=1e-13, atol=1e-15)


ALL_PINS = [
    pin_bf16_all_patterns, pin_e4m3_all_codes, pin_resolve_golden, pin_resolve_logical_content,
    pin_dense_bruteforce, pin_ratio0_sdpa, pin_two_column_golden, pin_closed_forms,
    pin_split_merge, pin_permutation_invariance, pin_fp8_scale_folding,
]
