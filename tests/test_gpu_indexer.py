"""Indexer logits and their top-k selection on the GPU against the float64 oracle.

Shapes follow FreeToken PR 634 ("Kernel time": 32 index heads, index head_dim 128, Full mode and
candidate mode, prefill and decode), scaled so the oracle finishes in seconds, plus the pages'
decode shapes at full size with every column compared, and edge cases (ragged tiles, several
sequences, candidates with -1 and non-causal entries anywhere, a bad block).

Tolerance, from the arithmetic: the keys enter the MMA exactly (every e2m1 code times its scale is a
bf16 value), products of bf16 values are exact in fp32, and the 128-term dot product accumulates
in fp32 on the tensor cores; the ReLU is exact; the 32-term weighted head sum is fp32 FMAs.  So
|gpu - oracle| <= u * (128 + 32 + 8) * sum_h |w_h| * sum_d |q_hd k_d|, taking u = 2^-22 (four
fp32 roundings' worth of slack for the tensor cores' accumulation order).  -inf must match
exactly.
"""
import numpy as np
import pytest
import torch

import sparse_paged_attention_gb300 as spa
from oracle import indexer as oi
from workloads import bf16_bits, indexer_inputs

pytestmark = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _run(x, dev, use_seq=False):
    g = lambda t: None if t is None else t.to(dev)
    out = spa.sparse_attn_indexer_logits(
        g(x.q), g(x.weights), g(x.key_pool), g(x.block_table), g(x.positions), ratio=x.ratio,
        num_cols=x.num_cols, cand=g(x.cand), seq_of_token=g(x.seq_of_token) if use_seq else None,
        num_seqs=x.num_seqs)
    st = spa.sparse_attn_paged_check_errors()
    return out.cpu().numpy(), st


def _bound(x, tokens):
    """Per-element tolerance (see the module docstring) for the listed queries."""
    q = np.abs(x.q.double().numpy())
    w = np.abs(x.weights.double().numpy())
    flat = x.key_pool.numpy().reshape(-1, 17)
    bt = x.block_table.numpy()
    nb, ps = x.key_pool.shape[0], x.key_pool.shape[1]
    sid = x.seq_ids()
    out = np.zeros((len(tokens), x.num_cols))
    for n, t in enumerate(tokens):
        js = np.arange(x.num_cols) if x.cand is None else x.cand[t].numpy().astype(np.int64)
        ok = (js >= 0) & (x.ratio * js + x.ratio - 1 <= int(x.positions[t]))
        cols = np.nonzero(ok)[0]
        if cols.size == 0:
            continue
        j = js[cols]
        blk = bt[sid[t], j // ps].astype(np.int64)
        live = (blk >= 0) & (blk < nb)
        cols, j, blk = cols[live], j[live], blk[live]
        k = np.abs(oi.unpack_rows(flat[blk * ps + j % ps]))
        out[n, cols] = (k @ q[t].T) @ w[t]
    return 2.0 ** -22 * (128 + 32 + 8) * out


def _compare(x, got, tokens):
    ref, err = oi.indexer_logits(bf16_bits(x.q), x.weights.numpy(), x.key_pool.numpy(),
                                 x.block_table.numpy(), x.positions.numpy(), x.seq_ids(),
                                 ratio=x.ratio, num_cols=x.num_cols,
                                 cand=None if x.cand is None else x.cand.numpy(), tokens=tokens)
    g = got[tokens].astype(np.float64)
    inf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(g), inf_ref), "the -inf pattern differs"
    assert np.isfinite(g[~inf_ref]).all()
    tol = _bound(x, tokens)
    with np.errstate(invalid="ignore"):   # -inf - -inf where both sides are -inf
        e = np.abs(g - ref)
    e[inf_ref] = 0
    bad = np.argwhere(e > tol)
    assert bad.size == 0, (len(bad), bad[:3], e.max())
    return err


CASES = {
    # prefill from position 0, one sequence: groups of eight queries share every key tile
    "full_prefill_s300_r2": dict(seqs=[np.arange(0, 300)], ratio=2, ps=16),
    # a ragged query count (not a multiple of 8) and a tail tile, ratio 1
    "full_prefill_s203_at900_r1": dict(seqs=[np.arange(900, 1103)], ratio=1, ps=64),
    # ratio 4 with a page size that does not divide the tile
    "full_prefill_s77_at5000_r4": dict(seqs=[np.arange(5000, 5077)], ratio=4, ps=24),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_full_mode_prefill(case):
    c = CASES[case]
    x = indexer_inputs(c["seqs"], c["ratio"], page_size=c["ps"], seed=11)
    got, st = _run(x, _dev())
    assert st == 0
    err = _compare(x, got, np.arange(x.q.shape[0]))
    assert not err


def test_full_mode_decode_several_sequences():
    """Four sequences at different lengths, one query each (sequence ids given: one query per
    key tile)."""
    seqs = [np.array([4095]), np.array([1000]), np.array([2047]), np.array([130])]
    x = indexer_inputs(seqs, 2, page_size=64, seed=12)
    got, st = _run(x, _dev(), use_seq=True)
    assert st == 0
    _compare(x, got, np.arange(4))


@pytest.mark.parametrize("fill", ["tail", "anywhere"])
def test_candidate_mode(fill):
    x = indexer_inputs([np.arange(1000, 1020)], 1, page_size=32, seed=13, cand_count=300,
                       cand_fill=fill)
    got, st = _run(x, _dev())
    assert st == 0
    _compare(x, got, np.arange(20))


def test_candidate_mode_several_sequences():
    seqs = [np.array([700, 701]), np.array([90]), np.array([333, 334, 335])]
    x = indexer_inputs(seqs, 1, page_size=16, seed=14, cand_count=260, cand_fill="anywhere")
    got, st = _run(x, _dev(), use_seq=True)
    assert st == 0
    _compare(x, got, np.arange(6))


def test_bad_block_is_flagged_and_masked():
    x = indexer_inputs([np.arange(600, 640)], 2, page_size=16, seed=15)
    x.block_table[0, 3] = x.key_pool.shape[0] + 7             # entries 48..63 point past the pool
    got, st = _run(x, _dev())
    assert st == spa.SPA_STATUS["SPA_ERR_INDEX"]
    err = _compare(x, got, np.arange(40))
    assert err and np.isneginf(got[:, 48:64]).all()


@pytest.mark.parametrize("ctx,ratio,B", [(131072, 2, 1), (131072, 1, 1), (32768, 2, 4)])
def test_pages_full_decode_shapes(ctx, ratio, B):
    """The page's Full decode shapes at full size: every column of every query compared."""
    x = indexer_inputs([np.array([ctx - 1])] * B, ratio, page_size=64, seed=16)
    got, st = _run(x, _dev(), use_seq=B > 1)
    assert st == 0
    _compare(x, got, np.arange(B))


def test_pages_candidate_decode_shape():
    x = indexer_inputs([np.array([131071])] * 4, 1, page_size=64, seed=17, cand_count=16384)
    got, st = _run(x, _dev(), use_seq=True)
    assert st == 0
    _compare(x, got, np.arange(4))


def test_pages_full_prefill_shape_sampled():
    """n 128 at position 130944, ratio 1 (131072 columns): sampled queries, all their columns."""
    x = indexer_inputs([np.arange(130944, 131072)], 1, page_size=64, seed=18)
    got, st = _run(x, _dev())
    assert st == 0
    _compare(x, got, np.array([0, 7, 8, 64, 127]))


# ---------------------------------------------------------------------------------------------
# top-k selection: exact against the oracle on seeded logits (ties, -inf, -0, few scored rows)
# ---------------------------------------------------------------------------------------------
def _topk_logits(T, N, seed, kind):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        lg = rng.standard_normal((T, N)).astype(np.float32)
    elif kind == "ties":
        lg = rng.integers(-3, 4, (T, N)).astype(np.float32)
        lg[rng.random((T, N)) < 0.3] = -0.0
    else:  # "sparse": most columns unscored
        lg = rng.standard_normal((T, N)).astype(np.float32)
        lg[rng.random((T, N)) < 0.97] = -np.inf
    lg[rng.random((T, N)) < 0.1] = -np.inf
    return lg


# Up to a sixteenth as many rows as SMs take a cluster of 16 CTAs per row, up to an eighth a
# cluster of 8 (12 rows), the row split in chunks (1001 and 4099 columns are not multiples of 4;
# 7 columns leave most CTAs of the cluster without any); 40 rows take one wide CTA per row; 160
# rows, more than SMs, take narrower CTAs (several per SM).
@pytest.mark.parametrize("T,N,k", [(4, 300, 16), (3, 65536, 512), (2, 131072, 2048), (5, 700, 900),
                                   (3, 1001, 64), (2, 7, 4), (12, 4099, 700), (12, 65536, 2048),
                                   (40, 2051, 300), (160, 4096, 256)])
@pytest.mark.parametrize("kind", ["normal", "ties", "sparse"])
def test_topk_exact(T, N, k, kind):
    dev = _dev()
    lg = _topk_logits(T, N, seed=N + k, kind=kind)
    got = spa.sparse_attn_indexer_topk(torch.from_numpy(lg).to(dev), k).cpu().numpy()
    want = oi.topk_entries(lg.astype(np.float64), k)
    assert np.array_equal(got, want)


def test_topk_candidate_ids():
    dev = _dev()
    rng = np.random.default_rng(30)
    lg = _topk_logits(6, 16384, seed=31, kind="ties")
    cand = np.stack([rng.permutation(131072)[:16384] for _ in range(6)]).astype(np.int32)
    got = spa.sparse_attn_indexer_topk(torch.from_numpy(lg).to(dev), 512,
                                       cand=torch.from_numpy(cand).to(dev)).cpu().numpy()
    assert np.array_equal(got, oi.topk_entries(lg.astype(np.float64), 512, cand=cand))


def test_paired_key_decoding_equals_per_code_decoding(tmp_path):
    """The indexer decodes key bytes two codes at a time (e2m1x2_to_bf16x2_bits in
    sparse_paged_attention_gb300/csrc/spa_indexer_math.cuh): for every byte and every ue8m0 scale
    but the NaN one, the bits equal the per-code decoding that the host test checks against the
    oracle (tests/indexer_dequant_check.cu)."""
    import os
    import shutil
    import subprocess
    _dev()
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    exe = str(tmp_path / "indexer_dequant_check")
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                        "-I", os.path.join(root, "sparse_paged_attention_gb300", "csrc"),
                        os.path.join(root, "tests", "indexer_dequant_check.cu"), "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    pairs, bad = (int(v) for v in out.stdout.split())
    assert pairs == 255 * 256 and bad == 0, (pairs, bad)
