"""Paged KV write on the GPU against the oracle: bit-exact pools and scales.

The write quantises with one fp32 scale per (token, kv_head) row (FreeToken clone PR 3, "Perf/kv
fp8 read path") and places every row in its page slot (FreeToken PR 633, pool layout).  Codes and
scales are integers and binary32 values decided the same way on both sides (binary32 scale and
quotients, round to nearest even), so the comparison is exact, byte for byte, including the slots
no token writes (they must keep their sentinel).
"""
import numpy as np
import pytest
import torch

import sparse_paged_attention_gb300 as spa
from oracle import kv_write as okw
from oracle_io import run_oracle
from workloads import bf16_bits, build, kv_write_inputs

pytestmark = pytest.mark.gpu

SENTINEL = 0x5A


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _run(inp, fp8, dev, num_seqs=None):
    nb, ps, D = inp.num_blocks, inp.page_size, inp.k.shape[1]
    elt = 1 if fp8 else 2
    kv = torch.full((nb, ps, 2, D * elt), SENTINEL, dtype=torch.uint8)
    ks = torch.full((nb * ps,), -7.0, dtype=torch.float32)
    vs = ks.clone()
    # oracle on host copies
    kv_o = kv.numpy().copy()
    ks_o, vs_o = ks.numpy().copy(), vs.numpy().copy()
    pool_o = kv_o if fp8 else kv_o.view(np.uint16).reshape(nb, ps, 2, D)
    dropped = okw.kv_write(bf16_bits(inp.k), bf16_bits(inp.v), inp.positions.numpy(),
                           inp.seq_of_token.numpy(), inp.block_table.numpy(), pool_o,
                           page_size=ps, k_scale=ks_o, v_scale=vs_o, fp8=fp8)
    # device
    kv_d = kv.to(dev) if fp8 else kv.view(torch.bfloat16).reshape(nb, ps, 2, D).to(dev)
    pool = spa.PagedPool(kv_d, inp.block_table.to(dev), ks.to(dev), vs.to(dev))
    fn = spa.sparse_attn_paged_kv_write_fp8 if fp8 else spa.sparse_attn_paged_kv_write
    fn(inp.k.to(dev), inp.v.to(dev), inp.positions.to(dev), pool,
       seq_of_token=inp.seq_of_token.to(dev), num_seqs=num_seqs)
    st = spa.sparse_attn_paged_check_errors()
    got_kv = kv_d.view(torch.uint8).cpu().numpy().reshape(kv_o.shape)
    return got_kv, pool.k_scale.cpu().numpy(), pool.v_scale.cpu().numpy(), kv_o, ks_o, vs_o, \
        dropped, st


CASES = {
    "d512_p64": dict(seqs=[np.arange(0, 300), np.arange(1000, 1100), np.array([7])], D=512, ps=64),
    "d64_p16": dict(seqs=[np.arange(0, 97), np.array([3, 40, 41, 500])], D=64, ps=16),
    "d256_p24": dict(seqs=[np.arange(10, 250, 3)], D=256, ps=24),
    "d128_p1": dict(seqs=[np.arange(0, 40), np.arange(0, 33)], D=128, ps=1),
}


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("fp8", [False, True])
def test_kv_write_bit_exact(case, fp8):
    c = CASES[case]
    inp = kv_write_inputs(c["seqs"], c["D"], c["ps"], seed=5)
    got_kv, got_ks, got_vs, kv_o, ks_o, vs_o, dropped, st = _run(inp, fp8, _dev())
    assert not dropped and st == 0
    assert np.array_equal(got_kv, kv_o.view(np.uint8).reshape(got_kv.shape))
    if fp8:
        assert np.array_equal(got_ks.view(np.uint32), ks_o.view(np.uint32))
        assert np.array_equal(got_vs.view(np.uint32), vs_o.view(np.uint32))


def test_kv_write_drops_bad_pages_and_flags_them():
    inp = kv_write_inputs([np.arange(0, 130)], 64, 16, seed=6)
    inp.block_table[0, 3] = inp.num_blocks + 4       # tokens 48..63 point past the pool
    inp.positions[100] = -1                           # a negative position
    got_kv, got_ks, got_vs, kv_o, ks_o, vs_o, dropped, st = _run(inp, True, _dev())
    assert dropped and st == spa.SPA_STATUS["SPA_ERR_INDEX"]
    assert np.array_equal(got_kv, kv_o) and np.array_equal(got_ks.view(np.uint32), ks_o.view(np.uint32))


def test_kv_write_then_e4m3_attention_over_the_written_pool():
    """The rows of the queries' own positions are rewritten through the kernel; e4m3 prefill over
    the GPU-written pools then matches the oracle attention over the oracle-written pools (which
    are byte-identical), within the e4m3 parity bar."""
    dev = _dev()
    w = build("kvw", seq_positions=[np.arange(200, 456)], num_heads=16, head_dim=128, window=64,
              topk=100, ratio=4, page_size=16, seed=8, fp8=True)
    nb, ps = w.win.kv.shape[0], w.win.kv.shape[1]
    inp = kv_write_inputs([np.arange(200, 456)], 128, ps, seed=9, specials=False)
    kv_d = w.win.kv.clone().to(dev)
    ks_d, vs_d = w.win.k_scale.clone().to(dev), w.win.v_scale.clone().to(dev)
    win = spa.PagedPool(kv_d, w.win.block_table.to(dev), ks_d, vs_d)
    spa.sparse_attn_paged_kv_write_fp8(inp.k.to(dev), inp.v.to(dev), inp.positions.to(dev), win,
                                       seq_of_token=inp.seq_of_token.to(dev))
    assert spa.sparse_attn_paged_check_errors() == 0
    kv_o = w.win.kv.numpy().copy()
    ks_o, vs_o = w.win.k_scale.numpy().copy(), w.win.v_scale.numpy().copy()
    okw.kv_write(bf16_bits(inp.k), bf16_bits(inp.v), inp.positions.numpy(), None,
                 w.win.block_table.numpy(), kv_o, page_size=ps, k_scale=ks_o, v_scale=vs_o,
                 fp8=True)
    assert np.array_equal(kv_d.cpu().numpy(), kv_o)
    assert np.array_equal(ks_d.cpu().numpy().view(np.uint32), ks_o.view(np.uint32))
    assert np.array_equal(vs_d.cpu().numpy().view(np.uint32), vs_o.view(np.uint32))
    # attention over the written pools
    w.win.kv = torch.from_numpy(kv_o)
    w.win.k_scale, w.win.v_scale = torch.from_numpy(ks_o), torch.from_numpy(vs_o)
    g = lambda t: None if t is None else t.to(dev)
    cmp = spa.PagedPool(g(w.cmp.kv), g(w.cmp.block_table), g(w.cmp.k_scale), g(w.cmp.v_scale))
    out = spa.sparse_attn_paged_prefill_fp8(g(w.q), win, cmp, g(w.topk_idx), g(w.positions),
                                            window=w.window, ratio=w.ratio, scale=w.scale,
                                            seq_of_token=g(w.seq_of_token))
    assert spa.sparse_attn_paged_check_errors() == 0
    toks = np.array([0, 1, 63, 64, 100, 200, 255])
    ref, _, _, err = run_oracle(w, tokens=toks)
    assert not err
    o = out.float().cpu().numpy().astype(np.float64)[toks]
    e = np.abs(o - ref)
    assert np.isfinite(o).all() and e.max() <= 2e-2 and e.mean() <= 2e-3, (e.max(), e.mean())


def test_e4m3_codes_match_ieee_division_for_every_input_pair(tmp_path):
    """The e4m3 write divides by the row scale with a correctly rounded reciprocal and one
    correction step (sparse_paged_attention_gb300/csrc/spa_kvwrite_quant.cuh).  A row's elements
    are bf16 values no larger in magnitude than the row maximum, so every pair the write can see
    is checked: every positive finite bf16 maximum m (scale m / 448) and every bf16 x with
    |x| <= m, both signs, plus zeros of both signs (about 10^9 pairs).  The codes equal the e4m3
    codes of the IEEE binary32 quotients.  Rows with a maximum below about 2^-79 divide instead:
    counted over every bf16 exponent alike they hold 3.5 % of the pairs, so more than 90 % of the
    pairs take the reciprocal path."""
    import os
    import shutil
    import subprocess
    _dev()
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    exe = str(tmp_path / "kvwrite_quant_check")
    r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                        "-I", os.path.join(root, "sparse_paged_attention_gb300", "csrc"),
                        os.path.join(root, "tests", "kvwrite_quant_check.cu"), "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    pairs, bad, fast, qdiff = (int(v) for v in out.stdout.split())
    assert pairs > 10 ** 9
    assert bad == 0, (bad, qdiff)
    assert fast > 0.9 * pairs, (fast, pairs)


def test_kv_write_more_than_32_groups_per_cta():
    """A CTA of the write takes every gridDim-th group of eight tokens, and each lane of a consumer
    warp resolves its warp's slot 32 groups ahead: with more than 32 groups per CTA (three CTAs
    per SM) the look-ahead is refilled mid-run.  34 groups per CTA, a partial last group, and a
    dropped token in a late group: the pool equals the oracle's bit for bit and the drop is
    flagged."""
    dev = _dev()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    T = 8 * 3 * sms * 34 + 5
    inp = kv_write_inputs([np.arange(0, T)], 64, 64, seed=12, specials=False)
    inp.positions[T - 100] = -1
    got_kv, got_ks, got_vs, kv_o, ks_o, vs_o, dropped, st = _run(inp, False, dev)
    assert dropped and st == spa.SPA_STATUS["SPA_ERR_INDEX"]
    assert np.array_equal(got_kv, kv_o.view(np.uint8).reshape(got_kv.shape))
