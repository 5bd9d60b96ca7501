"""The decode entry point that allocates nothing, against the ordinary decode entry point and
against the float64 oracle.

Some callers cannot call cudaMalloc where they decode (their device allocator belongs to another
runtime, or their host has no allocator hooks at that point).  For them
sparse_attn_paged_decode_noalloc keeps the split-K partials in a scratch array built into the
library and merges them with the separate merge kernel.  This file is collected last so that a run
stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import sparse_paged_attention_gb300 as spa
from oracle_io import run_oracle
from workloads import build, make

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
SCRATCH_BYTES = 16 << 20      # SPA_NOALLOC_SCRATCH_BYTES in include/sparse_attn_paged.h


def _call_noalloc_c(lib, d, out):
    """Straight through the C ABI: q, pools, problem and out; no workspace argument."""
    w = d["w"]
    prob = spa._problem_c(d["q"], d["win"], d["tk"], d["pos"], d["sot"], w.window, w.ratio,
                          w.scale, None)
    win = spa._pool_c(d["win"], False)
    cmp = spa._pool_c(d["cmp"], False) if d["cmp"] is not None else None
    return lib.sparse_attn_paged_decode_noalloc(
        d["q"].data_ptr(), ctypes.byref(win), ctypes.byref(cmp) if cmp is not None else None,
        ctypes.byref(prob), out.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _on_device(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = make(name)
    dev = torch.device("cuda:0")
    g = lambda t: None if t is None else t.to(dev)
    return {"w": w, "q": g(w.q), "pos": g(w.positions), "sot": g(w.seq_of_token),
            "tk": g(w.topk_idx) if w.topk > 0 else None,
            "win": spa.PagedPool(g(w.win.kv), g(w.win.block_table)),
            "cmp": None if w.cmp is None else spa.PagedPool(g(w.cmp.kv), g(w.cmp.block_table))}


def _within(out, ref, what):
    err = np.abs(out.float().cpu().numpy().astype(np.float64) - ref)
    assert np.all(np.isfinite(err)), what
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (what, err.max(), err.mean())


@pytest.mark.parametrize("name", ["decode_b8_r4", "decode_b8_r128", "decode_b8_r0",
                                  "decode_b1_r4", "tiny_r4"])
def test_noalloc_matches_decode_and_oracle_twice(name):
    d = _on_device(name)
    lib = spa.load_library()
    w = d["w"]
    ref = spa.sparse_attn_paged_decode(d["q"], d["win"], d["cmp"], d["tk"], d["pos"],
                                       window=w.window, ratio=w.ratio, scale=w.scale,
                                       seq_of_token=d["sot"])
    ref_np = ref.float().cpu().numpy().astype(np.float64)
    exact, _, _, _ = run_oracle(w)          # the float64 definition itself
    for call in range(2):                   # the shared scratch keeps the previous call's partials
        out = torch.full_like(d["q"], float("nan"))
        assert _call_noalloc_c(lib, d, out) == 0
        assert spa.sparse_attn_paged_check_errors() == 0
        _within(out, ref_np, f"{name} call {call}: against sparse_attn_paged_decode")
        _within(out, exact, f"{name} call {call}: against the oracle")


def test_noalloc_lowers_its_split_count_to_fit():
    """32 decode queries of 64 heads x 512 over 640 columns: on 152 SMs the split plan would take
    4 splits, whose partials (16.8 MB) exceed the built-in array; the entry point takes fewer,
    longer splits instead of failing."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = build("decode_b32_r4_at1023", seq_positions=[np.array([1023])] * 32, num_heads=64,
              head_dim=512, window=128, topk=512, ratio=4, page_size=64, decode=True, seed=7)
    dev = torch.device("cuda:0")
    g = lambda t: None if t is None else t.to(dev)
    d = {"w": w, "q": g(w.q), "pos": g(w.positions), "sot": g(w.seq_of_token),
         "tk": g(w.topk_idx), "win": spa.PagedPool(g(w.win.kv), g(w.win.block_table)),
         "cmp": spa.PagedPool(g(w.cmp.kv), g(w.cmp.block_table))}
    exact, _, _, _ = run_oracle(w)
    lib = spa.load_library()
    for call in range(2):
        out = torch.full_like(d["q"], float("nan"))
        assert _call_noalloc_c(lib, d, out) == 0
        assert spa.sparse_attn_paged_check_errors() == 0
        _within(out, exact, f"32 queries, call {call}: against the oracle")


def test_noalloc_rejects_problems_beyond_its_scratch():
    d = _on_device("decode_b8_r4")
    lib = spa.load_library()
    # 4096 tokens of 64 heads x 512 need far more partial storage than the built-in array holds
    q = torch.zeros((4096, 64, 512), dtype=torch.bfloat16, device=d["q"].device)
    pos = torch.full((4096,), 32767, dtype=torch.int32, device=q.device)
    sot = torch.zeros(4096, dtype=torch.int32, device=q.device)
    tk = torch.full((4096, 512), -1, dtype=torch.int32, device=q.device)
    big = dict(d, q=q, pos=pos, sot=sot, tk=tk)
    # fp32 partials of at least one split per query: 4096 x 64 x 512 x 4 bytes = 512 MiB
    need = 4096 * 64 * 512 * 4
    assert need > SCRATCH_BYTES
    out = torch.empty_like(q)
    assert _call_noalloc_c(lib, big, out) == spa.SPA_STATUS["SPA_ERR_WORKSPACE"]

