"""Prefill from host buffers against the device-buffer call: bit for bit.

sparse_attn_paged_prefill_host takes q, the top-k lists, the positions (and sequence ids) and the
output in page-locked host memory, and moves them through device staging memory a chunk of tokens
at a time, copies in, kernels and copies out of consecutive chunks overlapping on the library's
own streams.  Each query's output depends only on its own inputs, so the result must equal the
device call's exactly: with chunks that divide the tokens, a ragged last chunk, one chunk larger
than the call, several sequences, and e4m3 pools.  The caller's stream alone is synchronised
before the output is read (the call makes that stream wait for all of its work).
"""
import numpy as np
import pytest
import torch

import sparse_paged_attention_gb300 as spa
from workloads import build, make

pytestmark = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _check(w, chunk):
    dev = _dev()
    g = lambda t: None if t is None else t.to(dev)
    win = spa.PagedPool(g(w.win.kv), g(w.win.block_table), g(w.win.k_scale), g(w.win.v_scale))
    cmp = None if w.cmp is None else spa.PagedPool(g(w.cmp.kv), g(w.cmp.block_table),
                                                   g(w.cmp.k_scale), g(w.cmp.v_scale))
    kw = dict(window=w.window, ratio=w.ratio, scale=w.scale)
    tk = w.topk_idx if w.topk > 0 else None
    dev_fn = spa.sparse_attn_paged_prefill_fp8 if w.fp8 else spa.sparse_attn_paged_prefill
    want = dev_fn(g(w.q), win, cmp, g(tk), g(w.positions), seq_of_token=g(w.seq_of_token), **kw)
    torch.cuda.synchronize()
    pin = lambda t: None if t is None else t.contiguous().pin_memory()
    call = spa.bind_prefill_host(pin(w.q), win, cmp, pin(tk), pin(w.positions),
                                 seq_of_token=pin(w.seq_of_token), chunk_tokens=chunk,
                                 fp8=w.fp8, **kw)
    for _ in range(2):                    # twice: the second call reuses the streams and events
        call.out.fill_(float("nan"))
        call()
        torch.cuda.current_stream().synchronize()
        assert spa.sparse_attn_paged_check_errors() == 0
        assert torch.equal(call.out.view(torch.int16), want.cpu().view(torch.int16))


@pytest.mark.parametrize("chunk", [512, 300, 4096])
def test_host_prefill_equals_device_prefill(chunk):
    _check(make("prefill_s2048_r4"), chunk)


def test_host_prefill_several_sequences_and_e4m3():
    w = build("host_seqs", seq_positions=[np.arange(0, 300), np.arange(500, 777), np.array([9])],
              num_heads=16, head_dim=128, window=64, topk=100, ratio=4, page_size=16, seed=41)
    _check(w, 128)
    w8 = build("host_fp8", seq_positions=[np.arange(1000, 1500)], num_heads=64, head_dim=512,
               window=128, topk=512, ratio=4, page_size=64, seed=42, fp8=True)
    _check(w8, 192)
