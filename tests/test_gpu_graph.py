"""The attention calls captured in a CUDA graph.

A serving loop records its decode step once and replays it with new queries in the same buffers.
That works only if a call allocates nothing, synchronises nothing and takes every pointer from its
arguments at launch.  The replayed result must equal, bit for bit, an eager call on the same
inputs: the kernels are deterministic (each output element is summed in one fixed order).
"""
import pytest
import torch

import sparse_paged_attention_gb300 as spa
from workloads import make

pytestmark = pytest.mark.gpu


def _setup(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = make(name)
    dev = torch.device("cuda:0")
    g = lambda t: None if t is None else t.to(dev)
    win = spa.PagedPool(g(w.win.kv), g(w.win.block_table), g(w.win.k_scale), g(w.win.v_scale))
    cmp = None if w.cmp is None else spa.PagedPool(g(w.cmp.kv), g(w.cmp.block_table),
                                                   g(w.cmp.k_scale), g(w.cmp.v_scale))
    tk = g(w.topk_idx) if w.topk > 0 else None
    kw = dict(window=w.window, ratio=w.ratio, scale=w.scale, seq_of_token=g(w.seq_of_token))
    if w.decode:
        fn = spa.sparse_attn_paged_decode_fp8 if w.fp8 else spa.sparse_attn_paged_decode
        n = spa.sparse_attn_paged_decode_workspace_size(g(w.q), win, tk, g(w.positions),
                                                        window=w.window, ratio=w.ratio,
                                                        scale=w.scale)
        kw["workspace"] = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
    else:
        fn = spa.sparse_attn_paged_prefill_fp8 if w.fp8 else spa.sparse_attn_paged_prefill
    return w, dev, g(w.q), g(w.positions), tk, win, cmp, fn, kw


@pytest.mark.parametrize("name", ["decode_b1_r4", "decode_b8_r4", "decode_b8_r0", "tiny_r4",
                                  "prefill_s2048_r4"])
def test_graph_replay_equals_eager(name):
    w, dev, q, pos, tk, win, cmp, fn, kw = _setup(name)
    out = torch.empty_like(q)
    fn(q, win, cmp, tk, pos, out=out, **kw)          # first call: kernel attributes, plan caches
    torch.cuda.synchronize()
    assert spa.sparse_attn_paged_check_errors() == 0

    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn(q, win, cmp, tk, pos, out=out, **kw)
    torch.cuda.current_stream().wait_stream(side)
    with torch.cuda.graph(graph):
        fn(q, win, cmp, tk, pos, out=out, **kw)

    gen = torch.Generator(device="cpu").manual_seed(7)
    for _ in range(2):                                # new queries in the captured buffers
        q.copy_(torch.randn(q.shape, generator=gen).to(q.dtype))
        if tk is not None:
            perm = torch.randperm(tk.shape[1], generator=gen)
            tk.copy_(tk[:, perm.to(dev)])             # same columns, another order
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert spa.sparse_attn_paged_check_errors() == 0
        eager = fn(q, win, cmp, tk, pos, **{k: v for k, v in kw.items()})
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


@pytest.mark.parametrize("name", ["decode_b1_r4", "prefill_s2048_r4"])
def test_bound_call_records_on_the_capturing_stream(name):
    """A call bound once (spa.bind_prefill / bind_decode, no stream given) launches on torch's
    current stream at call time, so recording it inside a graph capture records the kernel: the
    replay rewrites out, bit for bit the eager result."""
    w, dev, q, pos, tk, win, cmp, fn, kw = _setup(name)
    bind = spa.bind_decode if w.decode else spa.bind_prefill
    call = bind(q, win, cmp, tk, pos, window=w.window, ratio=w.ratio, scale=w.scale,
                seq_of_token=kw["seq_of_token"], fp8=w.fp8)
    call()
    torch.cuda.synchronize()
    assert spa.sparse_attn_paged_check_errors() == 0
    eager = call.out.clone()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    with torch.cuda.graph(graph):
        call()
    call.out.fill_(float("nan"))
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert spa.sparse_attn_paged_check_errors() == 0
    assert torch.equal(call.out.view(torch.int16), eager.view(torch.int16))
