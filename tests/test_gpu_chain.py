"""One decode step as the pages chain it, on one stream with no host synchronisation.

A decode step writes the new token's K and V rows into the window pool (FreeToken PR 633, the
paged KV write), scores the compressed entries with the indexer (FreeToken PR 634, Full mode),
keeps the 512 best as the attention's top-k list, and attends over the window and those entries.
Each kernel reads what a kernel before it wrote.  The small grids of a decode step launch with
programmatic dependent launch: a kernel may start while the one before it still runs, and it
waits inside before its first global memory access.

Run back to back, eagerly and replayed from a CUDA graph, with every buffer a later kernel reads
poisoned first (the written window row, the logits, the top-k list, the output), the step gives
bit for bit the results of the same calls with a device synchronisation after each: the kernels
are deterministic, so any read that ran ahead of its producer would show.  The top-k list is then
checked exactly against the oracle's top-k of the step's own logits, and the attention output
against the float64 oracle over the pools and list the step produced.
"""
import numpy as np
import pytest
import torch

import sparse_paged_attention_gb300 as spa
from oracle import indexer as oi
from oracle_io import run_oracle
from workloads import build, indexer_inputs, kv_write_inputs

pytestmark = pytest.mark.gpu

P = 8191          # the step's position: 2048 compressed entries at ratio 4
RATIO, K, W, D, PS = 4, 512, 128, 512, 64


class Step:
    def __init__(self, dev):
        self.w = w = build("chain", seq_positions=[np.array([P])], num_heads=64, head_dim=D,
                           window=W, topk=K, ratio=RATIO, page_size=PS, seed=31, decode=True)
        x = indexer_inputs([np.array([P])], RATIO, seed=32)
        new = kv_write_inputs([np.array([P])], D, PS, seed=33, specials=False)
        g = lambda t: t.to(dev)
        self.pos = g(w.positions)
        self.q = g(w.q)
        self.win = spa.PagedPool(g(w.win.kv), g(w.win.block_table), None, None)
        self.cmp = spa.PagedPool(g(w.cmp.kv), g(w.cmp.block_table), None, None)
        self.k_new, self.v_new = g(new.k), g(new.v)
        self.xq, self.xw = g(x.q), g(x.weights)
        self.keys, self.kbt = g(x.key_pool), g(x.block_table)
        self.ncols = x.num_cols
        assert self.ncols == (P + 1) // RATIO
        self.logits = torch.empty((1, self.ncols), dtype=torch.float32, device=dev)
        self.topk = torch.empty((1, K), dtype=torch.int32, device=dev)
        self.out = torch.empty_like(self.q)
        n = spa.sparse_attn_paged_decode_workspace_size(self.q, self.win, self.topk, self.pos,
                                                        window=W, ratio=RATIO, scale=w.scale)
        self.ws = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
        page = int(w.win.block_table[0, P // PS])
        self.row = (page, P % PS)   # the window slot the step writes

    def poison(self):
        self.win.kv[self.row[0], self.row[1]] = 100.0
        self.logits.fill_(float("nan"))
        self.topk.fill_(-1)
        self.out.fill_(float("nan"))

    def calls(self):
        yield lambda: spa.sparse_attn_paged_kv_write(self.k_new, self.v_new, self.pos, self.win)
        yield lambda: spa.sparse_attn_indexer_logits(self.xq, self.xw, self.keys, self.kbt,
                                                     self.pos, ratio=RATIO, num_cols=self.ncols,
                                                     out=self.logits)
        yield lambda: spa.sparse_attn_indexer_topk(self.logits, K, out=self.topk)
        yield lambda: spa.sparse_attn_paged_decode(self.q, self.win, self.cmp, self.topk, self.pos,
                                                   window=W, ratio=RATIO, scale=self.w.scale,
                                                   out=self.out, workspace=self.ws)

    def run(self, sync_each):
        for c in self.calls():
            c()
            if sync_each:
                torch.cuda.synchronize()

    def results(self):
        return (self.win.kv[self.row[0], self.row[1]].clone(), self.logits.clone(),
                self.topk.clone(), self.out.clone())


def _equal(a, b):
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))


def test_decode_step_chained_equals_serialised_and_the_oracle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    s = Step(dev)
    s.run(sync_each=True)                  # first calls: kernel attributes, plan caches
    assert spa.sparse_attn_paged_check_errors() == 0

    s.poison()
    s.run(sync_each=True)
    ref = s.results()
    assert torch.isfinite(ref[3].float()).all()

    s.poison()
    s.run(sync_each=False)
    torch.cuda.synchronize()
    _equal(s.results(), ref)

    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        s.run(sync_each=False)
    torch.cuda.current_stream().wait_stream(side)
    with torch.cuda.graph(graph):
        s.run(sync_each=False)
    for _ in range(2):
        s.poison()
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        _equal(s.results(), ref)
    assert spa.sparse_attn_paged_check_errors() == 0

    # the top-k stage: exactly the oracle's selection from the step's own logits
    logits = ref[1].cpu().numpy().astype(np.float64)
    assert np.array_equal(ref[2].cpu().numpy(), oi.topk_entries(logits, K))
    # the attention: the oracle over the pools as the step left them and its top-k list
    w = s.w
    w.win.kv = s.win.kv.cpu()
    w.topk_idx = ref[2].cpu()
    want, _, _, err = run_oracle(w)
    assert not err
    o = ref[3].float().cpu().numpy().astype(np.float64)
    e = np.abs(o - want)
    assert e.max() <= 2e-2 and e.mean() <= 2e-3, (e.max(), e.mean())
