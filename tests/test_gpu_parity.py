"""CUDA path against the float64 oracle, element by element, through the C ABI (needs a GPU).

Tolerances on bf16 outputs: max |gpu - oracle| <= 2e-2 and mean |gpu - oracle| <= 2e-3 (the
contract), plus a tighter regression gate for bf16 pools: mean |gpu - oracle| <= 1% of mean |oracle|
(rounding the output to bf16 alone costs about 0.15%).  The column list must match exactly.
"""
import numpy as np
import pytest
import torch

import sparse_paged_attention_gb300 as spa
from oracle_io import oracle_columns, run_oracle
from workloads import build, make

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
MEAN_ABS = 2e-3
REL_MEAN_GATE_BF16 = 1e-2


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


class OnDevice:
    """The workload's tensors on the GPU, in the binding's terms."""

    def __init__(self, w, dev):
        g = lambda t: None if t is None else t.to(dev)
        self.w = w
        self.q = g(w.q)
        self.pos = g(w.positions)
        self.tk = g(w.topk_idx) if w.topk > 0 else None
        self.sot = g(w.seq_of_token)
        self.win = spa.PagedPool(g(w.win.kv), g(w.win.block_table), g(w.win.k_scale),
                                 g(w.win.v_scale))
        self.cmp = None if w.cmp is None else spa.PagedPool(
            g(w.cmp.kv), g(w.cmp.block_table), g(w.cmp.k_scale), g(w.cmp.v_scale))

    def kw(self):
        return dict(window=self.w.window, ratio=self.w.ratio, scale=self.w.scale,
                    seq_of_token=self.sot)

    def prefill(self):
        fn = spa.sparse_attn_paged_prefill_fp8 if self.w.fp8 else spa.sparse_attn_paged_prefill
        return fn(self.q, self.win, self.cmp, self.tk, self.pos, **self.kw())

    def decode(self):
        fn = spa.sparse_attn_paged_decode_fp8 if self.w.fp8 else spa.sparse_attn_paged_decode
        return fn(self.q, self.win, self.cmp, self.tk, self.pos, **self.kw())

    def columns(self):
        return spa.sparse_attn_paged_resolve_columns(self.win, self.cmp, self.tk, self.pos,
                                                     window=self.w.window, ratio=self.w.ratio,
                                                     seq_of_token=self.sot)


def compare(out, ref, tokens=None, gate=None, what=""):
    o = out.float().cpu().numpy().astype(np.float64)
    if tokens is not None:
        o = o[np.asarray(tokens)]
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    err = np.abs(o - ref)
    mx, mean = float(err.max()), float(err.mean())
    print(f"{what}: max abs {mx:.3e} mean abs {mean:.3e}")
    assert mx <= MAX_ABS, (what, mx)
    assert mean <= MEAN_ABS, (what, mean)
    if gate is not None:
        rel = mean / float(np.abs(ref).mean())
        print(f"{what}: mean abs / mean |ref| = {rel:.2e}")
        assert rel <= gate, (what, rel, gate)
    return mx, mean


def check_no_device_error():
    assert spa.sparse_attn_paged_check_errors() == 0


# --- column lists: exact -----------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny_r4", "decode_b1_r4", "decode_b8_r128", "decode_b8_r4",
                                  "decode_b8_r0", "prefill_s8192_r4", "prefill_fp8_s4096_r4"])
def test_column_dump_exact(name):
    d = OnDevice(make(name), _dev())
    cols = d.columns().cpu().numpy().astype(np.int64)
    ref, err = oracle_columns(d.w)
    check_no_device_error()
    assert not err
    assert np.array_equal(cols, ref)


# --- the named workloads -----------------------------------------------------------------------

def test_tiny_prefill_and_decode():
    d = OnDevice(make("tiny_r4"), _dev())
    ref, _, _, _ = run_oracle(d.w)
    compare(d.prefill(), ref, gate=REL_MEAN_GATE_BF16, what="tiny prefill")
    compare(d.decode(), ref, gate=REL_MEAN_GATE_BF16, what="tiny decode")
    check_no_device_error()


@pytest.mark.parametrize("name", ["decode_b1_r4", "decode_b8_r128", "decode_b8_r4", "decode_b8_r0",
                                  "decode_b1_r128", "decode_b1_r0"])
def test_decode_workloads(name):
    d = OnDevice(make(name), _dev())
    ref, _, _, _ = run_oracle(d.w)
    compare(d.decode(), ref, gate=REL_MEAN_GATE_BF16, what=f"{name} decode")
    compare(d.prefill(), ref, gate=REL_MEAN_GATE_BF16, what=f"{name} via prefill")
    check_no_device_error()


def _sample_tokens(T, n, seed):
    rng = np.random.default_rng(seed)
    edge = [0, 1, 2, 3, 4, 126, 127, 128, 129, 2046, 2047, 2048, T - 2, T - 1]
    picks = set(t for t in edge if 0 <= t < T)
    picks |= set(rng.choice(T, size=n, replace=False).tolist())
    return sorted(picks)


def test_prefill_s8192_sampled():
    d = OnDevice(make("prefill_s8192_r4"), _dev())
    out = d.prefill()
    check_no_device_error()
    check_convex_bound(out, d.w)
    toks = _sample_tokens(d.w.num_tokens, 50, 1)
    ref, _, _, _ = run_oracle(d.w, tokens=toks)
    compare(out, ref, tokens=toks, gate=REL_MEAN_GATE_BF16, what="prefill S8192 (sampled)")
    # query 0 sees one column (token 0): its output is that V row rounded to bf16
    v0 = d.w.win.kv[int(d.w.win.block_table[0, 0]), 0, 1]
    assert torch.equal(out[0].cpu(), v0.expand(d.w.num_heads, -1))


def check_convex_bound(out, w):
    """Every output is a convex combination of V rows: |out| <= max |V| over the referenced rows
    (bf16 rounding of the output adds at most 2^-8 of that), at every query and head."""
    vals = []
    for pool in (w.win, w.cmp):
        if pool is None:
            continue
        if w.fp8:   # e4m3 code value times the row's V scale
            nb, ps = pool.kv.shape[0], pool.kv.shape[1]
            v = pool.kv[:, :, 1].contiguous().view(torch.float8_e4m3fn).float() * \
                pool.v_scale.view(nb, ps, 1)
        else:
            v = pool.kv[:, :, 1].float()
        vals.append(v[torch.isfinite(v)].abs().max())
    vmax = float(max(vals)) * (1 + 2.0 ** -8)
    o = out.float()
    assert bool(torch.isfinite(o).all()), "non-finite output"
    assert float(o.abs().max()) <= vmax, (float(o.abs().max()), vmax)


@pytest.mark.parametrize("name", ["prefill_s8192_r128", "prefill_s8192_r0",
                                  "prefill_s4096at28672_r4", "prefill_s2048_r4"])
def test_benched_prefill_sampled(name):
    """The other prefill shapes the bench times, at full size in the bench's launch configuration:
    sampled queries against the oracle, every output against the convexity bound."""
    d = OnDevice(make(name), _dev())
    out = d.prefill()
    check_no_device_error()
    check_convex_bound(out, d.w)
    toks = _sample_tokens(d.w.num_tokens, 40, 3)
    ref, _, _, _ = run_oracle(d.w, tokens=toks)
    compare(out, ref, tokens=toks, gate=REL_MEAN_GATE_BF16, what=f"{name} (sampled)")


def test_prefill_window_only_sampled():
    """Window-only prefill over many queries per CTA (no resolver warp: each item's short column
    set is resolved by the gather warps themselves)."""
    d = OnDevice(make("prefill_s2048_r0"), _dev())
    out = d.prefill()
    check_no_device_error()
    toks = _sample_tokens(d.w.num_tokens, 40, 2)
    ref, _, _, _ = run_oracle(d.w, tokens=toks)
    compare(out, ref, tokens=toks, gate=REL_MEAN_GATE_BF16, what="prefill S2048 r0 (sampled)")


# --- generality (FreeToken PR 633, "Correctness and tests": heads 20/16/128, windows 100/50,
#     top-k widths that are not tile multiples, zero counts, the ratio-0 alias, pool views with a
#     row offset) ---------------------------------------------------------------------------------

EDGE = {
    "heads20_w100": dict(num_heads=20, window=100, topk=37, ratio=4, head_dim=512),
    "heads16_w50": dict(num_heads=16, window=50, topk=200, ratio=4, head_dim=256),
    "heads128": dict(num_heads=128, window=128, topk=64, ratio=4, head_dim=128),
    "heads70_d64": dict(num_heads=70, window=33, topk=130, ratio=2, head_dim=64),
    "ratio0_alias": dict(num_heads=64, window=128, topk=0, ratio=0, head_dim=512),
    "topk_only": dict(num_heads=8, window=0, topk=300, ratio=4, head_dim=128),
    "zero_counts": dict(num_heads=8, window=16, topk=40, ratio=4, head_dim=64, topk_fill="empty"),
    "minus1_anywhere": dict(num_heads=12, window=24, topk=150, ratio=4, head_dim=192,
                            topk_fill="anywhere"),
    "row_offset": dict(num_heads=64, window=128, topk=100, ratio=4, head_dim=512, row_offset=3),
    "duplicates": dict(num_heads=8, window=8, topk=20, ratio=4, head_dim=64, duplicate_topk=True),
    "page1": dict(num_heads=8, window=20, topk=20, ratio=4, head_dim=64, page_size=1),
    # a page size that is not a power of two takes the division path of the page lookup
    "page24": dict(num_heads=8, window=40, topk=60, ratio=4, head_dim=64, page_size=24),
    "cols1024": dict(num_heads=64, window=512, topk=512, ratio=2, head_dim=512),
}


@pytest.mark.parametrize("case", sorted(EDGE))
@pytest.mark.parametrize("mode", ["prefill", "decode"])
def test_edge_cases(case, mode):
    kw = dict(EDGE[case])
    kw.setdefault("page_size", 16)
    seqs = [np.array([0, 5, 77, 300, 1500]), np.array([2, 999]), np.array([4095])]
    w = build(case, seq_positions=seqs, seed=7, **kw)
    d = OnDevice(w, _dev())
    out = d.prefill() if mode == "prefill" else d.decode()
    check_no_device_error()
    ref, _, _, err = run_oracle(w)
    assert not err
    compare(out, ref, gate=REL_MEAN_GATE_BF16, what=f"{case} {mode}")
    cols = d.columns().cpu().numpy().astype(np.int64)
    assert np.array_equal(cols, oracle_columns(w)[0])


# The same shapes with more queries than SMs: CTAs then take several items, and bf16 rows move by
# tensor-map gathers (four rows a copy; a group of four that straddles the end of the window
# rows, as in the first queries of a sequence, goes row by row).  Sampled queries: the first
# positions (ragged windows), tile edges, and the tokens of the other sequences.
MANY_SAMPLE = [0, 1, 2, 3, 5, 7, 11, 31, 63, 64, 65, 127, 128, 129, 190, 199, 200, 201, 202]


@pytest.mark.parametrize("case", sorted(EDGE))
def test_edge_cases_many_items(case):
    kw = dict(EDGE[case])
    kw.setdefault("page_size", 16)
    seqs = [np.arange(0, 200), np.array([2, 999]), np.array([4095])]
    w = build(case, seq_positions=seqs, seed=9, **kw)
    d = OnDevice(w, _dev())
    out = d.prefill()
    check_no_device_error()
    ref, _, _, err = run_oracle(w, tokens=np.array(MANY_SAMPLE))
    assert not err
    compare(out, ref, tokens=np.array(MANY_SAMPLE), gate=REL_MEAN_GATE_BF16,
            what=f"{case} prefill, several items per CTA")


def test_bad_block_id_is_reported_and_dropped():
    w = build("bad", seq_positions=[np.array([40, 41])], num_heads=8, head_dim=64, window=8,
              topk=8, ratio=4, page_size=4, seed=3)
    w.win.block_table[0, 10] = w.win.num_blocks + 5       # page of tokens 40..43
    d = OnDevice(w, _dev())
    out = d.prefill()
    assert spa.sparse_attn_paged_check_errors() == spa.SPA_STATUS["SPA_ERR_INDEX"]
    ref, _, cols, err = run_oracle(w)
    assert err
    compare(out, ref, what="bad block id")
    assert np.array_equal(d.columns().cpu().numpy().astype(np.int64), cols)
    assert spa.sparse_attn_paged_check_errors() == spa.SPA_STATUS["SPA_ERR_INDEX"]
    check_no_device_error()


def test_misaligned_pool_view_rejected():
    dev = _dev()
    w = make("tiny_r4")
    d = OnDevice(w, dev)
    flat = d.win.kv.reshape(-1)
    n = (d.win.kv.shape[0] - 1) * d.win.kv[0].numel()
    bad = flat[1:1 + n].view(d.win.kv.shape[0] - 1, *d.win.kv.shape[1:])   # starts 2 bytes in
    pool = spa.PagedPool(bad, d.win.block_table)
    with pytest.raises(spa.SpaError) as e:
        spa.sparse_attn_paged_prefill(d.q, pool, d.cmp, d.tk, d.pos, **d.kw())
    assert e.value.status == spa.SPA_STATUS["SPA_ERR_ALIGN"]


def test_stream_and_repeatability():
    d = OnDevice(make("decode_b8_r4"), _dev())
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = d.decode()
        b = d.decode()
    s.synchronize()
    assert torch.equal(a, b)          # same inputs, same plan: bitwise identical
    c = d.prefill()
    assert torch.equal(d.prefill(), c)


@pytest.mark.parametrize("name", ["prefill_s2048_r4", "prefill_s2048_r0", "prefill_fp8_s4096_r4",
                                  "tiny_r4"])
def test_back_to_back_calls_are_identical(name):
    """Many calls queued back to back (no synchronisation between them), eagerly and replayed from
    a CUDA graph: every output equals the first bit for bit.  The kernels sum each element in one
    fixed order, so any difference would be a race between the pipeline's roles (a ring slot
    refilled while still read, a barrier phase taken for the wrong fill)."""
    d = OnDevice(make(name), _dev())
    first = d.prefill()
    torch.cuda.synchronize()
    check_no_device_error()
    bind = spa.bind_prefill(d.q, d.win, d.cmp, d.tk, d.pos, fp8=d.w.fp8, **d.kw())
    outs = []
    for _ in range(24):
        bind()
        outs.append(bind.out.clone())
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        bind()
    torch.cuda.current_stream().wait_stream(side)
    with torch.cuda.graph(graph):
        for _ in range(4):
            bind()
    for _ in range(6):
        graph.replay()
        outs.append(bind.out.clone())
    torch.cuda.synchronize()
    check_no_device_error()
    ref = first.view(torch.int16)
    bad = [i for i, o in enumerate(outs) if not torch.equal(o.view(torch.int16), ref)]
    assert not bad, f"calls {bad[:8]} differ from the first"


# --- e4m3 pools (FreeToken clone PR 3, "Perf/kv fp8 read path") -------------------------------

REL_MEAN_GATE_FP8 = 2e-2


def test_fp8_prefill_chunk_sampled():
    d = OnDevice(make("prefill_fp8_s4096_r4"), _dev())
    out = d.prefill()
    check_no_device_error()
    check_convex_bound(out, d.w)
    toks = _sample_tokens(d.w.num_tokens, 40, 2)
    ref, _, _, _ = run_oracle(d.w, tokens=toks)
    compare(out, ref, tokens=toks, gate=REL_MEAN_GATE_FP8, what="fp8 prefill chunk (sampled)")


FP8_EDGE = {
    "fp8_decode_b1": dict(seqs=[[32767]], num_heads=64, window=128, topk=512, ratio=4,
                          head_dim=512, page_size=64),
    "fp8_d64_h8": dict(num_heads=8, window=16, topk=40, ratio=4, head_dim=64),
    "fp8_d192_h20": dict(num_heads=20, window=50, topk=77, ratio=4, head_dim=192),
    "fp8_h128_anywhere": dict(num_heads=128, window=33, topk=150, ratio=2, head_dim=256,
                              topk_fill="anywhere"),
    "fp8_ratio0": dict(num_heads=64, window=128, topk=0, ratio=0, head_dim=512),
}


@pytest.mark.parametrize("case", sorted(FP8_EDGE))
@pytest.mark.parametrize("mode", ["prefill", "decode"])
def test_fp8_cases(case, mode):
    kw = dict(FP8_EDGE[case])
    kw.setdefault("page_size", 16)
    seqs = [np.array(s) for s in kw.pop("seqs", [[0, 5, 77, 300, 1500], [2, 999], [4095]])]
    w = build(case, seq_positions=seqs, seed=11, fp8=True, decode=(mode == "decode"), **kw)
    d = OnDevice(w, _dev())
    out = d.prefill() if mode == "prefill" else d.decode()
    check_no_device_error()
    ref, _, _, err = run_oracle(w)
    assert not err
    compare(out, ref, gate=REL_MEAN_GATE_FP8, what=f"{case} {mode}")


@pytest.mark.parametrize("case", sorted(c for c in FP8_EDGE if c != "fp8_decode_b1"))
def test_fp8_cases_many_items(case):
    """e4m3 pools with more queries than SMs: tensor-map gathers where a row is a whole number of
    128-byte boxes (head_dim 256, 512), cp.async with a resolver warp otherwise (64, 192)."""
    kw = dict(FP8_EDGE[case])
    kw.setdefault("page_size", 16)
    seqs = [np.arange(0, 200), np.array([2, 999]), np.array([4095])]
    w = build(case, seq_positions=seqs, seed=13, fp8=True, **kw)
    d = OnDevice(w, _dev())
    out = d.prefill()
    check_no_device_error()
    ref, _, _, err = run_oracle(w, tokens=np.array(MANY_SAMPLE))
    assert not err
    compare(out, ref, tokens=np.array(MANY_SAMPLE), gate=REL_MEAN_GATE_FP8,
            what=f"{case} prefill, several items per CTA")
