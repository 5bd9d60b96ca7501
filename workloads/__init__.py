"""Seeded synthetic workloads for sparse paged attention.

This module only draws data: queries, paged K/V pools, block tables, top-k index lists and
positions. It holds none of the attention arithmetic, so both the float64 oracle (``oracle/``)
and the CUDA library (``sparse_paged_attention_gb300``) can be fed from it without sharing code.

Shapes follow the DeepSeek-V4 sparse attention workloads timed on the FreeToken PR 633 page
("Kernel time" table: 64 heads, head_dim 512, 128-token window, index top-k 512, compress ratio
r in {4, 128, 0}).  Storage conventions (one kv_head; K and V rows of a token stored next to each
other) are readings of what the pages leave open:

* pool ``kv``: ``[num_blocks, page_size, 2, head_dim]``; index ``[..., 0, :]`` is K, ``[..., 1, :]``
  is V. Element type bf16, or e4m3 codes stored as uint8 with fp32 ``k_scale``/``v_scale`` per
  physical row (``block * page_size + slot``).
* the window pool holds every token of a sequence at its absolute position, addressed through the
  sequence's window block table (logical page ``pos // page_size``).
* the compressed pool holds compressed entry ``j`` of a sequence at logical page ``j // page_size``
  of its compressed block table; entry ``j`` summarises tokens ``r*j .. r*j + r - 1``.
* top-k rows list compressed entry indices, padded with -1 at the tail.

Pages that no query of the workload reads, and the spare pages of an oversized pool, are filled with
NaN (bf16 0x7FC0, e4m3 0x7F, scale NaN) so that a stray read shows up in the output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np
import torch

BF16_NAN_BITS = 0x7FC0
E4M3_NAN_CODE = 0x7F
E4M3_MAX = 448.0

__all__ = [
    "Pool", "Workload", "build", "make", "concat_batch", "CONFIG_NAMES", "bf16_bits",
    "pool_rows_referenced",
]


@dataclass
class Pool:
    """One paged K/V pool plus the block table that maps each sequence's logical pages."""

    kv: torch.Tensor                      # [num_blocks, page_size, 2, D] bf16 or uint8 (e4m3)
    block_table: torch.Tensor             # int32 [num_seqs, stride]; -1 = unmapped
    k_scale: Optional[torch.Tensor] = None  # float32 [num_blocks * page_size] (fp8 only)
    v_scale: Optional[torch.Tensor] = None

    @property
    def num_blocks(self) -> int:
        return int(self.kv.shape[0])

    @property
    def page_size(self) -> int:
        return int(self.kv.shape[1])


@dataclass
class Workload:
    name: str
    fp8: bool
    decode: bool
    num_heads: int
    head_dim: int
    window: int
    topk: int
    ratio: int
    page_size: int
    scale: float
    q: torch.Tensor                        # bf16 [T, H, D]
    positions: torch.Tensor                # int32 [T]
    seq_of_token: Optional[torch.Tensor]   # int32 [T] or None (all tokens belong to sequence 0)
    topk_idx: torch.Tensor                 # int32 [T, K]
    win: Pool
    cmp: Optional[Pool]
    meta: dict = field(default_factory=dict)

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_seqs(self) -> int:
        return int(self.win.block_table.shape[0])

    def seq_ids(self) -> np.ndarray:
        if self.seq_of_token is None:
            return np.zeros(self.num_tokens, dtype=np.int64)
        return self.seq_of_token.numpy().astype(np.int64)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw uint16 bit patterns of a bf16 tensor (numpy has no bf16 type)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _assign_pages(g: torch.Generator, pages_per_seq: Sequence[int], oversize: int):
    """Random physical pages for every sequence from one shared pool.

    Returns (num_blocks, table[int32 B x stride]) with -1 in unused table slots.
    """
    total = int(sum(pages_per_seq))
    num_blocks = max(1, total * oversize)
    perm = torch.randperm(num_blocks, generator=g)[:total].to(torch.int32)
    stride = max(1, max(pages_per_seq) if pages_per_seq else 1)
    table = torch.full((len(pages_per_seq), stride), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(pages_per_seq):
        table[b, :n] = perm[off:off + n]
        off += n
    return num_blocks, table


def _fill_pool(g: torch.Generator, num_blocks: int, page_size: int, head_dim: int,
               referenced_pages: np.ndarray, fp8: bool, row_offset: int = 0):
    """Pool storage: N(0,1) rows on referenced pages, NaN poison elsewhere.

    ``row_offset`` extra leading rows (poisoned) model a pool that is a view into a larger
    allocation; the returned tensors are views that start after them.
    """
    nrows = num_blocks * page_size
    pages = np.nonzero(referenced_pages)[0]
    if fp8:
        flat = torch.full((row_offset + nrows, 2, head_dim), E4M3_NAN_CODE, dtype=torch.uint8)
        ks = torch.full((row_offset + nrows,), float("nan"), dtype=torch.float32)
        vs = torch.full((row_offset + nrows,), float("nan"), dtype=torch.float32)
        kv = flat[row_offset:].view(num_blocks, page_size, 2, head_dim)
        if len(pages):
            x = torch.randn(len(pages), page_size, 2, head_dim, generator=g)
            amax = x.abs().amax(dim=-1)                       # [n, ps, 2]
            sc = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
            codes = (x / sc.unsqueeze(-1)).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
            idx = torch.from_numpy(pages.astype(np.int64))
            kv[idx] = codes.view(torch.uint8)
            rows = (idx.view(-1, 1) * page_size + torch.arange(page_size)).reshape(-1)
            ks[row_offset:][rows] = sc[..., 0].reshape(-1)
            vs[row_offset:][rows] = sc[..., 1].reshape(-1)
        return kv, ks[row_offset:], vs[row_offset:]
    flat = torch.full((row_offset + nrows, 2, head_dim), 0, dtype=torch.int16)
    flat.fill_(np.int16(BF16_NAN_BITS).item())
    flat = flat.view(torch.bfloat16)
    kv = flat[row_offset:].view(num_blocks, page_size, 2, head_dim)
    if len(pages):
        idx = torch.from_numpy(pages.astype(np.int64))
        kv[idx] = torch.randn(len(pages), page_size, 2, head_dim, generator=g).to(torch.bfloat16)
    return kv, None, None


def build(name: str, *, seq_positions: Sequence[np.ndarray], num_heads: int, head_dim: int,
          window: int, topk: int, ratio: int, page_size: int, fp8: bool = False, seed: int = 0,
          oversize: int = 2, decode: bool = False, scale: Optional[float] = None,
          cmp_entries: Optional[Sequence[int]] = None, row_offset: int = 0,
          topk_fill: str = "sample", duplicate_topk: bool = False) -> Workload:
    """Draw one workload.

    seq_positions[b] lists the absolute positions of the queries of sequence b (queries are laid
    out sequence after sequence).  ``cmp_entries[b]`` overrides the number of compressed entries
    stored for sequence b (default: every entry whose tokens all lie at or before the sequence's
    last position, i.e. ``(max_pos + 1) // ratio``).

    topk_fill:
      "sample"  - min(K, valid) distinct entries drawn uniformly from the causally valid range,
                  random order, -1 at the tail;
      "anywhere" - like "sample" but the -1 padding is scattered among the entries and some
                  non-causal (future) entries are mixed in, which must be masked;
      "empty"   - every entry -1.
    """
    g = torch.Generator().manual_seed(seed)
    B = len(seq_positions)
    pos_list = [np.asarray(p, dtype=np.int64) for p in seq_positions]
    max_pos = [int(p.max()) for p in pos_list]
    T = int(sum(len(p) for p in pos_list))
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)

    # block tables
    win_pages = [math.ceil((mp + 1) / page_size) for mp in max_pos]
    win_blocks, win_bt = _assign_pages(g, win_pages, oversize)
    if ratio > 0:
        if cmp_entries is None:
            cmp_entries = [(mp + 1) // ratio for mp in max_pos]
        cmp_pages = [max(1, math.ceil(n / page_size)) for n in cmp_entries]
        cmp_blocks, cmp_bt = _assign_pages(g, cmp_pages, oversize)
    else:
        cmp_entries = [0] * B

    # queries
    positions = torch.from_numpy(np.concatenate(pos_list).astype(np.int32))
    seq_of_token = torch.from_numpy(
        np.concatenate([np.full(len(p), b, dtype=np.int32) for b, p in enumerate(pos_list)]))
    q = torch.randn(T, num_heads, head_dim, generator=g).to(torch.bfloat16)

    # top-k index lists
    topk_idx = torch.full((T, topk), -1, dtype=torch.int32)
    if topk > 0 and ratio > 0 and topk_fill != "empty":
        t = 0
        for b, pl in enumerate(pos_list):
            for p in pl:
                valid = min(int(cmp_entries[b]), (int(p) + 1) // ratio)
                k_eff = min(topk, valid)
                if k_eff > 0:
                    sel = torch.randperm(valid, generator=g)[:k_eff].to(torch.int32)
                    if duplicate_topk and k_eff >= 2:
                        sel[-1] = sel[0]
                    topk_idx[t, :k_eff] = sel
                if topk_fill == "anywhere":
                    row = topk_idx[t].clone()
                    future_hi = int(cmp_entries[b])
                    if valid < future_hi:
                        nf = min(3, topk - k_eff)
                        fut = torch.randint(valid, future_hi, (nf,), generator=g, dtype=torch.int32)
                        row[k_eff:k_eff + nf] = fut
                    topk_idx[t] = row[torch.randperm(topk, generator=g)]
                t += 1

    # which physical pages any query reads
    win_ref = np.zeros(win_blocks, dtype=bool)
    win_bt_np = win_bt.numpy()
    t = 0
    for b, pl in enumerate(pos_list):
        for p in pl:
            lo = max(0, int(p) - window + 1) if window > 0 else int(p) + 1
            for lp in range(lo // page_size, int(p) // page_size + 1):
                if lo <= int(p):
                    win_ref[win_bt_np[b, lp]] = True
            t += 1
    win_kv, win_ks, win_vs = _fill_pool(g, win_blocks, page_size, head_dim, win_ref, fp8,
                                        row_offset)
    win = Pool(win_kv, win_bt, win_ks, win_vs)

    cmp = None
    if ratio > 0:
        cmp_ref = np.zeros(cmp_blocks, dtype=bool)
        cmp_bt_np = cmp_bt.numpy()
        tk = topk_idx.numpy()
        sot = seq_of_token.numpy()
        for t in range(T):
            js = tk[t]
            js = js[(js >= 0) & (js < int(cmp_entries[sot[t]]))]
            if len(js):
                cmp_ref[cmp_bt_np[sot[t], js // page_size]] = True
        cmp_kv, cmp_ks, cmp_vs = _fill_pool(g, cmp_blocks, page_size, head_dim, cmp_ref, fp8,
                                            row_offset)
        cmp = Pool(cmp_kv, cmp_bt, cmp_ks, cmp_vs)

    return Workload(name=name, fp8=fp8, decode=decode, num_heads=num_heads, head_dim=head_dim,
                    window=window, topk=topk, ratio=ratio, page_size=page_size, scale=float(scale),
                    q=q, positions=positions, seq_of_token=seq_of_token if (decode or B > 1) else None,
                    topk_idx=topk_idx, win=win, cmp=cmp,
                    meta={"seed": seed, "cmp_entries": list(cmp_entries), "oversize": oversize,
                          "row_offset": row_offset})


def pool_rows_referenced(w: Workload) -> int:
    """Number of (query, column) pairs that resolve to a row: used for byte/flop accounting."""
    total = 0
    pos = w.positions.numpy().astype(np.int64)
    sot = w.seq_ids()
    tk = w.topk_idx.numpy()
    for t in range(w.num_tokens):
        p = int(pos[t])
        total += min(p + 1, w.window)
        if w.ratio > 0 and w.topk > 0:
            js = tk[t]
            n_ent = int(w.meta["cmp_entries"][sot[t]])
            total += int(np.count_nonzero((js >= 0) & (w.ratio * js + w.ratio - 1 <= p)
                                          & (js < n_ent)))
    return total


# Workloads named after what they are.  Sizes follow the FreeToken PR 633 "Kernel time" shapes
# (64 heads, head_dim 512, window 128, top-k 512, page size 64).
CONFIG_NAMES = (
    "tiny_r4",              # 16 queries @ 240..255, 8 heads, D 64, window 16, top-k 32 of 64 (r 4)
    "decode_b1_r4",         # B 1 @ 32767, 64 heads, D 512, window 128, top-k 512 of 8192 (r 4)
    "decode_b8_r128",       # B 8 @ 32767, top-k 256 of 256 (r 128)
    "decode_b8_r4",         # B 8 @ 32767, top-k 512 of 8192 (r 4)
    "decode_b8_r0",         # B 8 @ 32767, window only
    "prefill_s8192_r4",     # 8192 queries from position 0, top-k 512 (r 4)
    "prefill_fp8_s4096_r4", # e4m3 pools, 4096 queries at 28672..32767, top-k 512 of 8192 (r 4)
)
# The remaining shapes of the same table.
PAGE_SHAPES = (
    "prefill_s2048_r4", "prefill_s4096at28672_r4", "prefill_s8192_r128", "prefill_s8192_r0",
    "decode_b1_r128", "decode_b1_r0",
)


def make(name: str, seed: int = 0) -> Workload:
    """The named workloads (seed 0 unless told otherwise)."""
    big = dict(num_heads=64, head_dim=512, window=128, page_size=64, seed=seed)
    topk_of = {128: 256, 4: 512, 0: 0}
    if name == "tiny_r4":
        return build(name, seq_positions=[np.arange(240, 256)], num_heads=8, head_dim=64,
                     window=16, topk=32, ratio=4, page_size=16, seed=seed, oversize=1)
    if name.startswith("decode_b"):
        bsz, r = name[len("decode_b"):].split("_r")
        r = int(r)
        return build(name, seq_positions=[np.array([32767])] * int(bsz), topk=topk_of[r],
                     ratio=r, decode=True, **big)
    if name == "prefill_fp8_s4096_r4":
        return build(name, seq_positions=[np.arange(28672, 32768)], topk=512, ratio=4, fp8=True,
                     cmp_entries=[8192], **big)
    if name == "prefill_s4096at28672_r4":
        return build(name, seq_positions=[np.arange(28672, 32768)], topk=512, ratio=4, **big)
    if name.startswith("prefill_s"):
        S, r = name[len("prefill_s"):].split("_r")
        r = int(r)
        return build(name, seq_positions=[np.arange(0, int(S))], topk=topk_of[r], ratio=r, **big)
    raise KeyError(name)


def _stack_tables(tables, offsets):
    """Block-table rows of several pools stacked, block ids shifted by each pool's offset (-1, an
    unmapped page, stays -1), padded with -1 to the widest stride."""
    width = max(int(t.shape[1]) for t in tables)
    rows = []
    for t, off in zip(tables, offsets):
        t = t.to(torch.int64)
        t = torch.where(t >= 0, t + off, t)
        pad = torch.full((t.shape[0], width - t.shape[1]), -1, dtype=torch.int64)
        rows.append(torch.cat([t, pad], dim=1))
    return torch.cat(rows).to(torch.int32)


def _concat_pools(pools):
    offsets = np.cumsum([0] + [p.num_blocks for p in pools[:-1]]).tolist()
    kv = torch.cat([p.kv for p in pools])
    bt = _stack_tables([p.block_table for p in pools], offsets)
    ks = vs = None
    if pools[0].k_scale is not None:
        ks = torch.cat([p.k_scale for p in pools])
        vs = torch.cat([p.v_scale for p in pools])
    return Pool(kv, bt, ks, vs)


def concat_batch(parts: Sequence[Workload], name: Optional[str] = None) -> Workload:
    """Independent workloads of one shape as a single batch: their sequences one after the other
    (sequence ids of part i shifted by the sequences of the parts before it), their pools
    concatenated (block ids shifted by the blocks before them).  Every query keeps its q, position,
    top-k list and the row values it reads, so a query's result in the batch is its result in its
    own part."""
    w0 = parts[0]
    for w in parts:
        for f in ("fp8", "num_heads", "head_dim", "window", "topk", "ratio", "page_size", "scale"):
            if getattr(w, f) != getattr(w0, f):
                raise ValueError(f"parts differ in {f}")
    sot, cmp_entries, base = [], [], 0
    for w in parts:
        sot.append(torch.from_numpy(w.seq_ids().astype(np.int32)) + base)
        cmp_entries += list(w.meta["cmp_entries"])
        base += w.num_seqs
    win = _concat_pools([w.win for w in parts])
    cmp = None if w0.cmp is None else _concat_pools([w.cmp for w in parts])
    return Workload(name=name or f"{w0.name}_x{len(parts)}", fp8=w0.fp8, decode=w0.decode,
                    num_heads=w0.num_heads, head_dim=w0.head_dim, window=w0.window,
                    topk=w0.topk, ratio=w0.ratio, page_size=w0.page_size, scale=w0.scale,
                    q=torch.cat([w.q for w in parts]),
                    positions=torch.cat([w.positions for w in parts]),
                    seq_of_token=torch.cat(sot), topk_idx=torch.cat([w.topk_idx for w in parts]),
                    win=win, cmp=cmp,
                    meta={"seed": [w.meta["seed"] for w in parts], "cmp_entries": cmp_entries,
                          "parts": len(parts)})


@dataclass
class KvWriteInputs:
    """New K/V rows of T tokens and the pages they go to (the paged KV write)."""
    k: torch.Tensor              # bf16 [T, D]
    v: torch.Tensor              # bf16 [T, D]
    positions: torch.Tensor      # int32 [T]
    seq_of_token: torch.Tensor   # int32 [T]
    block_table: torch.Tensor    # int32 [B, stride]
    num_blocks: int
    page_size: int


def kv_write_inputs(seq_positions: Sequence[np.ndarray], head_dim: int, page_size: int,
                    seed: int = 0, oversize: int = 2, specials: bool = True) -> KvWriteInputs:
    """Seeded inputs of a KV write: N(0,1) bf16 rows for tokens at the given positions of each
    sequence, random pages from a pool `oversize` times larger than needed.  With `specials`, a few
    rows are made awkward for the quantiser: all zeros, mixed signed zeros, one large element among
    tiny ones (subnormal codes), and values at the half-way points between e4m3 codes."""
    g = torch.Generator().manual_seed(seed)
    pos = np.concatenate([np.asarray(p, dtype=np.int64) for p in seq_positions])
    sid = np.concatenate([np.full(len(p), b, dtype=np.int64) for b, p in enumerate(seq_positions)])
    pages = [int(np.max(p)) // page_size + 1 if len(p) else 1 for p in seq_positions]
    num_blocks, table = _assign_pages(g, pages, oversize)
    T = len(pos)
    k = torch.randn(T, head_dim, generator=g)
    v = torch.randn(T, head_dim, generator=g)
    if specials and T >= 4:
        k[0] = 0.0
        v[0] = -0.0
        k[1, ::2] = -0.0
        k[1, 1::2] = 0.0
        k[1, 0] = 3.0
        k[2] = torch.randn(head_dim, generator=g) * 1e-4
        k[2, 5] = 1000.0
        # x = 448 * (m + 0.5) / 2^j / 448 * amax -> exact half-way points once divided by the scale
        v[3] = torch.tensor([((8 + (i % 8)) + 0.5) * 2.0 ** (-(i % 6)) for i in range(head_dim)])
        v[3, 0] = 448.0
    return KvWriteInputs(k.to(torch.bfloat16), v.to(torch.bfloat16),
                         torch.from_numpy(pos.astype(np.int32)),
                         torch.from_numpy(sid.astype(np.int32)), table, num_blocks, page_size)


# gated-pool shapes timed on the pages (FreeToken PR 633, "Kernel time": B, R, D)
GATED_POOL_SHAPES = [(b, r, d) for b in (1, 8) for r in (8, 128) for d in (128, 512)]


def gated_pool_inputs(B: int, R: int, D: int, seed: int = 0, gate_std: float = 2.0,
                      view: str = "dense"):
    """Seeded gated-pool inputs: kv ~ N(0,1) and gates ~ N(0, gate_std^2), fp32 [B, R, D].

    ``view`` makes strided views of larger buffers, as a compressor's state slices would be:
    "dense" (contiguous), "row_pad" (rows 8 floats apart more than D, i.e. a [B, R, D + 8] buffer
    cut to D), "every_other_row" (a [B, 2R, D] buffer, rows 0, 2, 4, ...), "odd_offset" (the view
    starts one float into its buffer, so rows are 4-byte but not 16-byte aligned).
    """
    g = torch.Generator().manual_seed(seed)

    def one(std):
        if view == "dense":
            t = torch.randn(B, R, D, generator=g) * std
            return t, t
        if view == "row_pad":
            buf = torch.randn(B, R, D + 8, generator=g) * std
            return buf, buf[:, :, :D]
        if view == "every_other_row":
            buf = torch.randn(B, 2 * R, D, generator=g) * std
            return buf, buf[:, ::2, :]
        if view == "odd_offset":
            buf = torch.randn(B * R * D + 1, generator=g) * std
            return buf, buf[1:].view(B, R, D)
        raise ValueError(view)
    kv_buf, kv = one(1.0)
    gate_buf, gate = one(gate_std)
    return kv_buf, kv, gate_buf, gate


# ----------------------------------------------------------------------------------------------
# indexer inputs (FreeToken PR 634: 32 index heads, index head_dim 128, fp4_e8m0_b32 key rows)
# ----------------------------------------------------------------------------------------------
INDEX_ROW_WORDS = 17
NAN_SCALES_WORD = -1       # 0xFFFFFFFF: all four ue8m0 scale bytes NaN (poison for stray reads)


@dataclass
class IndexerInputs:
    q: torch.Tensor             # bf16 [T, H, 128]
    weights: torch.Tensor       # fp32 [T, H]
    key_pool: torch.Tensor      # int32 [num_blocks, page_size, 17]
    block_table: torch.Tensor   # int32 [B, stride]
    positions: torch.Tensor     # int32 [T]
    seq_of_token: torch.Tensor  # int32 [T]
    ratio: int
    num_cols: int
    cand: Optional[torch.Tensor] = None   # int32 [T, num_cols] (candidate mode)

    @property
    def num_seqs(self) -> int:
        return int(self.block_table.shape[0])

    def seq_ids(self) -> np.ndarray:
        return self.seq_of_token.numpy().astype(np.int64)


def indexer_inputs(seq_positions: Sequence[np.ndarray], ratio: int, *, num_heads: int = 32,
                   page_size: int = 64, seed: int = 0, num_cols: Optional[int] = None,
                   cand_count: Optional[int] = None, cand_fill: str = "tail",
                   scale_exps=(121, 127), oversize: int = 2) -> IndexerInputs:
    """Seeded indexer inputs.

    Queries ~ N(0,1) in bf16, weights ~ N(0,1)/sqrt(H) in fp32.  Key rows of every compressed entry
    each sequence has (``(max position + 1) // ratio``): uniformly random e2m1 nibbles and ue8m0
    scale bytes drawn from ``scale_exps`` (inclusive), in random pages of a pool ``oversize`` times
    larger; spare rows carry NaN scales.  Full mode: ``num_cols`` defaults to the largest entry
    count.  Candidate mode (``cand_count``): per query a random choice of its causal entries,
    padded with -1 at the tail ("tail") or with -1 and non-causal entries scattered ("anywhere").
    """
    g = torch.Generator().manual_seed(seed)
    pos = np.concatenate([np.asarray(p, dtype=np.int64) for p in seq_positions])
    sid = np.concatenate([np.full(len(p), b, dtype=np.int64) for b, p in enumerate(seq_positions)])
    T = len(pos)
    entries = [max(0, (int(np.max(p)) + 1) // ratio) if len(p) else 0 for p in seq_positions]
    pages = [max(1, -(-e // page_size)) for e in entries]
    num_blocks, table = _assign_pages(g, pages, oversize)
    words = torch.randint(-(1 << 31), (1 << 31) - 1, (num_blocks * page_size, INDEX_ROW_WORDS),
                          generator=g, dtype=torch.int64)
    lo, hi = scale_exps
    sc = torch.randint(lo, hi + 1, (num_blocks * page_size, 4), generator=g, dtype=torch.int64)
    words[:, 16] = sc[:, 0] | (sc[:, 1] << 8) | (sc[:, 2] << 16) | (sc[:, 3] << 24)
    words = ((words + (1 << 31)) % (1 << 32) - (1 << 31)).to(torch.int32)
    used = torch.zeros(num_blocks, dtype=torch.bool)
    used[table[table >= 0].long()] = True
    rows_used = used.repeat_interleave(page_size)
    words[~rows_used, 16] = NAN_SCALES_WORD
    key_pool = words.view(num_blocks, page_size, INDEX_ROW_WORDS)
    q = torch.randn(T, num_heads, 128, generator=g).to(torch.bfloat16)
    weights = torch.randn(T, num_heads, generator=g) / float(np.sqrt(num_heads))
    cand = None
    if cand_count is None:
        ncols = max(entries) if num_cols is None else num_cols
    else:
        ncols = cand_count
        cand = torch.full((T, cand_count), -1, dtype=torch.int32)
        for t in range(T):
            valid = (int(pos[t]) + 1) // ratio
            k = min(valid, cand_count)
            pick = torch.randperm(valid, generator=g)[:k].to(torch.int32) if valid else \
                torch.empty(0, dtype=torch.int32)
            cand[t, :k] = pick
            if cand_fill == "anywhere" and cand_count >= 4:
                slots = torch.randperm(cand_count, generator=g)[:max(1, cand_count // 8)]
                cand[t, slots[0::2]] = -1
                cand[t, slots[1::2]] = int(pos[t]) // ratio + 1     # one entry past causality
    return IndexerInputs(q, weights, key_pool, table,
                         torch.from_numpy(pos.astype(np.int32)),
                         torch.from_numpy(sid.astype(np.int32)), ratio, ncols, cand)
