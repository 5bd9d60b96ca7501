"""Indexer logits over packed fp4 key rows: the scores the top-k selection of compressed entries
is taken from.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain numpy in float64, recomputed from the
definitions; shares no code with the CUDA library.

What it follows:

* FreeToken PR 634, "perf(kernel): read dsv41 indexer key rows as int32 words", call path and
  "Changes": the indexer scores key rows stored as ``fp4_e8m0_b32`` at index head_dim 128, each
  row 17 int32 words, 16 words of e2m1 codes and 1 word of ue8m0 scales, one scale per 32
  elements; "Kernel time": 32 index heads, head_dim 128; Full mode scores every causal compressed
  entry, candidate mode a given list per query; "Correctness and tests": the dequantised value of
  every (code, scale) pair is a bf16 value, and code 0x8 is -0.
* OCP Microscaling Formats (MX) v1.0: E2M1 elements (sign, 2 exponent bits with bias 1, 1 mantissa
  bit; 0, 0.5, 1, 1.5, 2, 3, 4, 6; no inf or NaN) and the E8M0 scale (2^(e - 127), 0xFF is NaN).

Readings (the pages print neither the logit formula nor the row's byte order):

* element order: byte i of the 64 code bytes (words 0..15, little-endian) holds elements 2i (low
  nibble) and 2i + 1 (high nibble); scale byte g of word 16 (little-endian) scales elements
  32g .. 32g + 31.
* logit: ``logit[t, j] = sum_h w[t, h] * max(0, q[t, h, :] . k[j, :])`` with bf16 queries and
  fp32 per-head weights (the form of DeepSeek's sparse-attention indexer, whose V4.1 variant the
  page optimises; the page itself gives only the key format and the head counts).
* entries: entry j of sequence b has its key row in a pool paged like the compressed KV pool,
  ``block_table[b][j // ps] * ps + j % ps``; it is causal for a query at position p iff
  ``r * j + r - 1 <= p`` (the compressed-entry rule of the attention).  Non-causal, padded (-1) or
  beyond-the-list entries score -inf; a page beyond the table or a block beyond the pool is an
  input error (-inf and the error flag).

Parity status: the format decoding is pinned to the OCP definitions and hand-worked rows
(tests/test_oracle_indexer.py, tests/golden/e2m1_codes.json); the logit formula is a reading,
pinned by closed forms (unit queries read single key elements, ReLU clips negative scores, the
weights act linearly) and by the identity between candidate and full mode.  The top-k selection
(``topk_entries``) is pinned by a brute-force sort with many ties and by the validity of its lists
as attention top-k lists.
"""
import numpy as np

from .sparse_attention import bf16_to_f64

ROW_WORDS = 17        # 16 words of e2m1 codes + 1 word of ue8m0 scales, head_dim 128
INDEX_HEAD_DIM = 128
SCALE_BLOCK = 32


def e2m1_to_f64(codes) -> np.ndarray:
    """OCP E2M1 codes (low 4 bits) -> float64: sign bit 3, exponent bits 2..1 (bias 1), mantissa
    bit 0; exponent 0 is subnormal (m * 0.5)."""
    c = np.asarray(codes, dtype=np.int64) & 0xF
    sign = np.where(c & 0x8, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = (c & 0x1).astype(np.float64)
    mag = np.where(e == 0, m * 0.5, np.ldexp(1.0 + m / 2.0, e - 1))
    return sign * mag


def e8m0_to_f64(exps) -> np.ndarray:
    """OCP E8M0 scale bytes -> float64: 2^(e - 127); 0xFF is NaN."""
    e = np.asarray(exps, dtype=np.int64) & 0xFF
    return np.where(e == 0xFF, np.nan, np.ldexp(1.0, e - 127))


def unpack_rows(words) -> np.ndarray:
    """Packed rows [..., 17] (int32 words) -> dequantised keys [..., 128] in float64."""
    w = np.ascontiguousarray(np.asarray(words, dtype=np.int32))
    if w.shape[-1] != ROW_WORDS:
        raise ValueError("a packed fp4_e8m0_b32 row is 17 int32 words")
    by = w.view(np.uint8).reshape(*w.shape[:-1], ROW_WORDS * 4)   # little-endian bytes
    code_bytes = by[..., :64].astype(np.int64)
    codes = np.empty((*w.shape[:-1], INDEX_HEAD_DIM), dtype=np.int64)
    codes[..., 0::2] = code_bytes & 0xF
    codes[..., 1::2] = code_bytes >> 4
    scales = e8m0_to_f64(by[..., 64:68])                            # [..., 4]
    return e2m1_to_f64(codes) * np.repeat(scales, SCALE_BLOCK, axis=-1)


def entry_row(j: int, b: int, block_table: np.ndarray, num_blocks: int, page_size: int):
    """Pool row of compressed entry j of sequence b, or None when the page or block is invalid."""
    if b < 0 or b >= block_table.shape[0]:
        return None
    page = j // page_size
    if page >= block_table.shape[1]:
        return None
    blk = int(block_table[b, page])
    if blk < 0 or blk >= num_blocks:
        return None
    return blk * page_size + j % page_size


def indexer_logits(q_bits, weights, key_pool, block_table, positions, seq_ids, *, ratio: int,
                   num_cols: int, cand=None, tokens=None):
    """Logits [n, num_cols] (float64, -inf where no entry is scored) and the input-error flag.

    q_bits: bf16 patterns [T, H, 128]; weights: [T, H]; key_pool: int32 [num_blocks, page_size, 17];
    block_table: [B, stride]; positions, seq_ids: [T].  Full mode (cand None): column c is entry c.
    Candidate mode: column c is entry ``cand[t, c]`` (-1: none).  ``tokens`` limits the queries.
    """
    q = bf16_to_f64(q_bits)
    wts = np.asarray(weights, dtype=np.float64)
    pool = np.asarray(key_pool, dtype=np.int32)
    nb, ps = pool.shape[0], pool.shape[1]
    flat = pool.reshape(nb * ps, ROW_WORDS)
    bt = np.asarray(block_table, dtype=np.int64)
    pos = np.asarray(positions, dtype=np.int64)
    sid = np.asarray(seq_ids, dtype=np.int64)
    T = q.shape[0]
    idx = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    out = np.full((len(idx), num_cols), -np.inf)
    error = False
    for n, t in enumerate(idx):
        p, b = int(pos[t]), int(sid[t])
        cols, rows = [], []
        for c in range(num_cols):
            j = c if cand is None else int(cand[t, c])
            if j < 0 or ratio < 1 or ratio * j + ratio - 1 > p:
                continue
            row = entry_row(j, b, bt, nb, ps)
            if row is None:
                error = True
                continue
            cols.append(c)
            rows.append(row)
        if not cols:
            continue
        k = unpack_rows(flat[np.asarray(rows)])            # [n_cols, 128]
        s = k @ q[t].T                                     # [n_cols, H] per-head scores
        out[n, np.asarray(cols)] = np.maximum(s, 0.0) @ wts[t]
    return out, error


def topk_entries(logits, k: int, cand=None) -> np.ndarray:
    """The top-k selection that follows the logits: for each query, the k scored entries with the
    largest logits, in decreasing order of logit, ties going to the smaller entry index; -1 fills
    the list when fewer than k entries were scored (finite logit).  ``cand`` maps candidate
    columns to entry ids (Full mode: column c is entry c).  Returns int32 [T, k], usable as the
    attention's top-k list.

    Reading: the page names a top-k step after the logits (its test list has a top-k test) but
    prints no rule; this is the plain one, with the tie rule made explicit so that the list is
    unique.
    """
    lg = np.asarray(logits, dtype=np.float64)
    T, n = lg.shape
    ids = np.broadcast_to(np.arange(n), (T, n)) if cand is None else np.asarray(cand, np.int64)
    out = np.full((T, k), -1, dtype=np.int32)
    for t in range(T):
        ok = np.isfinite(lg[t])
        vals, ents = lg[t][ok], ids[t][ok]
        order = np.lexsort((ents, -vals))          # by logit descending, then entry ascending
        take = order[:k]
        out[t, :len(take)] = ents[take]
    return out
