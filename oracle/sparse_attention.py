"""Plain float64 restatement of sparse paged attention (test infrastructure only).

Column set of one query (sequence b, absolute position p), from the FreeToken PR 633 page
("Changes": the per-column choice between window pool and compressed pool) and the workload
descriptions on the same page ("128-token window, index top-k 512"):

* window columns c = 0 .. W-1 hold token ``p - W + 1 + c``; the column exists iff that token is
  >= 0.  Its row is ``win_bt[b][tok // ps] * ps + tok % ps`` in the window pool.
* top-k columns c = W .. W+K-1 hold compressed entry ``j = topk[t][c - W]``; the column exists iff
  ``j >= 0``, the ratio r > 0, and the entry is causal, ``r*j + r - 1 <= p`` (all the tokens it
  summarises are at or before p).  Its row is ``cmp_bt[b][j // ps] * ps + j % ps``.
* a column whose page lies outside its block table, or whose physical block is outside the pool,
  is an input error: it is dropped and the error flag is raised.

Attention over the existing columns is the textbook softmax: ``s_c = scale * q . k_c``,
``w = exp(s - max s) / sum exp(s - max s)``, ``out = sum_c w_c v_c``, ``lse = max s + ln sum``.
A query with no column gets ``out = 0`` and ``lse = -inf``.
"""
from __future__ import annotations

import numpy as np

# Column dump encoding: (pool << 30) | physical row; -1 where no column exists.
COL_POOL_SHIFT = 30


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float64.  bf16 is the top half of an IEEE binary32, so the value
    is the binary32 whose high 16 bits are ``bits`` and whose low 16 bits are zero."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):      # signalling-NaN patterns stay NaN
        return b.view(np.float32).astype(np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3 ("fn" variant) codes -> float64, from the format definition.

    sign = bit 7, exponent = bits 6..3 (bias 7), mantissa = bits 2..0.
    exponent 0: subnormal, (-1)^s * 2^-6 * m/8.  S.1111.111: NaN (no infinities).
    otherwise (-1)^s * 2^(e-7) * (1 + m/8).  Largest finite magnitude 448 (S.1111.110).
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    val = sign * val
    return np.where((e == 0xF) & ((c & 0x7) == 0x7), np.nan, val)


def resolve_columns(positions, seq_ids, win_bt, win_num_blocks, cmp_bt, cmp_num_blocks,
                    topk_idx, *, window: int, ratio: int, page_size: int):
    """Integer column list ``[T, W + K]`` in the dump encoding, and an input-error flag.

    Parity: exact (integer).  Pinned by a hand-derived example (tests/golden/resolve_small.json),
    by the logical-content check (every resolved row holds the token or entry it should) and by
    the column-count identity  #columns = min(p + 1, W) + #{valid top-k}.
    """
    pos = np.asarray(positions, dtype=np.int64)
    sid = np.asarray(seq_ids, dtype=np.int64)
    T = pos.shape[0]
    tk = np.asarray(topk_idx, dtype=np.int64).reshape(T, -1)
    K = tk.shape[1]
    cols = np.full((T, window + K), -1, dtype=np.int64)
    error = False
    p = pos[:, None]

    if window > 0:
        wbt = np.asarray(win_bt, dtype=np.int64)
        c = np.arange(window, dtype=np.int64)[None, :]
        tok = p - window + 1 + c
        exists = tok >= 0
        lp = np.where(exists, tok // page_size, 0)
        in_table = lp < wbt.shape[1]
        phys = wbt[sid[:, None], np.where(in_table, lp, 0)]
        ok = exists & in_table & (phys >= 0) & (phys < win_num_blocks)
        error |= bool(np.any(exists & ~ok))
        rows = phys * page_size + np.where(exists, tok % page_size, 0)
        cols[:, :window] = np.where(ok, rows, -1)

    if ratio > 0 and K > 0:
        cbt = np.asarray(cmp_bt, dtype=np.int64)
        j = tk
        exists = (j >= 0) & (ratio * j + ratio - 1 <= p)
        lp = np.where(exists, j // page_size, 0)
        in_table = lp < cbt.shape[1]
        phys = cbt[sid[:, None], np.where(in_table, lp, 0)]
        ok = exists & in_table & (phys >= 0) & (phys < cmp_num_blocks)
        error |= bool(np.any(exists & ~ok))
        rows = phys * page_size + np.where(exists, j % page_size, 0)
        cols[:, window:] = np.where(ok, (1 << COL_POOL_SHIFT) | rows, -1)
    return cols, error


def gather_rows(pool_kv, rows, *, fp8: bool, k_scale=None, v_scale=None):
    """K and V rows (float64) of the physical ``rows`` of one pool.

    ``pool_kv`` is ``[num_blocks, page_size, 2, D]``: bf16 bit patterns (uint16) or e4m3 codes
    (uint8).  For e4m3 the value is ``code_value * scale[row]`` with separate K and V scales
    (FreeToken clone PR 3, part 1: the scale is per (token, kv_head)).
    Parity: exact widening; pinned through the e4m3 and bf16 code tables.
    """
    D = pool_kv.shape[-1]
    flat = pool_kv.reshape(-1, 2, D)
    r = np.asarray(rows, dtype=np.int64)
    if fp8:
        k = e4m3_to_f64(flat[r, 0, :]) * np.asarray(k_scale, dtype=np.float64)[r][:, None]
        v = e4m3_to_f64(flat[r, 1, :]) * np.asarray(v_scale, dtype=np.float64)[r][:, None]
    else:
        k = bf16_to_f64(flat[r, 0, :])
        v = bf16_to_f64(flat[r, 1, :])
    return k, v


def attend(q, k, v, scale: float):
    """Softmax attention of every head of one query over the given columns.

    q: [H, D]; k, v: [C, D] float64.  Returns (out [H, D], lse [H]).
    Parity: the definition itself; pinned against dense brute-force masked attention, against
    torch's scaled_dot_product_attention (ratio 0) and against closed forms.
    """
    H, D = q.shape
    if k.shape[0] == 0:
        return np.zeros((H, D)), np.full(H, -np.inf)
    s = scale * (q @ k.T)                       # [H, C]
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    out = (e @ v) / l
    lse = m[:, 0] + np.log(l[:, 0])
    return out, lse


def _columns_of(cols_row):
    valid = cols_row >= 0
    pool = np.where(valid, cols_row >> COL_POOL_SHIFT, -1)
    row = np.where(valid, cols_row & ((1 << COL_POOL_SHIFT) - 1), -1)
    return pool[valid], row[valid]


def _query_kv(cols_row, win_kv, cmp_kv, fp8, win_k_scale, win_v_scale, cmp_k_scale,
              cmp_v_scale):
    pool, row = _columns_of(cols_row)
    D = win_kv.shape[-1]
    k = np.empty((len(row), D))
    v = np.empty((len(row), D))
    for pid, kv, ks, vs in ((0, win_kv, win_k_scale, win_v_scale),
                            (1, cmp_kv, cmp_k_scale, cmp_v_scale)):
        sel = pool == pid
        if np.any(sel):
            k[sel], v[sel] = gather_rows(kv, row[sel], fp8=fp8, k_scale=ks, v_scale=vs)
    return k, v


def sparse_paged_attention(q_bits, positions, seq_ids, win_kv, win_bt, cmp_kv, cmp_bt, topk_idx,
                           *, window: int, ratio: int, page_size: int, scale: float,
                           fp8: bool = False, win_k_scale=None, win_v_scale=None,
                           cmp_k_scale=None, cmp_v_scale=None, tokens=None):
    """Sparse paged attention of the queries listed in ``tokens`` (default: all).

    q_bits: uint16 bf16 patterns [T, H, D].  Pools as in ``gather_rows``; ``cmp_kv``/``cmp_bt``
    may be None when ratio == 0.  Returns (out [n, H, D], lse [n, H], cols [T, W+K], error).
    """
    pos = np.asarray(positions, dtype=np.int64)
    sid = np.asarray(seq_ids, dtype=np.int64)
    cols, error = resolve_columns(
        pos, sid, win_bt, win_kv.shape[0],
        cmp_bt if cmp_bt is not None else np.zeros((1, 1), np.int64),
        cmp_kv.shape[0] if cmp_kv is not None else 0,
        topk_idx, window=window, ratio=ratio, page_size=page_size)
    T, H, D = q_bits.shape
    idx = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    out = np.zeros((len(idx), H, D))
    lse = np.zeros((len(idx), H))
    for n, t in enumerate(idx):
        k, v = _query_kv(cols[t], win_kv, cmp_kv, fp8, win_k_scale, win_v_scale, cmp_k_scale,
                         cmp_v_scale)
        q = bf16_to_f64(q_bits[t])
        out[n], lse[n] = attend(q, k, v, scale)
    return out, lse, cols, error


def decode_split_k(q, k, v, scale: float, bounds):
    """Split-K partials of one query: for each column range [bounds[i], bounds[i+1]) the
    normalised partial output and its log-sum-exp (the 'splitk' decode of FreeToken PR 633,
    call paths).  Empty ranges give (0, -inf).  Parity: pinned by merge == single pass."""
    parts = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        parts.append(attend(q, k[a:b], v[a:b], scale))
    return parts


def merge_partials(parts):
    """Log-sum-exp merge of split partials: L = max_s lse_s, w_s = exp(lse_s - L),
    out = sum_s w_s O_s / sum_s w_s, lse = L + ln sum_s w_s.  Heads whose every partial is empty
    get out = 0, lse = -inf."""
    outs = np.stack([o for o, _ in parts])          # [S, H, D]
    lses = np.stack([l for _, l in parts])          # [S, H]
    H = lses.shape[1]
    out = np.zeros(outs.shape[1:])
    lse = np.full(H, -np.inf)
    for h in range(H):
        fin = np.isfinite(lses[:, h])
        if not np.any(fin):
            continue
        L = lses[fin, h].max()
        w = np.exp(lses[fin, h] - L)
        out[h] = (w[:, None] * outs[fin, h, :]).sum(axis=0) / w.sum()
        lse[h] = L + np.log(w.sum())
    return out, lse
