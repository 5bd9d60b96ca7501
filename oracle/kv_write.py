"""Paged KV write with e4m3 quantisation: the step that fills the pools the attention reads.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain numpy, recomputed from the
definitions; shares no code with the CUDA library.

What it follows:

* FreeToken PR 633, call paths and "Changes": a pool is [num_blocks][page_size][2][D], K row then V
  row per slot; a token at position x of sequence b lives in slot
  ``block_table[b][x // page_size] * page_size + x % page_size``.
* FreeToken clone PR 3, "Perf/kv fp8 read path", part 1: one fp32 scale per (token, kv_head),
  separately for K and V, with e4m3 codes whose value times the scale is the stored element; the
  largest e4m3 magnitude is 448.  Reading (the page prints no write kernel): the scale is
  ``max|x| / 448`` so that the largest element maps to 448, 1 for an all-zero row, and each code
  is the e4m3 value nearest to ``x / scale``.
* OCP 8-bit floating point specification, E4M3 ("fn"): bias 7, 3 mantissa bits, subnormals
  ``m * 2^-9``, no infinities, S.1111.111 NaN, largest finite 448; round to nearest, ties to the
  even mantissa.

Precision: the scale and the quotients are IEEE binary32 operations (numpy float32 arithmetic is
correctly rounded), because they decide integer codes and the write kernel takes them in fp32; the
rounding to e4m3 is then exact on the binary32 value.

Parity status: exact (integer codes and binary32 scales).  Pinned by tests/test_oracle_kv_write.py:
brute-force nearest-code search over every finite code, ties, saturation, zeros of either sign and
the subnormal range for the encoder; a hand-placed tiny write for the slot arithmetic.
"""
import numpy as np

from .sparse_attention import bf16_to_f64

E4M3_MAX = 448.0


def e4m3_encode_rne(x) -> np.ndarray:
    """Finite values -> OCP E4M3 codes: round to nearest, ties to even, saturating to +-448.

    The rounding quantum of a magnitude a is 2^(e-3) with e = floor(log2 a) for normals
    (2^-6 <= a), and 2^-9 below (subnormals, e clamped to -6); a / quantum is then rounded half to
    even (np.rint) and the result re-encoded as sign | exponent | mantissa.
    """
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x).astype(np.int64)
    a = np.abs(x)
    _, exp2 = np.frexp(np.where(a > 0, a, 1.0))          # a = f * 2^exp2, 0.5 <= f < 1
    e = np.clip(exp2 - 1, -6, 8)                           # floor(log2 a), clamped
    q = np.ldexp(1.0, e - 3)
    v = np.minimum(np.rint(a / q) * q, E4M3_MAX)           # rounded magnitude, saturated
    # encode v
    _, ve = np.frexp(np.where(v > 0, v, 1.0))
    ve = ve - 1                                            # floor(log2 v)
    sub = (v > 0) & (ve < -6)
    m_sub = np.rint(v / 2.0 ** -9).astype(np.int64)        # subnormal: v = m * 2^-9
    m_norm = np.rint(v / np.ldexp(1.0, ve - 3)).astype(np.int64) - 8
    exp_field = np.where(v == 0, 0, np.where(sub, 0, ve + 7))
    man_field = np.where(v == 0, 0, np.where(sub, m_sub, m_norm))
    return ((sign << 7) | (exp_field << 3) | man_field).astype(np.uint8)


def quantize_row_e4m3(x_f32: np.ndarray):
    """One row of binary32 values -> (e4m3 codes, binary32 scale)."""
    x = np.asarray(x_f32, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0)
    scale = np.float32(amax / np.float32(E4M3_MAX)) if amax > 0 else np.float32(1.0)
    return e4m3_encode_rne(x / scale), scale


def slot_of(x: int, b: int, block_table: np.ndarray, num_blocks: int, page_size: int):
    """The pool slot of position x of sequence b, or None (the token is dropped)."""
    if x < 0 or b < 0 or b >= block_table.shape[0]:
        return None
    page = x // page_size
    if page >= block_table.shape[1]:
        return None
    blk = int(block_table[b, page])
    if blk < 0 or blk >= num_blocks:
        return None
    return blk * page_size + x % page_size


def kv_write(k_bits, v_bits, positions, seq_of_token, block_table, pool_kv, *, page_size,
             k_scale=None, v_scale=None, fp8: bool):
    """Write the rows of T tokens into a pool, in place.

    ``k_bits``, ``v_bits``: bf16 bit patterns [T][D] (uint16).  ``pool_kv``: [num_blocks,
    page_size, 2, D], uint16 bf16 patterns (fp8 False) or uint8 codes (fp8 True), with
    ``k_scale``/``v_scale`` float32 [num_blocks * page_size].  Returns True when some token was
    dropped (the device error flag).
    """
    k_bits = np.asarray(k_bits, dtype=np.uint16)
    v_bits = np.asarray(v_bits, dtype=np.uint16)
    pos = np.asarray(positions, dtype=np.int64)
    T = k_bits.shape[0]
    sid = np.zeros(T, dtype=np.int64) if seq_of_token is None else np.asarray(seq_of_token,
                                                                               dtype=np.int64)
    bt = np.asarray(block_table, dtype=np.int64)
    nb = pool_kv.shape[0]
    flat = pool_kv.reshape(nb * page_size, 2, -1)
    dropped = False
    for t in range(T):
        row = slot_of(int(pos[t]), int(sid[t]), bt, nb, page_size)
        if row is None:
            dropped = True
            continue
        for kv, bits, scales in ((0, k_bits[t], k_scale), (1, v_bits[t], v_scale)):
            if not fp8:
                flat[row, kv] = bits
            else:
                x = bf16_to_f64(bits).astype(np.float32)   # exact: bf16 is a binary32 prefix
                codes, s = quantize_row_e4m3(x)
                flat[row, kv] = codes
                scales[row] = s
    return dropped
