"""Gated pool of the KV compressor: a softmax-weighted sum over R rows, per channel.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain numpy in float64, recomputed from
the definition; shares no code with the CUDA library.

What it follows:

* FreeToken PR 633, call paths: the DeepSeek-V4 compressor's decode step calls ``gated_pool`` to
  fold R buffered rows into one compressed entry; "Changes": the kernel runs two loops over R, the
  first taking a maximum; "Kernel time": shapes B in {1, 8}, R in {8, 128}, D in {128, 512};
  "Correctness and tests": R = 1/3/5/7/9/16/127/129, D = 300/100/64, bf16 and fp32 outputs,
  strided input views.

Reading (the page prints no formula): the gate is a softmax over the R rows taken separately for
every channel, and the pooled value is the gate-weighted sum of the kv rows,

    out[b, d] = sum_r exp(score[b, r, d] - M[b, d]) * kv[b, r, d] / sum_r exp(score[b, r, d] - M[b, d])
    M[b, d]   = max_r score[b, r, d]

which is what a max pass followed by one exp-and-accumulate pass computes.  Inputs are binary32
(the compressor's running state); the output is binary32 or bf16 (round to nearest even).

Parity status: the formula is a reading, not fixed by the pages; the oracle's arithmetic is pinned
by tests/test_oracle_gated_pool.py to closed forms (R = 1, equal gates, one dominant gate, the
two-row logistic weight) and to invariants (a per-channel shift of the gates, a permutation of
the rows).
"""
import numpy as np


def gated_pool(kv, score) -> np.ndarray:
    """kv, score: [B, R, D] (any real dtype, widened to float64) -> pooled [B, D] in float64.

    R = 0 has no rows to weight: the result is 0 (the device kernel writes zeros too).
    """
    kv = np.asarray(kv, dtype=np.float64)
    score = np.asarray(score, dtype=np.float64)
    if kv.shape != score.shape or kv.ndim != 3:
        raise ValueError("kv and score must both be [B, R, D]")
    B, R, D = kv.shape
    out = np.zeros((B, D))
    if R == 0:
        return out
    for b in range(B):
        m = score[b].max(axis=0)                 # first pass over R: the per-channel maximum
        num = np.zeros(D)
        den = np.zeros(D)
        for r in range(R):                       # second pass: weights and weighted sum
            e = np.exp(score[b, r] - m)
            den += e
            num += e * kv[b, r]
        out[b] = num / den
    return out


def round_to_bf16_bits(x) -> np.ndarray:
    """float64 -> bf16 bit patterns (uint16), rounding to nearest even via binary32.

    Two roundings (f64 -> f32 -> bf16) match one direct rounding except at ties created by the
    first step; the kernel's output goes through the same two steps (fp32 result, then bf16).
    """
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    nan = np.isnan(f)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    return np.where(nan, np.uint16(0x7FC0), r)
