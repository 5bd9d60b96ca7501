"""Partition of a batch of queries across ranks (one process per GPU, no data-path collective).

Every query's result depends only on its own q, position, top-k list and the pool rows those
select, so the queries can be split across GPUs in any way, each GPU holding the pools (or the
pages its queries touch), and the union of the shards' outputs is the output of the whole batch.
Two partitions:

* ``"sequence"``: whole sequences, in contiguous groups of about equal size (decode batches, and
  batches of independent prefill sequences);
* ``"query_block"``: blocks of ``block`` consecutive queries dealt round-robin (one long prefill:
  later queries have more causally valid top-k entries, so interleaving balances the shards).
"""
from __future__ import annotations

from typing import Optional

import numpy as np

__all__ = ["shard_tokens"]


def shard_tokens(num_tokens: int, seq_of_token: Optional[np.ndarray], rank: int, world: int, *,
                 by: str = "sequence", block: int = 128) -> np.ndarray:
    """Indices (int64, increasing) of the queries of shard ``rank`` of ``world``.  Every query is
    in exactly one shard."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    idx = np.arange(num_tokens, dtype=np.int64)
    if by == "query_block":
        if block < 1:
            raise ValueError("block must be positive")
        return idx[(idx // block) % world == rank]
    if by != "sequence":
        raise ValueError(f"unknown partition {by!r}")
    sid = (np.zeros(num_tokens, dtype=np.int64) if seq_of_token is None
           else np.asarray(seq_of_token, dtype=np.int64))
    seqs = np.unique(sid)
    lo = (len(seqs) * rank) // world
    hi = (len(seqs) * (rank + 1)) // world
    return idx[np.isin(sid, seqs[lo:hi])]
