"""Float64 CPU oracle for DeepSeek-V4-style sparse paged attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or link this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its ``cpu_baseline`` leg and its
``--impl reference`` arm) use it.  It shares no code with the CUDA library: it takes plain numpy
arrays and recomputes everything from the definitions, in float64.

What it follows (sources are the pages' titles and sections):

* FreeToken PR 633, "perf(kernel): keep 16-byte kv loads in dsv4 sparse attention ...", call paths
  and "Changes": every query attends over one column set drawn from two paged pools; each column
  selects the window pool or the compressed pool and resolves its page.
* the same page, "Kernel time" (shapes) and "Correctness and tests" (edge cases: zero counts,
  the ratio-0 alias, pool views with a row offset).
* FreeToken clone PR 3, "Perf/kv fp8 read path", part 1: e4m3 K/V rows with a per-(token,
  kv_head) scale; scores and probabilities are the plain dequantised products.
* OCP 8-bit floating point specification, E4M3 ("fn": no infinities, S.1111.111 is NaN,
  max normal 448) and bfloat16 (the upper 16 bits of IEEE binary32).

Parity status of each function is stated in its docstring.  Every function below is pinned by
``tests/test_oracle_pins.py``; the paged KV write (``oracle.kv_write``: e4m3 encoding with round
to nearest even, one scale per row, slot placement) by ``tests/test_oracle_kv_write.py``; the
compressor's gated pool (``oracle.gated_pool``: a per-channel softmax over R rows weighting the kv
rows, a stated reading) by ``tests/test_oracle_gated_pool.py``; the indexer logits over packed fp4
key rows (``oracle.indexer``: OCP E2M1/E8M0 decoding, a stated logit reading) by
``tests/test_oracle_indexer.py``.
"""
from .sparse_attention import (  # noqa: F401
    COL_POOL_SHIFT,
    attend,
    bf16_to_f64,
    decode_split_k,
    e4m3_to_f64,
    gather_rows,
    merge_partials,
    resolve_columns,
    sparse_paged_attention,
)
from . import gated_pool, indexer, kv_write  # noqa: F401
