"""The indexer kernels' element arithmetic, run on the CPU through a host build of the very header
the kernels include (sparse_paged_attention_gb300/csrc/spa_indexer_math.cuh), against the oracle.

* fp4_e8m0_b32 decoding: every E2M1 code times every E8M0 scale byte gives the bf16 bits of the
  oracle's exact value (FreeToken PR 634, "Correctness and tests": every code/scale pair is a bf16
  value; past the bf16 range the product is inf in both, and scale 0xFF is NaN).
* the top-k order key: sorting scored entries by it gives the oracle's top-k order (decreasing
  logit, ties to the smaller entry, -0 equal to +0, only finite logits scored).
"""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from oracle import indexer as oi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def host_exe(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = tmp_path_factory.mktemp("imh") / "indexer_math_host"
    r = subprocess.run([nvcc, "-std=c++17", "-O2",
                        "-I", os.path.join(ROOT, "sparse_paged_attention_gb300", "csrc"),
                        os.path.join(ROOT, "tests", "indexer_math_host.cu"), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return str(exe)


def test_decode_matches_the_oracle_for_every_code_and_scale(host_exe):
    out = subprocess.run([host_exe, "decode"], capture_output=True, text=True, check=True).stdout
    rows = [line.split() for line in out.splitlines()]
    assert len(rows) == 16 * 256
    codes = np.array([int(r[0], 16) for r in rows])
    scales = np.array([int(r[1], 16) for r in rows])
    got = np.array([int(r[2], 16) for r in rows], dtype=np.uint16)
    want_f = oi.e2m1_to_f64(codes) * oi.e8m0_to_f64(scales)
    want = torch.from_numpy(want_f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(want_f)
    assert (scales[nan] == 255).all()
    got_f = torch.from_numpy(got.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.isnan(got_f[nan]).all()
    assert np.array_equal(got[~nan], want[~nan])


def test_order_key_gives_the_oracle_top_k_order(host_exe):
    rng = np.random.default_rng(40)
    n = 3000
    vals = np.concatenate([
        rng.integers(-3, 4, n // 2).astype(np.float32),                   # many ties
        (rng.standard_normal(n // 2) * np.exp2(rng.integers(-140, 120, n // 2))).astype(np.float32),
    ])
    specials = np.array([0.0, -0.0, -np.inf, np.inf, np.nan, 3.4028235e38, -3.4028235e38,
                         1e-45, -1e-45], dtype=np.float32)
    vals[:len(specials)] = specials
    ids = rng.permutation(1 << 20)[:n].astype(np.uint32)
    stdin = "".join(f"{int(b):x} {int(i)}\n" for b, i in zip(vals.view(np.uint32), ids))
    out = subprocess.run([host_exe, "keys"], input=stdin, capture_output=True, text=True,
                         check=True).stdout.split()
    assert len(out) == n
    scored = np.array([k != "-" for k in out])
    assert np.array_equal(scored, np.isfinite(vals))
    keys = [int(k, 16) for k in out if k != "-"]
    order = np.array(ids[scored])[np.argsort(np.array(keys, dtype=np.uint64))[::-1]]
    want = oi.topk_entries(vals[None].astype(np.float64), int(scored.sum()),
                           cand=ids[None].astype(np.int64))[0]
    assert np.array_equal(order, want.astype(np.int64))
