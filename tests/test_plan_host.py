"""Split plan of the decode path whose split-K partials live in global memory (a caller workspace
or the library's built-in scratch array), run on the CPU through a host build of the header the
library calls (sparse_paged_attention_gb300/csrc/spa_plan.h).

The number of splits follows the SM count, so the same problem needs more partial bytes on a GPU
with more SMs; a bounded buffer must bound the split count instead of failing on such a GPU.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SCRATCH = 16 << 20            # the no-allocation entry point's built-in array
MERGE_MAX_SPLITS = 32


@pytest.fixture(scope="module")
def plan_exe(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = tmp_path_factory.mktemp("plan") / "plan_host"
    r = subprocess.run([cxx, "-std=c++17", "-O2", "-I",
                        os.path.join(ROOT, "sparse_paged_attention_gb300", "csrc"),
                        os.path.join(ROOT, "tests", "plan_host.cpp"), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return str(exe)


def _plan(exe, cases):
    text = "".join(" ".join(str(v) for v in c) + "\n" for c in cases)
    out = subprocess.run([exe], input=text, capture_output=True, text=True, check=True).stdout
    return [tuple(int(v) for v in line.split()) for line in out.splitlines()]


def _bytes(T, H, D, S):
    a = lambda x: (x + 255) // 256 * 256
    return a(T * S * H * D * 4) + a(T * S * H * 4)


def test_split_count_follows_the_sm_count_without_a_cap(plan_exe):
    # decode B8, 64 heads, head_dim 512, 640 columns: 160 SMs want 20 splits (about 21 MiB)
    (s, c, b), = _plan(plan_exe, [(640, 8, 64, 512, 160, MERGE_MAX_SPLITS, 2 ** 63)])
    assert (s, c) == (20, 32) and b == _bytes(8, 64, 512, 20) > SCRATCH


@pytest.mark.parametrize("sms", [132, 148, 152, 160, 192, 264, 1024])
@pytest.mark.parametrize("T,C", [(1, 640), (8, 640), (8, 384), (8, 128), (4, 1024), (8, 1000)])
def test_capped_plan_fits_and_covers_every_column(plan_exe, sms, T, C):
    H, D = 64, 512
    (s, c, b), = _plan(plan_exe, [(C, T, H, D, sms, MERGE_MAX_SPLITS, SCRATCH)])
    assert b == _bytes(T, H, D, s)
    assert 1 <= s <= MERGE_MAX_SPLITS
    assert s * c >= C and (s - 1) * c < C           # every column in exactly one split
    if s > 1:
        assert b <= SCRATCH
    # the cap only removes splits: never more than the uncapped plan
    (s0, _, _), = _plan(plan_exe, [(C, T, H, D, sms, MERGE_MAX_SPLITS, 2 ** 63)])
    assert s <= s0
    if _bytes(T, H, D, s0) <= SCRATCH:
        assert s == s0


def test_one_split_when_nothing_smaller_fits(plan_exe):
    # 64 tokens x 128 heads x 512: one split alone is 16 MiB of O plus the LSEs, over the cap
    (s, c, b), = _plan(plan_exe, [(640, 64, 128, 512, 152, MERGE_MAX_SPLITS, SCRATCH)])
    assert (s, c) == (1, 640) and b > SCRATCH


@pytest.fixture(scope="module")
def chunks_exe(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = tmp_path_factory.mktemp("chunks") / "host_chunks"
    r = subprocess.run([cxx, "-std=c++17", "-O2", "-I",
                        os.path.join(ROOT, "sparse_paged_attention_gb300", "csrc"),
                        os.path.join(ROOT, "tests", "host_chunks.cpp"), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return str(exe)


def test_host_prefill_chunks_cover_every_token_once(chunks_exe):
    """The prefill from host buffers takes the tokens in order, a quarter chunk first and last
    and full chunks between: the chunks cover [0, T) exactly, each holds 1 to tc tokens (what a
    staging slot holds), and a long call is mostly full chunks."""
    cases = [(T, min(chunk, T)) for T in (1, 2, 3, 5, 7, 100, 255, 256, 257, 577, 1025, 2048,
                                          8191, 8192, 30001)
             for chunk in (1, 2, 3, 4, 5, 7, 128, 192, 300, 512, 1024, 4096)]
    text = "".join(f"{T} {tc}\n" for T, tc in cases)
    out = subprocess.run([chunks_exe], input=text, capture_output=True, text=True, check=True)
    lines = out.stdout.splitlines()
    assert len(lines) == len(cases)
    for (T, tc), line in zip(cases, lines):
        sizes = [int(v) for v in line.split()]
        assert sum(sizes) == T and all(1 <= n <= tc for n in sizes), (T, tc, sizes)
        if T >= 4 * tc >= 16:
            assert sizes[0] == tc // 4 and sizes.count(tc) >= len(sizes) - 3, (T, tc, sizes)
    sizes = [int(v) for v in lines[cases.index((8192, 1024))].split()]
    assert sizes == [256] + [1024] * 7 + [512, 256]
