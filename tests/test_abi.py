"""The C ABI library: builds for sm_103a, loads, exports every declared symbol, and rejects bad
arguments on the host before touching the GPU (CPU only)."""
import ctypes
import glob
import os
import re

import pytest

import sparse_paged_attention_gb300 as spa
from sparse_paged_attention_gb300 import SpaPoolC, SpaProblemC

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(spa.library_path()):
        from sparse_paged_attention_gb300.build import build_library
        build_library()
    return spa.load_library()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(sparse_attn_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("sparse_attn_paged_prefill", "sparse_attn_paged_decode",
                 "sparse_attn_paged_prefill_fp8", "sparse_attn_paged_decode_fp8",
                 "sparse_attn_paged_resolve_columns", "sparse_attn_paged_check_errors",
                 "sparse_attn_paged_kv_write", "sparse_attn_paged_kv_write_fp8",
                 "sparse_attn_gated_pool"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_strerror_and_version(lib):
    for code, name in [(0, "SPA_OK"), (1, "SPA_ERR_NULL"), (2, "SPA_ERR_ALIGN"),
                       (4, "SPA_ERR_UNSUPPORTED"), (8, "SPA_ERR_INDEX"), (16, "SPA_ERR_TIMEOUT")]:
        assert spa.sparse_attn_paged_strerror(code).startswith(name)
    assert b"sm_103a" in lib.sparse_attn_paged_version()


@pytest.fixture
def no_device():
    """The validation tests below hand made-up device addresses to the entry points.  A call that
    passes host validation would launch a kernel on them, so they run only where no GPU is
    visible (the library then stops at its device query)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("made-up device addresses: host validation is tested without a GPU")


def _args(D=512, W=128, K=512, ratio=4, T=1, kv=0x1000, q=0x2000, out=0x3000):
    pool = SpaPoolC(kv, None, None, 0x4000, 64, 64, 16)
    cpool = SpaPoolC(kv, None, None, 0x5000, 64, 64, 16)
    prob = SpaProblemC(T, 1, 64, D, W, K, ratio, 0.04, 0x6000, None, 0x7000)
    return pool, cpool, prob, q, out


def _prefill(lib, pool, cpool, prob, q, out):
    return lib.sparse_attn_paged_prefill(q, ctypes.byref(pool),
                                         ctypes.byref(cpool) if cpool is not None else None,
                                         ctypes.byref(prob) if prob is not None else None, out,
                                         None)


def test_host_validation(lib, no_device):
    S = spa.SPA_STATUS
    pool, cpool, prob, q, out = _args()
    assert _prefill(lib, pool, cpool, None, q, out) == S["SPA_ERR_NULL"]
    assert _prefill(lib, pool, cpool, prob, None, out) == S["SPA_ERR_NULL"]
    assert _prefill(lib, pool, cpool, prob, q + 2, out) == S["SPA_ERR_ALIGN"]
    assert _prefill(lib, pool, cpool, prob, q, out + 8) == S["SPA_ERR_ALIGN"]
    p2, c2, *_ = _args(kv=0x1002)
    assert _prefill(lib, p2, c2, prob, q, out) == S["SPA_ERR_ALIGN"]
    assert _prefill(lib, pool, None, prob, q, out) == S["SPA_ERR_NULL"]       # ratio > 0 needs cmp
    for D in (32, 96, 576, 1024):
        _, _, pr, *_ = _args(D=D)
        assert _prefill(lib, pool, cpool, pr, q, out) == S["SPA_ERR_UNSUPPORTED"]
    _, _, pr, *_ = _args(W=600, K=600)
    assert _prefill(lib, pool, cpool, pr, q, out) == S["SPA_ERR_UNSUPPORTED"]
    # window + top-k past the int32 range must not wrap below the column limit
    _, _, pr, *_ = _args(W=2**31 - 1, K=2)
    assert _prefill(lib, pool, cpool, pr, q, out) == S["SPA_ERR_UNSUPPORTED"]
    assert lib.sparse_attn_paged_resolve_columns(ctypes.byref(pool), ctypes.byref(cpool),
                                                 ctypes.byref(pr), 0x8000, None) == \
        S["SPA_ERR_UNSUPPORTED"]
    _, _, pr, *_ = _args(W=-1)
    assert _prefill(lib, pool, cpool, pr, q, out) == S["SPA_ERR_SHAPE"]
    _, _, pr, *_ = _args(T=0)
    assert _prefill(lib, pool, cpool, pr, q, out) == S["SPA_OK"]             # nothing to do
    big = SpaPoolC(0x1000, None, None, 0x4000, 1 << 25, 64, 16)
    assert _prefill(lib, big, cpool, prob, q, out) == S["SPA_ERR_UNSUPPORTED"]
    # fp8 pools need their scales
    assert lib.sparse_attn_paged_prefill_fp8(q, ctypes.byref(pool), ctypes.byref(cpool),
                                             ctypes.byref(prob), out, None) == S["SPA_ERR_NULL"]
    # decode: with no device visible the call stops at the device query
    assert lib.sparse_attn_paged_decode(q, ctypes.byref(pool), ctypes.byref(cpool),
                                        ctypes.byref(prob), out, None, 0, None) in (
        S["SPA_ERR_NULL"], S["SPA_ERR_CUDA"])


def test_gated_pool_host_validation(lib, no_device):
    S = spa.SPA_STATUS
    f = lib.sparse_attn_gated_pool
    kv, g, out = 0x10000, 0x20000, 0x30000

    def call(kv=kv, g=g, B=8, R=128, D=512, sb=65536, sr=512, out=out, dt=0, osb=512):
        return f(kv, g, B, R, D, sb, sr, sb, sr, out, dt, osb, None)
    assert call(B=-1) == S["SPA_ERR_SHAPE"]
    assert call(R=-1) == S["SPA_ERR_SHAPE"]
    assert call(sr=-4) == S["SPA_ERR_SHAPE"]
    assert call(osb=-1) == S["SPA_ERR_SHAPE"]
    assert call(dt=2) == S["SPA_ERR_UNSUPPORTED"]
    assert call(B=0) == S["SPA_OK"] and call(D=0) == S["SPA_OK"]     # nothing to do
    assert call(kv=None) == S["SPA_ERR_NULL"] and call(out=None) == S["SPA_ERR_NULL"]
    assert call(kv=kv + 2) == S["SPA_ERR_ALIGN"] and call(g=g + 1) == S["SPA_ERR_ALIGN"]
    assert call(out=out + 2) == S["SPA_ERR_ALIGN"]                   # fp32 out: 4-byte aligned


def test_indexer_host_validation(lib, no_device):
    S = spa.SPA_STATUS
    f = lib.sparse_attn_indexer_logits
    keys = SpaPoolC(0x1000, None, None, 0x2000, 64, 64, 16)
    q, w, pos, out = 0x3000, 0x4000, 0x5000, 0x6000

    def call(q=q, w=w, T=4, H=32, keys=keys, pos=pos, B=1, r=2, cand=None, n=1024, out=out):
        return f(q, w, T, H, ctypes.byref(keys) if keys is not None else None, pos, None, B, r,
                 cand, n, out, None)
    assert call(T=-1) == S["SPA_ERR_SHAPE"] and call(n=-1) == S["SPA_ERR_SHAPE"]
    assert call(r=0) == S["SPA_ERR_SHAPE"] and call(B=0) == S["SPA_ERR_SHAPE"]
    assert call(H=16) == S["SPA_ERR_UNSUPPORTED"]
    assert call(T=0) == S["SPA_OK"] and call(n=0) == S["SPA_OK"]          # nothing to do
    assert call(q=None) == S["SPA_ERR_NULL"] and call(keys=None) == S["SPA_ERR_NULL"]
    assert call(out=None) == S["SPA_ERR_NULL"]
    assert call(q=q + 8) == S["SPA_ERR_ALIGN"] and call(out=out + 2) == S["SPA_ERR_ALIGN"]
    assert call(keys=SpaPoolC(0x1002, None, None, 0x2000, 64, 64, 16)) == S["SPA_ERR_ALIGN"]
    assert call(keys=SpaPoolC(0x1000, None, None, 0x2000, 0, 64, 16)) == S["SPA_ERR_SHAPE"]


def test_topk_host_validation(lib, no_device):
    S = spa.SPA_STATUS
    f = lib.sparse_attn_indexer_topk
    assert f(0x1000, -1, 10, None, 4, 0x2000, None) == S["SPA_ERR_SHAPE"]
    assert f(0x1000, 2, 10, None, -1, 0x2000, None) == S["SPA_ERR_SHAPE"]
    assert f(0x1000, 2, 10, None, 4096, 0x2000, None) == S["SPA_ERR_UNSUPPORTED"]
    assert f(0x1000, 0, 10, None, 4, 0x2000, None) == S["SPA_OK"]
    assert f(0x1000, 2, 10, None, 0, 0x2000, None) == S["SPA_OK"]
    assert f(None, 2, 10, None, 4, 0x2000, None) == S["SPA_ERR_NULL"]
    assert f(0x1000, 2, 10, None, 4, None, None) == S["SPA_ERR_NULL"]
    assert f(0x1002, 2, 10, None, 4, 0x2000, None) == S["SPA_ERR_ALIGN"]
    assert f(0x1000, 2, 10, 0x3001, 4, 0x2000, None) == S["SPA_ERR_ALIGN"]


def test_header_is_plain_c_and_every_entry_point_links(lib, tmp_path):
    """A C99 program that includes the header, takes the address of every declared entry point
    and links against the library builds and runs (it calls only the version query)."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    names = declared_functions()
    src = tmp_path / "abi.c"
    src.write_text(
        '#include "sparse_attn_paged.h"\n#include <stdio.h>\n'
        "typedef void (*fn)(void);\n"
        "int main(void) {\n"
        "  const fn all[] = {\n" + "".join(f"    (fn){n},\n" for n in names) + "  };\n"
        '  printf("%d %s\\n", (int)(sizeof all / sizeof all[0]), sparse_attn_paged_version());\n'
        "  return 0;\n}\n")
    exe = tmp_path / "abi"
    libdir = os.path.dirname(spa.library_path())
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror",
                        "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                        "-L", libdir, "-lspa_gb300", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    n, version = out.stdout.split(" ", 1)
    assert int(n) == len(names) and "sm_103a" in version


def test_host_prefill_staging_and_argument_checks(lib, no_device):
    """The host-buffer prefill: the staging size of a chunk (two slots, each q and out chunks
    in bf16, the top-k lists, positions and sequence ids, every part 256-byte aligned), and the
    argument checks made before any device work."""
    S = spa.SPA_STATUS
    T, H, D, K, chunk = 8192, 64, 512, 512, 1024
    prob = SpaProblemC(T, 1, H, D, 128, K, 4, 0.04, 0x6000, None, 0x7000)
    rows = chunk * H * D * 2                           # 64 MiB of bf16 rows per chunk
    slot = 2 * rows + chunk * K * 4 + 2 * 4096          # q, out, top-k lists, positions, seq ids
    assert lib.sparse_attn_paged_prefill_host_staging_size(ctypes.byref(prob), chunk) == 2 * slot
    # a chunk larger than the call is cut to the call; 3 tokens of 4-byte arrays take 256 bytes
    small = SpaProblemC(3, 1, 8, 64, 16, 32, 4, 0.1, 0x6000, None, 0x7000)
    assert lib.sparse_attn_paged_prefill_host_staging_size(ctypes.byref(small), 1000) == \
        2 * (2 * 3072 + 512 + 256 + 256)
    assert lib.sparse_attn_paged_prefill_host_staging_size(ctypes.byref(prob), 0) == 0
    assert lib.sparse_attn_paged_prefill_host_staging_size(None, chunk) == 0
    pool, cpool, pr, q, out = _args()
    f = lib.sparse_attn_paged_prefill_host
    need = lib.sparse_attn_paged_prefill_host_staging_size(ctypes.byref(pr), 64)
    call = lambda chunk, st, nbytes: f(q, ctypes.byref(pool), ctypes.byref(cpool),
                                       ctypes.byref(pr), out, chunk, st, nbytes, None)
    assert call(0, 0x100000, need) == S["SPA_ERR_SHAPE"]
    assert call(64, None, need) == S["SPA_ERR_NULL"]
    assert call(64, 0x100010, need) == S["SPA_ERR_ALIGN"]          # 16- but not 256-byte aligned
    assert call(64, 0x100000, need - 1) == S["SPA_ERR_WORKSPACE"]
    assert f(q, ctypes.byref(pool), ctypes.byref(cpool), None, out, 64, 0x100000, need,
             None) == S["SPA_ERR_NULL"]
    assert lib.sparse_attn_paged_prefill_host_fp8(q, ctypes.byref(pool), ctypes.byref(cpool),
                                                  ctypes.byref(pr), out, 64, 0x100000, need,
                                                  None) == S["SPA_ERR_NULL"]   # fp8 needs scales
