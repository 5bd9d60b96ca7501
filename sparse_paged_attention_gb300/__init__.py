"""GB300 (sm_103a) sparse paged attention: a thin ctypes binding over the C ABI.

The C ABI is declared in ``include/sparse_attn_paged.h``; this module only marshals torch tensors
into its plain pointers and sizes (every step of the computation runs in the library's CUDA
kernels).  The shared library is built in-tree by ``sparse_paged_attention_gb300.build`` and is
loaded on first use; when it is missing every call raises, there is no other code path.

Pools are any object with ``kv`` ([num_blocks, page_size, 2, head_dim] bf16 or uint8 e4m3 codes),
``block_table`` (int32 [num_seqs, stride]) and, for e4m3 pools, ``k_scale``/``v_scale`` (fp32
[num_blocks * page_size]) attributes, e.g. :class:`PagedPool`.
"""
from __future__ import annotations

import ctypes
import os
from typing import NamedTuple, Optional

import torch

__all__ = [
    "PagedPool", "SpaError", "library_path", "load_library", "sparse_attn_paged_prefill",
    "sparse_attn_paged_prefill_fp8", "sparse_attn_paged_decode", "sparse_attn_paged_decode_fp8",
    "sparse_attn_paged_decode_workspace_size", "sparse_attn_paged_decode_noalloc",
    "sparse_attn_paged_resolve_columns", "sparse_attn_paged_kv_write",
    "sparse_attn_paged_kv_write_fp8", "sparse_attn_gated_pool", "sparse_attn_indexer_logits",
    "sparse_attn_indexer_topk", "sparse_attn_paged_prefill_host",
    "sparse_attn_paged_prefill_host_fp8", "BoundCall", "bind_prefill", "bind_prefill_host",
    "bind_decode",
    "sparse_attn_paged_check_errors", "sparse_attn_paged_strerror", "SPA_STATUS",
]

SPA_STATUS = {
    "SPA_OK": 0, "SPA_ERR_NULL": 1, "SPA_ERR_ALIGN": 2, "SPA_ERR_SHAPE": 3,
    "SPA_ERR_UNSUPPORTED": 4, "SPA_ERR_WORKSPACE": 5, "SPA_ERR_CUDA": 6, "SPA_ERR_INDEX": 8,
    "SPA_ERR_TIMEOUT": 16,
}

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_HERE, "_lib", "libspa_gb300.so")


class SpaPoolC(ctypes.Structure):
    _fields_ = [("kv", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int64), ("page_size", ctypes.c_int32),
                ("bt_stride", ctypes.c_int32)]


class SpaProblemC(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int32), ("num_seqs", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("window", ctypes.c_int32), ("topk", ctypes.c_int32), ("ratio", ctypes.c_int32),
                ("scale", ctypes.c_float), ("positions", ctypes.c_void_p),
                ("seq_of_token", ctypes.c_void_p), ("topk_idx", ctypes.c_void_p)]


class SpaError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load_library()
        msg = lib.sparse_attn_paged_strerror(status).decode()
        if status == SPA_STATUS["SPA_ERR_CUDA"]:
            msg += ": " + lib.sparse_attn_paged_last_cuda_error().decode()
        super().__init__(f"{where}: {msg}")
        self.status = status


_lib = None


def load_library():
    """Load the in-tree shared library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m sparse_paged_attention_gb300.build`")
    lib = ctypes.CDLL(path)
    P, PP, PR = ctypes.c_void_p, ctypes.POINTER(SpaPoolC), ctypes.POINTER(SpaProblemC)
    for name in ("sparse_attn_paged_prefill", "sparse_attn_paged_prefill_fp8"):
        f = getattr(lib, name)
        f.argtypes = [P, PP, PP, PR, P, P]
        f.restype = ctypes.c_int
    for name in ("sparse_attn_paged_decode", "sparse_attn_paged_decode_fp8"):
        f = getattr(lib, name)
        f.argtypes = [P, PP, PP, PR, P, P, ctypes.c_size_t, P]
        f.restype = ctypes.c_int
    lib.sparse_attn_paged_prefill_host_staging_size.argtypes = [PR, ctypes.c_int32]
    lib.sparse_attn_paged_prefill_host_staging_size.restype = ctypes.c_size_t
    for name in ("sparse_attn_paged_prefill_host", "sparse_attn_paged_prefill_host_fp8"):
        f = getattr(lib, name)
        f.argtypes = [P, PP, PP, PR, P, ctypes.c_int32, P, ctypes.c_size_t, P]
        f.restype = ctypes.c_int
    lib.sparse_attn_paged_decode_noalloc.argtypes = [P, PP, PP, PR, P, P]
    lib.sparse_attn_paged_decode_noalloc.restype = ctypes.c_int
    lib.sparse_attn_paged_decode_workspace_size.argtypes = [PR]
    lib.sparse_attn_paged_decode_workspace_size.restype = ctypes.c_size_t
    lib.sparse_attn_paged_resolve_columns.argtypes = [PP, PP, PR, P, P]
    lib.sparse_attn_paged_resolve_columns.restype = ctypes.c_int
    I32 = ctypes.c_int32
    for name in ("sparse_attn_paged_kv_write", "sparse_attn_paged_kv_write_fp8"):
        f = getattr(lib, name)
        f.argtypes = [P, P, I32, I32, P, P, I32, PP, P]
        f.restype = ctypes.c_int
    I64 = ctypes.c_int64
    lib.sparse_attn_gated_pool.argtypes = [P, P, I32, I32, I32, I64, I64, I64, I64, P, I32, I64, P]
    lib.sparse_attn_gated_pool.restype = ctypes.c_int
    lib.sparse_attn_indexer_logits.argtypes = [P, P, I32, I32, PP, P, P, I32, I32, P, I32, P, P]
    lib.sparse_attn_indexer_logits.restype = ctypes.c_int
    lib.sparse_attn_indexer_topk.argtypes = [P, I32, I32, P, I32, P, P]
    lib.sparse_attn_indexer_topk.restype = ctypes.c_int
    lib.sparse_attn_paged_check_errors.argtypes = [P]
    lib.sparse_attn_paged_check_errors.restype = ctypes.c_int
    lib.sparse_attn_paged_strerror.argtypes = [ctypes.c_int]
    lib.sparse_attn_paged_strerror.restype = ctypes.c_char_p
    lib.sparse_attn_paged_last_cuda_error.argtypes = []
    lib.sparse_attn_paged_last_cuda_error.restype = ctypes.c_char_p
    lib.sparse_attn_paged_version.argtypes = []
    lib.sparse_attn_paged_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


class PagedPool(NamedTuple):
    kv: torch.Tensor
    block_table: torch.Tensor
    k_scale: Optional[torch.Tensor] = None
    v_scale: Optional[torch.Tensor] = None


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _pool_c(pool, fp8: bool) -> Optional[SpaPoolC]:
    if pool is None:
        return None
    kv, bt = pool.kv, pool.block_table
    want = torch.uint8 if fp8 else torch.bfloat16
    if kv.dtype != want:
        raise TypeError(f"pool kv must be {want}, got {kv.dtype}")
    if kv.dim() != 4 or kv.shape[2] != 2 or not kv.is_contiguous():
        raise ValueError("pool kv must be a contiguous [num_blocks, page_size, 2, head_dim] tensor")
    if bt.dtype != torch.int32 or bt.dim() != 2 or not bt.is_contiguous():
        raise ValueError("block_table must be a contiguous int32 [num_seqs, stride] tensor")
    ks = getattr(pool, "k_scale", None) if fp8 else None
    vs = getattr(pool, "v_scale", None) if fp8 else None
    return SpaPoolC(kv.data_ptr(), _ptr(ks), _ptr(vs), bt.data_ptr(), kv.shape[0], kv.shape[1],
                    bt.shape[1])


def _problem_c(q, win, topk_idx, positions, seq_of_token, window, ratio, scale, num_seqs):
    T, H, D = q.shape
    K = 0 if topk_idx is None else int(topk_idx.shape[1])
    for name, t in (("positions", positions), ("topk_idx", topk_idx), ("seq_of_token", seq_of_token)):
        if t is not None and (t.dtype != torch.int32 or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous int32 tensor")
    B = int(win.block_table.shape[0]) if num_seqs is None else int(num_seqs)
    return SpaProblemC(T, B, H, D, int(window), K, int(ratio), float(scale), positions.data_ptr(),
                       _ptr(seq_of_token), _ptr(topk_idx) if K > 0 else None)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check_q(q):
    if q.dtype != torch.bfloat16 or q.dim() != 3 or not q.is_contiguous():
        raise ValueError("q must be a contiguous bf16 [num_tokens, num_heads, head_dim] tensor")


def _prefill(fp8, q, win, cmp, topk_idx, positions, *, window, ratio, scale, seq_of_token=None,
             out=None, num_seqs=None, stream=None):
    lib = load_library()
    _check_q(q)
    if out is None:
        out = torch.empty_like(q)
    prob = _problem_c(q, win, topk_idx, positions, seq_of_token, window, ratio, scale, num_seqs)
    w, c = _pool_c(win, fp8), _pool_c(cmp, fp8)
    fn = lib.sparse_attn_paged_prefill_fp8 if fp8 else lib.sparse_attn_paged_prefill
    st = fn(q.data_ptr(), ctypes.byref(w), ctypes.byref(c) if c is not None else None,
            ctypes.byref(prob), out.data_ptr(), _stream(stream))
    if st != 0:
        raise SpaError(st, fn.__name__)
    return out


def sparse_attn_paged_prefill(q, win, cmp, topk_idx, positions, **kw):
    """out[T, H, D] (bf16) of sparse paged attention, one pass per query (see the C header)."""
    return _prefill(False, q, win, cmp, topk_idx, positions, **kw)


def sparse_attn_paged_prefill_fp8(q, win, cmp, topk_idx, positions, **kw):
    """Same with e4m3 pools (uint8 codes plus fp32 k_scale/v_scale per row)."""
    return _prefill(True, q, win, cmp, topk_idx, positions, **kw)


def sparse_attn_paged_decode_workspace_size(q, win, topk_idx, positions, *, window, ratio, scale,
                                            seq_of_token=None, num_seqs=None) -> int:
    lib = load_library()
    prob = _problem_c(q, win, topk_idx, positions, seq_of_token, window, ratio, scale, num_seqs)
    return int(lib.sparse_attn_paged_decode_workspace_size(ctypes.byref(prob)))


def _decode(fp8, q, win, cmp, topk_idx, positions, *, window, ratio, scale, seq_of_token=None,
            out=None, workspace=None, num_seqs=None, stream=None):
    lib = load_library()
    _check_q(q)
    if out is None:
        out = torch.empty_like(q)
    prob = _problem_c(q, win, topk_idx, positions, seq_of_token, window, ratio, scale, num_seqs)
    if workspace is None:
        nbytes = int(lib.sparse_attn_paged_decode_workspace_size(ctypes.byref(prob)))
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    w, c = _pool_c(win, fp8), _pool_c(cmp, fp8)
    fn = lib.sparse_attn_paged_decode_fp8 if fp8 else lib.sparse_attn_paged_decode
    st = fn(q.data_ptr(), ctypes.byref(w), ctypes.byref(c) if c is not None else None,
            ctypes.byref(prob), out.data_ptr(), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream(stream))
    if st != 0:
        raise SpaError(st, fn.__name__)
    return out


def sparse_attn_paged_decode(q, win, cmp, topk_idx, positions, **kw):
    """Split-K decode plus log-sum-exp merge; allocates the workspace with torch if none given."""
    return _decode(False, q, win, cmp, topk_idx, positions, **kw)


def sparse_attn_paged_decode_fp8(q, win, cmp, topk_idx, positions, **kw):
    return _decode(True, q, win, cmp, topk_idx, positions, **kw)


def sparse_attn_paged_decode_noalloc(q, win, cmp, topk_idx, positions, *, window, ratio, scale,
                                     seq_of_token=None, out=None, num_seqs=None, stream=None):
    """Decode whose split-K partials use the library's built-in scratch array instead of a
    workspace (for callers that cannot allocate device memory where they decode).  `out` must be
    passed by such a caller; without it this wrapper allocates one with torch for convenience."""
    lib = load_library()
    _check_q(q)
    if out is None:
        out = torch.empty_like(q)
    prob = _problem_c(q, win, topk_idx, positions, seq_of_token, window, ratio, scale, num_seqs)
    w, c = _pool_c(win, False), _pool_c(cmp, False)
    st = lib.sparse_attn_paged_decode_noalloc(q.data_ptr(), ctypes.byref(w),
                                              ctypes.byref(c) if c is not None else None,
                                              ctypes.byref(prob), out.data_ptr(), _stream(stream))
    if st != 0:
        raise SpaError(st, "sparse_attn_paged_decode_noalloc")
    return out


def _kv_write(fp8, k, v, positions, pool, *, seq_of_token=None, num_seqs=None, stream=None):
    lib = load_library()
    for name, t in (("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or t.dim() != 2 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 [num_tokens, head_dim] tensor")
    if k.shape != v.shape:
        raise ValueError("k and v must have the same shape")
    for name, t in (("positions", positions), ("seq_of_token", seq_of_token)):
        if t is not None and (t.dtype != torch.int32 or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous int32 tensor")
    T, D = int(k.shape[0]), int(k.shape[1])
    B = int(pool.block_table.shape[0]) if num_seqs is None else int(num_seqs)
    c = _pool_c(pool, fp8)
    fn = lib.sparse_attn_paged_kv_write_fp8 if fp8 else lib.sparse_attn_paged_kv_write
    st = fn(k.data_ptr(), v.data_ptr(), T, D, positions.data_ptr(), _ptr(seq_of_token), B,
            ctypes.byref(c), _stream(stream))
    if st != 0:
        raise SpaError(st, fn.__name__)


class BoundCall:
    """One attention call with its C argument structs built once.

    Calling the object re-issues the same C call on the same tensors (whose contents may change
    between calls), with no per-call marshalling: what a serving loop or a timing loop wants.  The
    call goes to the stream given at bind time, or, if none was given, to torch's current stream at
    the time of the call (so that it can be recorded into a CUDA graph on the capturing stream).
    The tensors are referenced here, so they stay alive as long as the object does.
    """

    def __init__(self, fn, args, keep, stream=None):
        self._fn, self._args, self._keep = fn, args, keep
        self._stream = None if stream is None else _stream(stream)

    def __call__(self):
        s = self._stream if self._stream is not None else \
            torch.cuda.current_stream().cuda_stream
        st = self._fn(*self._args, s)
        if st != 0:
            raise SpaError(st, self._fn.__name__)


def bind_prefill(q, win, cmp, topk_idx, positions, *, window, ratio, scale, seq_of_token=None,
                 out=None, num_seqs=None, stream=None, fp8=False) -> BoundCall:
    """``sparse_attn_paged_prefill[_fp8]`` on fixed tensors, as a zero-argument callable."""
    lib = load_library()
    _check_q(q)
    if out is None:
        out = torch.empty_like(q)
    prob = _problem_c(q, win, topk_idx, positions, seq_of_token, window, ratio, scale, num_seqs)
    w, c = _pool_c(win, fp8), _pool_c(cmp, fp8)
    fn = lib.sparse_attn_paged_prefill_fp8 if fp8 else lib.sparse_attn_paged_prefill
    args = (q.data_ptr(), ctypes.byref(w), ctypes.byref(c) if c is not None else None,
            ctypes.byref(prob), out.data_ptr())
    call = BoundCall(fn, args, (q, win, cmp, topk_idx, positions, seq_of_token, out, w, c, prob),
                     stream)
    call.out = out
    return call


def bind_prefill_host(q, win, cmp, topk_idx, positions, *, window, ratio, scale,
                      seq_of_token=None, out=None, num_seqs=None, chunk_tokens=1024, staging=None,
                      stream=None, fp8=False) -> BoundCall:
    """``sparse_attn_paged_prefill_host[_fp8]`` on fixed tensors, as a zero-argument callable.

    q, topk_idx, positions, seq_of_token and out are CPU tensors (page-locked, ``pin_memory()``,
    for the copies to overlap); the pools are on the GPU.  The device staging memory is allocated
    here once when not given.  ``call.out`` is complete once the call's stream has reached the
    point after the call."""
    lib = load_library()
    _check_q(q)
    for name, t in (("q", q), ("positions", positions), ("topk_idx", topk_idx),
                    ("seq_of_token", seq_of_token), ("out", out)):
        if t is not None and t.is_cuda:
            raise ValueError(f"{name} must be a host tensor")
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    if out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 host tensor shaped like q")
    prob = _problem_c(q, win, topk_idx, positions, seq_of_token, window, ratio, scale, num_seqs)
    if staging is None:
        nbytes = int(lib.sparse_attn_paged_prefill_host_staging_size(ctypes.byref(prob),
                                                                     int(chunk_tokens)))
        staging = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=win.kv.device)
    w, c = _pool_c(win, fp8), _pool_c(cmp, fp8)
    fn = lib.sparse_attn_paged_prefill_host_fp8 if fp8 else lib.sparse_attn_paged_prefill_host
    args = (q.data_ptr(), ctypes.byref(w), ctypes.byref(c) if c is not None else None,
            ctypes.byref(prob), out.data_ptr(), int(chunk_tokens), staging.data_ptr(),
            staging.numel() * staging.element_size())
    call = BoundCall(fn, args, (q, win, cmp, topk_idx, positions, seq_of_token, out, staging,
                                w, c, prob), stream)
    call.out = out
    call.staging = staging
    return call


def sparse_attn_paged_prefill_host(q, win, cmp, topk_idx, positions, **kw):
    """Prefill from host tensors (q, top-k lists, positions, out on the CPU; pools on the GPU),
    chunk by chunk through device staging memory, copies and kernels overlapping; returns the
    host output (complete once the stream has passed the call: synchronise before reading)."""
    call = bind_prefill_host(q, win, cmp, topk_idx, positions, **kw)
    call()
    return call.out


def sparse_attn_paged_prefill_host_fp8(q, win, cmp, topk_idx, positions, **kw):
    return sparse_attn_paged_prefill_host(q, win, cmp, topk_idx, positions, fp8=True, **kw)


def bind_decode(q, win, cmp, topk_idx, positions, *, window, ratio, scale, seq_of_token=None,
                out=None, workspace=None, num_seqs=None, stream=None, fp8=False) -> BoundCall:
    """``sparse_attn_paged_decode[_fp8]`` on fixed tensors, as a zero-argument callable (the
    workspace, when the plan needs one, is allocated here once)."""
    lib = load_library()
    _check_q(q)
    if out is None:
        out = torch.empty_like(q)
    prob = _problem_c(q, win, topk_idx, positions, seq_of_token, window, ratio, scale, num_seqs)
    if workspace is None:
        nbytes = int(lib.sparse_attn_paged_decode_workspace_size(ctypes.byref(prob)))
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    w, c = _pool_c(win, fp8), _pool_c(cmp, fp8)
    fn = lib.sparse_attn_paged_decode_fp8 if fp8 else lib.sparse_attn_paged_decode
    args = (q.data_ptr(), ctypes.byref(w), ctypes.byref(c) if c is not None else None,
            ctypes.byref(prob), out.data_ptr(), workspace.data_ptr(),
            workspace.numel() * workspace.element_size())
    call = BoundCall(fn, args, (q, win, cmp, topk_idx, positions, seq_of_token, out, workspace,
                                w, c, prob), stream)
    call.out = out
    call.workspace = workspace
    return call


def sparse_attn_paged_kv_write(k, v, positions, pool, **kw):
    """Copy the K and V rows of new tokens (bf16 [T, D]) into their slots of a bf16 pool."""
    _kv_write(False, k, v, positions, pool, **kw)


def sparse_attn_paged_kv_write_fp8(k, v, positions, pool, **kw):
    """Quantise the K and V rows of new tokens to e4m3 (one scale per row) into an e4m3 pool."""
    _kv_write(True, k, v, positions, pool, **kw)


def sparse_attn_gated_pool(kv, gate, out=None, *, out_dtype=torch.float32, stream=None):
    """The compressor's gated pool: ``out[b, d] = sum_r softmax_r(gate[b, :, d]) * kv[b, r, d]``.

    ``kv`` and ``gate``: fp32 CUDA tensors [B, R, D] with a contiguous last dimension (strided
    views otherwise allowed).  ``out``: [B, D] fp32 or bf16 with a contiguous last dimension, made
    here when not given (of ``out_dtype``).
    """
    lib = load_library()
    for name, t in (("kv", kv), ("gate", gate)):
        if t.dtype != torch.float32 or t.dim() != 3 or (t.shape[2] > 1 and t.stride(2) != 1):
            raise ValueError(f"{name} must be an fp32 [B, R, D] tensor with unit last stride")
    if kv.shape != gate.shape:
        raise ValueError("kv and gate must have the same shape")
    B, R, D = (int(x) for x in kv.shape)
    if out is None:
        out = torch.empty((B, D), dtype=out_dtype, device=kv.device)
    if out.dtype not in (torch.float32, torch.bfloat16) or tuple(out.shape) != (B, D) or \
            (D > 1 and out.stride(1) != 1):
        raise ValueError("out must be an fp32 or bf16 [B, D] tensor with unit last stride")
    dt = 1 if out.dtype == torch.bfloat16 else 0
    st = lib.sparse_attn_gated_pool(kv.data_ptr(), gate.data_ptr(), B, R, D, kv.stride(0),
                                    kv.stride(1), gate.stride(0), gate.stride(1), out.data_ptr(),
                                    dt, out.stride(0), _stream(stream))
    if st != 0:
        raise SpaError(st, "sparse_attn_gated_pool")
    return out


def sparse_attn_indexer_logits(q, weights, key_pool, block_table, positions, *, ratio,
                               num_cols=None, cand=None, seq_of_token=None, num_seqs=None,
                               out=None, stream=None):
    """Indexer logits over packed fp4_e8m0_b32 key rows (int32 [num_blocks, page_size, 17]):
    ``logits[t, c] = sum_h weights[t, h] * relu(q[t, h] . k[j])`` with j = c (Full mode) or
    ``cand[t, c]``; -inf where the entry does not exist.  Returns fp32 [T, num_cols]."""
    lib = load_library()
    if q.dtype != torch.bfloat16 or q.dim() != 3 or not q.is_contiguous():
        raise ValueError("q must be a contiguous bf16 [T, heads, 128] tensor")
    if weights.dtype != torch.float32 or tuple(weights.shape) != tuple(q.shape[:2]) or \
            not weights.is_contiguous():
        raise ValueError("weights must be a contiguous fp32 [T, heads] tensor")
    if key_pool.dtype != torch.int32 or key_pool.dim() != 3 or key_pool.shape[2] != 17 or \
            not key_pool.is_contiguous():
        raise ValueError("key_pool must be a contiguous int32 [num_blocks, page_size, 17] tensor")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or \
            not block_table.is_contiguous():
        raise ValueError("block_table must be a contiguous int32 [num_seqs, stride] tensor")
    for name, t in (("positions", positions), ("seq_of_token", seq_of_token), ("cand", cand)):
        if t is not None and (t.dtype != torch.int32 or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous int32 tensor")
    T, H = int(q.shape[0]), int(q.shape[1])
    if cand is not None:
        num_cols = int(cand.shape[1])
    if num_cols is None:
        raise ValueError("Full mode needs num_cols")
    if out is None:
        out = torch.empty((T, num_cols), dtype=torch.float32, device=q.device)
    B = int(block_table.shape[0]) if num_seqs is None else int(num_seqs)
    pool = SpaPoolC(key_pool.data_ptr(), None, None, block_table.data_ptr(), key_pool.shape[0],
                    key_pool.shape[1], block_table.shape[1])
    st = lib.sparse_attn_indexer_logits(q.data_ptr(), weights.data_ptr(), T, H,
                                        ctypes.byref(pool), positions.data_ptr(),
                                        _ptr(seq_of_token), B, int(ratio), _ptr(cand),
                                        int(num_cols), out.data_ptr(), _stream(stream))
    if st != 0:
        raise SpaError(st, "sparse_attn_indexer_logits")
    return out


def sparse_attn_indexer_topk(logits, k, *, cand=None, out=None, stream=None):
    """The k entries with the largest finite logits per row (fp32 [T, N]), in decreasing order of
    logit, ties to the smaller entry, -1 fill; column c is entry c or ``cand[t, c]``.  Returns
    int32 [T, k], usable as the attention's top-k list."""
    lib = load_library()
    if logits.dtype != torch.float32 or logits.dim() != 2 or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous fp32 [T, N] tensor")
    if cand is not None and (cand.dtype != torch.int32 or cand.shape != logits.shape or
                             not cand.is_contiguous()):
        raise ValueError("cand must be a contiguous int32 tensor shaped like logits")
    T, N = int(logits.shape[0]), int(logits.shape[1])
    if out is None:
        out = torch.empty((T, int(k)), dtype=torch.int32, device=logits.device)
    st = lib.sparse_attn_indexer_topk(logits.data_ptr(), T, N, _ptr(cand), int(k),
                                      out.data_ptr(), _stream(stream))
    if st != 0:
        raise SpaError(st, "sparse_attn_indexer_topk")
    return out


def sparse_attn_paged_resolve_columns(win, cmp, topk_idx, positions, *, window, ratio,
                                      seq_of_token=None, num_seqs=None, head_dim=64,
                                      stream=None) -> torch.Tensor:
    """Integer column list [T, W + K]: window rows, (1 << 30) | compressed rows, -1 if absent."""
    lib = load_library()
    T = int(positions.shape[0])
    K = 0 if topk_idx is None else int(topk_idx.shape[1])
    cols = torch.full((T, window + K), -1, dtype=torch.int32, device=positions.device)
    dummy_q = torch.empty((T, 1, head_dim), dtype=torch.bfloat16, device="meta")
    prob = _problem_c(dummy_q, win, topk_idx, positions, seq_of_token, window, ratio, 1.0,
                      num_seqs)
    w = _pool_c(win, win.kv.dtype == torch.uint8)
    c = _pool_c(cmp, cmp.kv.dtype == torch.uint8) if cmp is not None else None
    st = lib.sparse_attn_paged_resolve_columns(ctypes.byref(w), ctypes.byref(c) if c is not None
                                               else None, ctypes.byref(prob), cols.data_ptr(),
                                               _stream(stream))
    if st != 0:
        raise SpaError(st, "sparse_attn_paged_resolve_columns")
    return cols


def sparse_attn_paged_check_errors(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word."""
    lib = load_library()
    st = lib.sparse_attn_paged_check_errors(_stream(stream))
    if st == SPA_STATUS["SPA_ERR_CUDA"]:
        raise SpaError(st, "sparse_attn_paged_check_errors")
    return st


def sparse_attn_paged_strerror(status: int) -> str:
    return load_library().sparse_attn_paged_strerror(status).decode()
