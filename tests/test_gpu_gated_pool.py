"""The compressor's gated pool on the GPU against the float64 oracle, element by element.

Shapes: the eight the pages time (FreeToken PR 633, "Kernel time": B in {1, 8}, R in {8, 128},
D in {128, 512}) and its edge cases ("Correctness and tests": R = 1/3/5/7/9/16/127/129,
D = 300/100/64, bf16 and fp32 outputs, strided views), plus R = 0.

Tolerance, from the kernel's arithmetic: every output is a ratio of two fp32 sums of at most R
terms, each term one `expf` (within 2 ulp) and one fused multiply-add, with one rescaling per
batch of eight rows and up to 16 warp states merged (three roundings each).  Relative to the
largest |kv| that enters the sum, that is at most (R + 64) roundings of 2^-24:
|gpu - oracle| <= (R + 64) * 2^-24 * max_r |kv[b, r, d]|.  A bf16 output adds its own rounding,
half an ulp: 2^-9 * |oracle| (taken as 2^-8 for the f64-to-f32-to-bf16 double rounding).
"""
import numpy as np
import pytest
import torch

import sparse_paged_attention_gb300 as spa
from oracle import gated_pool as ogp
from workloads import GATED_POOL_SHAPES, gated_pool_inputs

pytestmark = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _to_dev(buf, view, dev):
    d = buf.to(dev)
    return d.as_strided(view.size(), view.stride(), view.storage_offset())


def _check(B, R, D, out_dtype, view="dense", seed=0, gate_std=2.0):
    dev = _dev()
    kv_buf, kv, gate_buf, gate = gated_pool_inputs(B, R, D, seed=seed, gate_std=gate_std,
                                                   view=view)
    out = spa.sparse_attn_gated_pool(_to_dev(kv_buf, kv, dev), _to_dev(gate_buf, gate, dev),
                                     out_dtype=out_dtype)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    ref = ogp.gated_pool(kv.numpy(), gate.numpy())
    kmax = np.abs(kv.numpy()).max(axis=1) if R > 0 else np.zeros((B, D))
    tol = (R + 64) * 2.0 ** -24 * kmax
    if out_dtype == torch.bfloat16:
        tol = tol + 2.0 ** -8 * np.abs(ref)
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    bad = np.argwhere(err > tol)
    assert bad.size == 0, (len(bad), bad[:3], err.max())
    return got, ref


@pytest.mark.parametrize("shape", GATED_POOL_SHAPES, ids=lambda s: "B%dR%dD%d" % s)
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_timed_shapes(shape, out_dtype):
    _check(*shape, out_dtype)


@pytest.mark.parametrize("R", [1, 3, 5, 7, 9, 16, 127, 129])
@pytest.mark.parametrize("D", [300, 100, 64])
def test_edge_rows_and_dims(R, D):
    _check(3, R, D, torch.float32 if (R + D) % 2 else torch.bfloat16, seed=R * 1000 + D)


@pytest.mark.parametrize("view", ["row_pad", "every_other_row", "odd_offset"])
@pytest.mark.parametrize("D", [512, 100])
def test_strided_views(view, D):
    _check(4, 33, D, torch.float32, view=view, seed=7)


def test_single_row_is_copied_exactly():
    got, ref = _check(5, 1, 256, torch.float32, seed=11)
    assert np.array_equal(got, ref)


def test_sharp_and_flat_gates():
    _check(2, 128, 512, torch.float32, seed=12, gate_std=30.0)     # near one-hot weights
    _check(2, 128, 512, torch.float32, seed=13, gate_std=1e-3)     # near the plain mean


def test_zero_rows_write_zeros():
    dev = _dev()
    kv = torch.empty((3, 0, 64), dtype=torch.float32, device=dev)
    out = torch.full((3, 64), 7.0, device=dev)
    spa.sparse_attn_gated_pool(kv, kv.clone(), out)
    assert not out.cpu().any()


def test_output_row_stride_leaves_the_gaps():
    dev = _dev()
    kv_buf, kv, gate_buf, gate = gated_pool_inputs(4, 16, 96, seed=14)
    big = torch.full((4, 128), -3.0, device=dev)
    spa.sparse_attn_gated_pool(kv.to(dev), gate.to(dev), big[:, :96])
    got = big.cpu().numpy()
    assert (got[:, 96:] == -3.0).all()
    ref = ogp.gated_pool(kv.numpy(), gate.numpy())
    assert np.abs(got[:, :96] - ref).max() <= 80 * 2.0 ** -24 * np.abs(kv.numpy()).max()


@pytest.mark.parametrize("B,R,D,view", [(160, 20, 512, "dense"), (200, 33, 128, "row_pad"),
                                        (156, 1, 256, "every_other_row")])
def test_wide_batches(B, R, D, view):
    """Enough CTAs for one per SM at 128 channels each: the 16-byte load path."""
    _check(B, R, D, torch.float32, view=view, seed=B + R)
