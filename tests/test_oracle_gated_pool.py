"""Pins of the gated-pool oracle (oracle/gated_pool.py) against closed forms and invariants.

The pooled value is a per-channel softmax over R rows of the gates, weighting the kv rows.  Each
pin below is a case whose answer follows from the mathematics alone, chosen so that a plausible
slip in the oracle (the softmax taken over D instead of R, no maximum subtracted, the gate and
value operands swapped, a missing normalisation) fails at least one of them;
``test_pins_catch_*`` plant those slips and check that.
"""
import numpy as np
import pytest
import torch

from oracle import gated_pool as ogp


def _rand(B, R, D, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    kv = rng.standard_normal((B, R, D)).astype(np.float32)
    sc = (rng.standard_normal((B, R, D)) * scale).astype(np.float32)
    return kv, sc


def test_single_row_returns_the_row():
    kv, sc = _rand(3, 1, 100, 0)
    assert np.array_equal(ogp.gated_pool(kv, sc), kv[:, 0].astype(np.float64))


def test_equal_gates_give_the_mean():
    kv, _ = _rand(2, 7, 64, 1)
    sc = np.full_like(kv, 0.37)
    np.testing.assert_allclose(ogp.gated_pool(kv, sc), kv.astype(np.float64).mean(axis=1),
                               rtol=0, atol=1e-14)


def test_one_dominant_gate_selects_its_row():
    kv, sc = _rand(2, 9, 300, 2)
    win = np.array([4, 0])
    for b in range(2):
        sc[b, win[b], :] = 1000.0       # exp(-1000 - x) underflows to 0 in float64 for the rest
    got = ogp.gated_pool(kv, sc)
    assert np.array_equal(got, kv[np.arange(2), win].astype(np.float64))


def test_two_rows_take_the_logistic_weight():
    rng = np.random.default_rng(3)
    kv = rng.standard_normal((1, 2, 64))
    sc = rng.standard_normal((1, 2, 64)) * 3
    w0 = 1.0 / (1.0 + np.exp(sc[0, 1] - sc[0, 0]))
    want = w0 * kv[0, 0] + (1 - w0) * kv[0, 1]
    np.testing.assert_allclose(ogp.gated_pool(kv, sc)[0], want, rtol=1e-13, atol=1e-15)


def test_large_gates_do_not_overflow():
    kv, sc = _rand(1, 16, 64, 4)
    got = ogp.gated_pool(kv, sc.astype(np.float64) + 5000.0)
    np.testing.assert_allclose(got, ogp.gated_pool(kv, sc), rtol=1e-12, atol=1e-14)


def test_per_channel_shift_and_row_permutation_leave_the_result():
    kv, sc = _rand(2, 13, 100, 5, scale=4.0)
    ref = ogp.gated_pool(kv, sc)
    shift = np.random.default_rng(6).standard_normal((2, 1, 100)) * 50
    np.testing.assert_allclose(ogp.gated_pool(kv, sc + shift), ref, rtol=1e-11, atol=1e-13)
    perm = np.random.default_rng(7).permutation(13)
    np.testing.assert_allclose(ogp.gated_pool(kv[:, perm], sc[:, perm]), ref, rtol=1e-13,
                               atol=1e-15)


def test_result_is_a_convex_combination():
    kv, sc = _rand(4, 129, 64, 8, scale=6.0)
    got = ogp.gated_pool(kv, sc)
    assert (got <= kv.max(axis=1) + 1e-12).all() and (got >= kv.min(axis=1) - 1e-12).all()


def test_zero_rows_give_zero():
    assert not ogp.gated_pool(np.zeros((2, 0, 8)), np.zeros((2, 0, 8))).any()


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(20000) * np.exp2(rng.integers(-30, 30, 20000)),
                        [0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 3.3895e38]])
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(ogp.round_to_bf16_bits(x), want.view(np.uint16))


def _planted(monkeypatch, fn):
    monkeypatch.setattr(ogp, "gated_pool", fn)


def _pins_fail():
    for pin in (test_single_row_returns_the_row, test_equal_gates_give_the_mean,
                test_one_dominant_gate_selects_its_row, test_two_rows_take_the_logistic_weight,
                test_large_gates_do_not_overflow):
        try:
            with np.errstate(all="ignore"):
                pin()
        except AssertionError:
            return True
    return False


def test_pins_catch_softmax_over_channels(monkeypatch):
    def wrong(kv, sc):
        kv, sc = np.asarray(kv, np.float64), np.asarray(sc, np.float64)
        e = np.exp(sc - sc.max(axis=2, keepdims=True))
        return (e / e.sum(axis=2, keepdims=True) * kv).sum(axis=1)
    _planted(monkeypatch, wrong)
    assert _pins_fail()


def test_pins_catch_a_missing_maximum(monkeypatch):
    def wrong(kv, sc):
        kv, sc = np.asarray(kv, np.float64), np.asarray(sc, np.float64)
        e = np.exp(sc)
        return (e * kv).sum(axis=1) / e.sum(axis=1)
    _planted(monkeypatch, wrong)
    assert _pins_fail()


def test_pins_catch_swapped_operands(monkeypatch):
    real = ogp.gated_pool
    _planted(monkeypatch, lambda kv, sc: real(sc, kv))
    assert _pins_fail()


def test_pins_catch_a_missing_normalisation(monkeypatch):
    def wrong(kv, sc):
        kv, sc = np.asarray(kv, np.float64), np.asarray(sc, np.float64)
        return (np.exp(sc - sc.max(axis=1, keepdims=True)) * kv).sum(axis=1)
    _planted(monkeypatch, wrong)
    assert _pins_fail()


@pytest.mark.parametrize("R", [1, 3, 129])
def test_matches_a_dense_textbook_softmax(R):
    """A second, vectorised statement of the same definition, through torch's softmax."""
    kv, sc = _rand(3, R, 100, 10 + R, scale=3.0)
    w = torch.softmax(torch.from_numpy(sc.astype(np.float64)), dim=1)
    want = (w * torch.from_numpy(kv.astype(np.float64))).sum(dim=1).numpy()
    np.testing.assert_allclose(ogp.gated_pool(kv, sc), want, rtol=1e-12, atol=1e-14)
