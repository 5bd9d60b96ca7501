"""Plant plausible mistakes in the oracle (on the CPU) and check that some pin catches each."""
import numpy as np
import pytest

import oracle.sparse_attention as O
import pins

_real_resolve = O.resolve_columns
_real_gather = O.gather_rows
_real_attend = O.attend
_real_e4m3 = O.e4m3_to_f64


def _window_off_by_one(*a, **k):
    cols, err = _real_resolve(*a, **k)
    W = k["window"]
    if W > 1:   # columns shifted one token into the past: the mistake p - W + c
        pos = np.asarray(a[0])
        shifted, _ = _real_resolve(pos - 1, *a[1:], **k)
        cols = cols.copy()
        cols[:, :W] = shifted[:, :W]
    return cols, err


def _causality_dropped_term(*a, **k):
    # r*j <= p instead of r*j + r - 1 <= p: pretend the query sits r - 1 positions later
    pos = np.asarray(a[0])
    cols, err = _real_resolve(*a, **k)
    late, _ = _real_resolve(pos + k["ratio"] - 1, *a[1:], **k)
    cols = cols.copy()
    W = k["window"]
    cols[:, W:] = late[:, W:]
    return cols, err


def _swapped_kv(*a, **k):
    kk, vv = _real_gather(*a, **k)
    return vv, kk


def _scale_dropped(q, k, v, scale):
    return _real_attend(q, k, v, 1.0)


def _softmax_sign(q, k, v, scale):
    return _real_attend(q, k, v, -scale)


def _e4m3_bias8(codes):
    return _real_e4m3(codes) * 0.5


def _transposed_operand(q, k, v, scale):
    # PV taken against the wrong operand: the K rows stand in for V
    return _real_attend(q, k, k, scale)


MUTANTS = [
    ("resolve_columns", _window_off_by_one),
    ("resolve_columns", _causality_dropped_term),
    ("gather_rows", _swapped_kv),
    ("attend", _scale_dropped),
    ("attend", _softmax_sign),
    ("attend", _transposed_operand),
    ("e4m3_to_f64", _e4m3_bias8),
]


@pytest.mark.parametrize("name,mutant", MUTANTS, ids=lambda x: getattr(x, "__name__", x))
def test_some_pin_catches(monkeypatch, name, mutant):
    monkeypatch.setattr(O, name, mutant)
    caught = []
    for pin in pins.ALL_PINS + [lambda: pins.pin_dense_bruteforce(fp8=True)]:
        try:
            pin()
        except AssertionError:
            caught.append(getattr(pin, "__name__", "fp8"))
    assert caught, f"no pin caught the planted mistake {mutant.__name__}"
