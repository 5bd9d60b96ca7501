"""Pins of the KV-write oracle (oracle/kv_write.py) against what the format and the mathematics fix.

The e4m3 encoder is checked by brute force: for every probe value the expected code is the finite
code nearest to it (the decoder, itself pinned by tests/golden/e4m3_codes.json, gives every code's
value), ties going to the code with the even mantissa, magnitudes past 448 saturating.
"""
import numpy as np

import oracle
from oracle import kv_write as okw

FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
VALUES = oracle.e4m3_to_f64(FINITE)


def brute_force_code(x: float) -> int:
    if x != x:
        raise ValueError("no NaN probes")
    if abs(x) >= 448.0:
        return 0x7E | (0x80 if x < 0 else 0)
    neg = np.signbit(x)
    same_sign = FINITE[(FINITE >= 0x80) == neg]
    vals = oracle.e4m3_to_f64(same_sign)
    d = np.abs(vals - x)
    best = d.min()
    cands = same_sign[d == best]
    if len(cands) > 1:                          # a tie: the even mantissa wins
        cands = cands[(cands & 1) == 0]
    assert len(cands) == 1, (x, cands)
    return int(cands[0])


def probes():
    pos = np.sort(np.unique(np.abs(VALUES)))
    mids = (pos[:-1] + pos[1:]) / 2
    f32 = np.float32
    near = np.concatenate([np.nextafter(mids.astype(f32), f32(np.inf)),
                           np.nextafter(mids.astype(f32), f32(-np.inf))]).astype(np.float64)
    rng = np.random.default_rng(0)
    rand = rng.standard_normal(4000) * np.exp2(rng.integers(-12, 9, 4000))
    tiny = rng.uniform(0, 2.0 ** -6, 500)
    big = np.array([448.0, 447.9, 448.1, 463.9, 464.0, 464.1, 479.9, 480.0, 1e4])
    vals = np.concatenate([pos, mids, near, rand, tiny, big]).astype(np.float32).astype(np.float64)
    return np.concatenate([vals, -vals, [0.0, -0.0]])


def test_encoder_matches_brute_force_nearest():
    xs = probes()
    got = okw.e4m3_encode_rne(xs)
    want = np.array([brute_force_code(float(x)) for x in xs], dtype=np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(xs[i], hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_encoder_ties_go_to_even_mantissa():
    # 1.0625 lies half-way between 1.0 (0x38) and 1.125 (0x39): even 0x38 wins; 1.1875 half-way
    # between 1.125 (0x39) and 1.25 (0x3a): even 0x3a wins
    assert okw.e4m3_encode_rne([1.0625, 1.1875, -1.0625]).tolist() == [0x38, 0x3A, 0xB8]


def test_encoder_round_trips_every_finite_code():
    assert np.array_equal(okw.e4m3_encode_rne(VALUES), FINITE)


def test_encoder_zero_subnormal_and_saturation():
    got = okw.e4m3_encode_rne([0.0, -0.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10, 448.0, 470.0, -1e9])
    assert got.tolist() == [0x00, 0x80, 0x01, 0x00, 0x02, 0x7E, 0x7E, 0xFE]


def test_quantize_row_maps_the_largest_element_to_448():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(512).astype(np.float32)
    codes, s = okw.quantize_row_e4m3(x)
    i = int(np.argmax(np.abs(x)))
    assert codes[i] in (0x7E, 0xFE)
    assert s == np.float32(np.float32(np.abs(x).max()) / np.float32(448.0))
    # every stored value times the scale is within half a code step of the input
    back = oracle.e4m3_to_f64(codes) * float(s)
    assert np.all(np.abs(back - x) <= np.abs(x) * 2.0 ** -4 + float(s) * 2.0 ** -10)


def test_quantize_all_zero_row_has_scale_one():
    codes, s = okw.quantize_row_e4m3(np.zeros(64, dtype=np.float32))
    assert s == 1.0 and not codes.any()


def test_kv_write_places_rows_by_hand():
    # 3 physical pages of 2 slots, D = 4; sequence 0 owns pages [2, 0]
    bt = np.array([[2, 0]], dtype=np.int32)
    pool = np.full((3, 2, 2, 4), 0x7777, dtype=np.uint16)
    k = np.arange(5 * 4, dtype=np.uint16).reshape(5, 4)
    v = k + 100
    dropped = okw.kv_write(k, v, [0, 1, 2, 3, 4], None, bt, pool, page_size=2, fp8=False)
    assert dropped                                   # position 4: page 2 is past the table
    flat = pool.reshape(6, 2, 4)
    assert np.array_equal(flat[4, 0], k[0]) and np.array_equal(flat[4, 1], v[0])   # page 2, slot 0
    assert np.array_equal(flat[5, 0], k[1])                                        # page 2, slot 1
    assert np.array_equal(flat[0, 0], k[2]) and np.array_equal(flat[1, 1], v[3])   # page 0
    assert (flat[2:4] == 0x7777).all()                                             # page 1 unused


def test_kv_write_fp8_drops_bad_block_ids():
    bt = np.array([[0, 7]], dtype=np.int32)          # block 7 does not exist (3 blocks)
    pool = np.zeros((3, 2, 2, 64), dtype=np.uint8)
    ks = np.full(6, -1.0, dtype=np.float32)
    vs = ks.copy()
    rng = np.random.default_rng(2)
    bits = (rng.standard_normal((3, 64)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    dropped = okw.kv_write(bits, bits, [0, 2, 3], None, bt, pool, page_size=2, k_scale=ks,
                           v_scale=vs, fp8=True)
    assert dropped
    assert ks[0] > 0 and (ks[1:] == -1.0).all()     # only position 0 (block 0, slot 0) written


def test_pins_catch_rounding_half_away_from_zero(monkeypatch):
    """A plausible slip, rounding ties away from zero instead of to even, fails the pins."""
    rint = np.rint
    monkeypatch.setattr(np, "rint", lambda a: np.floor(np.asarray(a) + 0.5))
    xs = probes()
    got = okw.e4m3_encode_rne(xs)
    monkeypatch.setattr(np, "rint", rint)
    want = np.array([brute_force_code(float(x)) for x in xs], dtype=np.uint8)
    assert (got != want).any()


def test_pins_catch_a_wrong_subnormal_quantum(monkeypatch):
    """Clamping the exponent at -7 instead of -6 (a subnormal step of 2^-10) fails the pins."""
    clip = np.clip
    monkeypatch.setattr(np, "clip", lambda a, lo, hi: clip(a, -7 if lo == -6 else lo, hi))
    xs = probes()
    got = okw.e4m3_encode_rne(xs)
    monkeypatch.setattr(np, "clip", clip)
    want = np.array([brute_force_code(float(x)) for x in xs], dtype=np.uint8)
    assert (got != want).any()
