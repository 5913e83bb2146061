"""Pins of the oracle's E4M3 / E2M1 conversions against things other than
itself: hand-derived spec landmarks, brute-force nearest-value search over the
decoded code table, torch's own float8_e4m3fn cast, and hand-checkable ties."""
import os

import numpy as np
import pytest
import torch

from oracle import fpformats as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                c, v = line.split()
                rows.append((int(c, 16), float(v)))
    return rows


def test_e4m3_decode_landmarks():
    for code, val in _read_table("e4m3_landmarks.txt"):
        got = float(F.e4m3_decode(np.array([code]))[0])
        assert got == val and np.signbit(got) == np.signbit(val), (hex(code), got, val)


def test_e4m3_nan_codes():
    assert np.isnan(F.e4m3_decode(np.array([0x7F, 0xFF]))).all()


def test_e2m1_table():
    for code, val in _read_table("e2m1_table.txt"):
        got = float(F.e2m1_decode(np.array([code]))[0])
        assert got == val and np.signbit(got) == np.signbit(val), (hex(code), got, val)


def test_encode_decode_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F])
    assert (F.e4m3_encode(F.e4m3_decode(codes)) == codes).all()
    codes4 = np.arange(16)
    assert (F.e2m1_encode(F.e2m1_decode(codes4)) == codes4).all()


def _brute_nearest(x, table_codes, table_vals):
    """Nearest finite value by exhaustive search; ties to the even code;
    magnitudes above the maximum saturate."""
    x = np.asarray(x, dtype=np.float64)
    d = np.abs(x[:, None] - table_vals[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among tied candidates prefer the even code (mantissa LSB 0)
    even = (table_codes[None, :] & 1) == 0
    pick = np.where(cand & even, 1, 0) * 2 + np.where(cand, 1, 0)
    j = pick.argmax(axis=1)
    return table_vals[j]


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_rounding_matches_bruteforce_search(fmt):
    rng = np.random.default_rng(123)
    if fmt == "e4m3":
        codes = np.array([c for c in range(128) if c != 0x7F])   # non-negative finite
        vals = F.e4m3_decode(codes)
        rnd, vmax, lo_exp, hi_exp = F.e4m3_round, 448.0, -14, 10
    else:
        codes = np.arange(8)
        vals = F.e2m1_decode(codes)
        rnd, vmax, lo_exp, hi_exp = F.e2m1_round, 6.0, -4, 4
    # log-uniform magnitudes across and beyond the range, random signs
    mags = np.exp2(rng.uniform(lo_exp, hi_exp, 200_000)).astype(np.float32)
    xs = mags * rng.choice([-1.0, 1.0], mags.size).astype(np.float32)
    # all exact midpoints between adjacent values and their float32 neighbours
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(0))
    xs = np.concatenate([xs, mids, up, dn, -mids, vals.astype(np.float32)])
    want = np.copysign(_brute_nearest(np.minimum(np.abs(xs), vmax), codes, vals), xs)
    got = rnd(xs)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(xs[i]), float(got[i]), float(want[i])) for i in bad[:5]]


def test_e2m1_hand_ties():
    xs = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -5.0, 7.0, 1e9, 0.2499], np.float32)
    want = np.array([0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, -4.0, 6.0, 6.0, 0.0])
    assert (F.e2m1_round(xs) == want).all()


def test_e4m3_saturation_and_hand_ties():
    xs = np.array([448.0, 449.0, 464.0, 465.0, 1e30, -1e30, 1.0625, 1.1875, 2.0 ** -10,
                   3 * 2.0 ** -10], np.float32)
    # 1.0625 is halfway between 1 and 1.125 -> even (1.0); 1.1875 -> 1.25 (even)
    # 2^-10 is halfway between 0 and 2^-9 -> 0; 3*2^-10 between 2^-9 and 2^-8 -> 2^-8
    want = np.array([448, 448, 448, 448, 448, -448, 1.0, 1.25, 0.0, 2.0 ** -8])
    assert (F.e4m3_round(xs) == want).all()


def test_e4m3_matches_torch_cast_in_range():
    """torch's float8_e4m3fn cast rounds to nearest-even; it maps values past
    the range to NaN instead of saturating, so compare inside the range."""
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(300_000).astype(np.float32) * np.float32(40.0),
        np.exp2(rng.uniform(-12, 8.8, 300_000)).astype(np.float32),
        rng.uniform(-448, 448, 100_000).astype(np.float32),
    ])
    x = x[np.abs(x) <= 448]
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    o = F.fp32_to_e4m3_code(x)
    # +-0 may differ in sign only
    same = (t == o) | (((t & 0x7F) == 0) & ((o & 0x7F) == 0))
    assert same.all(), np.nonzero(~same)[0][:5]


def test_pack_unpack_e2m1():
    codes = np.arange(32, dtype=np.uint8).reshape(2, 16) & 0xF
    p = F.pack_e2m1(codes)
    assert p.shape == (2, 8)
    assert p[0, 0] == (codes[0, 0] | (codes[0, 1] << 4))
    assert (F.unpack_e2m1(p) == codes).all()
