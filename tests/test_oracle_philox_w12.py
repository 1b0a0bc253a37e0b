"""Pins for the oracle's Philox generator and W12 codec (CPU only)."""
import os

import numpy as np
import pytest

from oracle import philox, w12
from oracle.decoder import bf16_bits_to_f64

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _kat_rows():
    rows = []
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(x, 16) for x in line.split()])
    return rows


@pytest.mark.parametrize("row", _kat_rows())
def test_philox_known_answers(row):
    ctr, key, want = row[:4], row[4:6], row[6:]
    got = philox.philox4x32_10(np.array(ctr), np.array(key))
    assert [int(x) for x in got] == want


def test_philox_vectorised_matches_scalar():
    ctrs = np.random.default_rng(1).integers(0, 2**32, size=(50, 4), dtype=np.uint64)
    keys = np.random.default_rng(2).integers(0, 2**32, size=(50, 2), dtype=np.uint64)
    batch = philox.philox4x32_10(ctrs, keys)
    for i in range(50):
        assert (philox.philox4x32_10(ctrs[i], keys[i]) == batch[i]).all()


def test_uniform_keying_and_range():
    u = philox.uniform(20261202, 7, np.arange(100000), 0)
    assert u.min() >= 0.0 and u.max() < 1.0
    assert np.all(u.astype(np.float32).astype(np.float64) == u)      # exact in float32
    assert np.all((u * 2**24) == np.floor(u * 2**24))                # a multiple of 2^-24
    assert abs(u.mean() - 0.5) < 0.005
    # the keying is exactly counter (position, stream, req_lo, req_hi), key (seed_lo, seed_hi)
    seed, req, pos, stream = 0x0123456789ABCDEF, (5 << 32) | 9, 4100, 1
    word = philox.philox4x32_10(np.array([pos, stream, 9, 5]), np.array([0x89ABCDEF, 0x01234567]))[0]
    assert philox.uniform(seed, req, pos, stream) == (int(word) >> 8) / 2**24
    # streams, positions and requests give different draws
    a = philox.uniform(1, 2, np.arange(64), 0)
    assert not np.array_equal(a, philox.uniform(1, 2, np.arange(64), 1))
    assert not np.array_equal(a, philox.uniform(1, 3, np.arange(64), 0))
    assert not np.array_equal(a, philox.uniform(2, 2, np.arange(64), 0))


def _ieee_value(bits):
    """Value of bf16 patterns from the IEEE definition, without reinterpreting bits."""
    b = np.asarray(bits, dtype=np.int64)
    s, e, m = b >> 15, (b >> 7) & 0xFF, b & 0x7F
    return np.where(s == 1, -1.0, 1.0) * np.ldexp(1.0 + m / 128.0, e - 127)


def test_w12_exhaustive_single_elements():
    allbits = np.arange(65536, dtype=np.uint16)
    e = (allbits.astype(np.int64) >> 7) & 0xFF
    ok = 0
    for b in allbits:
        want_ok = 1 <= ((int(b) >> 7) & 0xFF) <= 254        # normal numbers only
        try:
            planes, base = w12.pack(np.array([[b]], dtype=np.uint16))
        except w12.NotRepresentable:
            assert not want_ok, hex(int(b))
            continue
        assert want_ok, hex(int(b))
        back = w12.unpack(planes, base, 1, 1)
        assert back[0, 0] == b
        ok += 1
    assert ok == int(((e >= 1) & (e <= 254)).sum())


def test_w12_window_rule_all_exponent_pairs():
    for e1 in range(1, 255, 3):
        for e2 in range(1, 255):
            t = np.array([[(e1 << 7) | 5, (1 << 15) | (e2 << 7) | 77]], dtype=np.uint16)
            fits = abs(e1 - e2) <= 15
            try:
                planes, base = w12.pack(t)
                assert fits
                assert base == min(e1, e2)
                assert (w12.unpack(planes, base, 1, 2) == t).all()
            except w12.NotRepresentable:
                assert not fits


def test_w12_layout_hand_example():
    # one row, three elements: codes chosen by hand
    #   b0 = +1.0      = 0x3f80: E 127, m 0
    #   b1 = -1.5      = 0xbfc0: E 127, m 64
    #   b2 = +2^-3*1.5 = 0x3e40: E 124, m 64 -> base 124
    t = np.array([[0x3F80, 0xBFC0, 0x3E40]], dtype=np.uint16)
    planes, base = w12.pack(t)
    assert base == 124
    # c = s<<11 | (E-base)<<7 | m:  c0 = 3<<7 = 0x180, c1 = 0x800|0x180|0x40 = 0x9c0, c2 = 0x040
    # group 0's word: slot 0 = element 0, slot 1 = element 2 (byte 0); slot 4 = element 1 (byte 2)
    assert planes.shape == (3, 4096)                       # one 64 x 128 tile per plane
    assert (planes[0] == 0).all()                                          # bits 0..3 are all 0
    assert planes[1, 0] == 0x48 and planes[1, 2] == 0x0C                  # bits 4..7: 8 | 4<<4; c1: C
    assert planes[2, 0] == 0x01 and planes[2, 2] == 0x09                  # bits 8..11: 1 | 0<<4; c1: 9
    assert planes[1, 1] == 0 and planes[2, 1] == 0 and planes[1, 3] == 0 and planes[2, 3] == 0
    assert (planes[:, 4:] == 0).all()
    assert (w12.unpack(planes, base, 1, 3) == t).all()


def test_w12_tile_placement_hand_example():
    # 65 x 131 matrix of +1.0 (code 0 with base 127) except element (64, 129) = -1.0
    # (code 0x800: nibble 8 in plane 2). It lies in tile (rt 1, kt 1) of a 2 x 2 grid,
    # tile row 0, group 0 (elements 128..135), element 1 of the group -> nibble slot 4,
    # i.e. the low nibble of byte 2 of the word: byte (1 * 2 + 1) * 4096 + 0 * 64 + 2.
    t = np.full((65, 131), 0x3F80, dtype=np.uint16)
    t[64, 129] = 0xBF80
    planes, base = w12.pack(t)
    assert base == 127 and planes.shape == (3, w12.plane_bytes(65, 131)) == (3, 4 * 4096)
    assert (planes[0] == 0).all() and (planes[1] == 0).all()
    nz = np.flatnonzero(planes[2])
    assert list(nz) == [3 * 4096 + 2] and planes[2, 3 * 4096 + 2] == 0x08
    assert (w12.unpack(planes, base, 65, 131) == t).all()


def test_w12_random_window_tensor_round_trip_and_values():
    import synth
    bits = synth.w12_window_bits(np.random.default_rng(3), (67, 688))
    planes, base = w12.pack(bits)
    assert planes.shape == (3, w12.plane_bytes(67, 688))
    back = w12.unpack(planes, base, 67, 688)
    assert (back == bits).all()
    assert np.array_equal(bf16_bits_to_f64(back), _ieee_value(bits))
