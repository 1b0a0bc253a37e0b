"""Pins for the oracle's grouped W12 form (per-64-row-block bases plus an escape list).

The per-tensor W12 window (SpecPilot digest, "Reasons": three 4-bit planes
rebuilt bit-exactly) cannot hold real weights with zeros or wide tails; the
grouped form extends it. Pinned by:
  * every one of the 65536 bf16 patterns round-trips exactly, zeros,
    subnormals, infinities and NaNs included (they are escapes);
  * the escape set and the bases equal their definition, recomputed
    element by element;
  * N(0, 0.02) bf16 weights round-trip exactly with escapes a tiny fraction;
  * on a 16-binade window tensor the grouped planes are byte-identical to
    the per-tensor planes and nothing escapes.
"""
import numpy as np

import synth
from oracle import w12


def _bf16_normal(shape, std, seed):
    import torch
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g) * std
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_every_pattern_round_trips():
    rng = np.random.default_rng(0)
    bits = rng.permutation(np.arange(65536, dtype=np.uint32)).astype(np.uint16).reshape(256, 256)
    planes, bases, off, esc = w12.pack_grouped(bits)
    assert np.array_equal(w12.unpack_grouped(planes, bases, off, esc, 256, 256), bits)


def test_bases_and_escapes_match_the_definition():
    rng = np.random.default_rng(1)
    # mixed blocks: wide tails, zeros, an all-zero block, ragged edges
    bits = _bf16_normal((150, 300), 0.02, 3)
    bits[rng.random(bits.shape) < 0.01] = 0
    bits[64:128] = 0
    bits[5, 7] = 0x7F80          # +inf
    bits[6, 8] = 0x0001          # subnormal
    planes, bases, off, esc = w12.pack_grouped(bits)
    e = (bits.astype(np.int64) >> 7) & 0xFF
    want_esc = set()
    for rb in range(3):
        blk = e[rb * 64:(rb + 1) * 64]
        normal = (blk >= 1) & (blk <= 254)
        base = max(1, int(blk[normal].max()) - 15) if normal.any() else 1
        assert bases[rb] == base
        for r, c in zip(*np.nonzero(~normal | (blk < base))):
            want_esc.add((rb * 64 + int(r), int(c)))
    got = set()
    for i in range(len(off) - 1):
        rb, kt = divmod(i, 3)
        for ent in esc[off[i]:off[i + 1]].astype(np.int64):
            r, c = rb * 64 + ((ent >> 23) & 63), kt * 128 + ((ent >> 16) & 127)
            assert ent & 0xFFFF == bits[r, c]
            got.add((int(r), int(c)))
    assert got == want_esc
    assert np.array_equal(w12.unpack_grouped(planes, bases, off, esc, *bits.shape), bits)


def test_normal_weights_round_trip_with_few_escapes():
    bits = _bf16_normal((512, 1024), 0.02, 7)
    planes, bases, off, esc = w12.pack_grouped(bits)
    assert np.array_equal(w12.unpack_grouped(planes, bases, off, esc, 512, 1024), bits)
    assert len(esc) < 1e-3 * bits.size
    try:
        w12.pack(bits)
        raise AssertionError("the per-tensor window should not hold N(0, 0.02) weights")
    except w12.NotRepresentable:
        pass


def test_window_tensor_matches_per_tensor_planes():
    gen = np.random.default_rng(9)
    bits = synth.w12_window_bits(gen, (128, 256))      # exponents 111 .. 126
    bits[0, 0] = (bits[0, 0] & 0x807F) | (111 << 7)
    bits[64, 0] = (bits[64, 0] & 0x807F) | (111 << 7)
    bits[0, 1] = (bits[0, 1] & 0x807F) | (126 << 7)
    bits[64, 1] = (bits[64, 1] & 0x807F) | (126 << 7)
    p1, base = w12.pack(bits)
    p2, bases, off, esc = w12.pack_grouped(bits)
    assert base == 111 and list(bases) == [111, 111] and len(esc) == 0
    assert np.array_equal(p1, p2)
