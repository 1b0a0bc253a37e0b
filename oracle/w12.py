"""W12 lossless weight codec (test infrastructure; see the package docstring).

SpecPilot digest, "Reasons": BF16 weights are split into three 4-bit
bit-planes and rebuilt bit-exactly inside the GEMM. The page fixes neither
the bit assignment nor the layout; this library's reading:

  bf16 pattern b: sign s = b >> 15, exponent E = (b >> 7) & 0xff, mantissa m = b & 0x7f.
  One base per tensor, base = min E. A tensor is representable iff every
  element is a normal number (1 <= E <= 254, so no +-0, subnormal, inf or
  NaN) and E - base <= 15 for every element (a 16-binade window).
  12-bit code c = s << 11 | (E - base) << 7 | m.
  plane p (p = 0, 1, 2) holds nibble p of c: (c >> 4p) & 15.
  Each plane is row-major [rows][ld] bytes, ld = ceil(cols / 32) * 16, with
  element k of a row in byte k // 2, low nibble for even k, high for odd k;
  padding nibbles are zero. Planes are stored back to back: plane 0, 1, 2.
"""
import numpy as np


class NotRepresentable(ValueError):
    pass


def row_bytes(cols):
    """Bytes per plane row: the row padded to a multiple of 32 elements."""
    return ((cols + 31) // 32) * 16


def fields(bits):
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    return b >> 15, (b >> 7) & 0xFF, b & 0x7F


def representable_mask(bits):
    """Per element: is it a normal bf16 number (the window is checked separately)."""
    _, e, _ = fields(bits)
    return (e >= 1) & (e <= 254)


def pack(bits):
    """Pack a 2-D uint16 array of bf16 patterns.

    Returns (planes uint8 [3, rows, ld], base). Raises NotRepresentable when
    the tensor is not representable; its argument counts the offending
    elements: those that are not normal numbers, plus the normal ones whose
    exponent exceeds (min exponent over normal elements) + 15.
    """
    bits = np.asarray(bits, dtype=np.uint16)
    if bits.ndim != 2:
        raise ValueError("pack expects a 2-D array")
    rows, cols = bits.shape
    s, e, m = fields(bits)
    normal = representable_mask(bits)
    base = int(e[normal].min()) if normal.any() else 1
    off = e - base
    # offending elements: the non-normal ones, plus the normal ones above the window
    bad = int((~normal).sum()) + int(((off > 15) & normal).sum())
    if bad:
        raise NotRepresentable(bad)
    code = (s << 11) | (off << 7) | m
    ld = row_bytes(cols)
    planes = np.zeros((3, rows, ld), dtype=np.uint8)
    for p in range(3):
        nib = np.zeros((rows, 2 * ld), dtype=np.int64)
        nib[:, :cols] = (code >> (4 * p)) & 0xF
        planes[p] = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    return planes, base


def unpack(planes, base, cols):
    """Inverse of pack: uint16 bf16 patterns [rows, cols]."""
    planes = np.asarray(planes, dtype=np.uint8)
    code = np.zeros(planes.shape[1:2] + (2 * planes.shape[2],), dtype=np.int64)
    for p in range(3):
        lo = planes[p].astype(np.int64) & 0xF
        hi = planes[p].astype(np.int64) >> 4
        nib = np.empty_like(code)
        nib[:, 0::2] = lo
        nib[:, 1::2] = hi
        code |= nib << (4 * p)
    code = code[:, :cols]
    s = code >> 11
    e = ((code >> 7) & 0xF) + base
    m = code & 0x7F
    return ((s << 15) | (e << 7) | m).astype(np.uint16)
