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
  Each plane is stored in tiles of 64 rows x 128 elements (4096 bytes): the
  matrix is padded with zero codes to a multiple of 64 rows and 128 columns,
  tile (rt, kt) (row block rt, column block kt, KT = ceil(cols / 128) blocks
  per row) starts at byte (rt * KT + kt) * 4096, and row r of the tile takes
  bytes r * 64 .. r * 64 + 63 of it. A tile row holds its 128 elements in
  groups of 8: group q in the little-endian 32-bit word at bytes 4q .. 4q+3,
  whose nibble slot s (bits 4s .. 4s+3) holds element 8q + 2s for s < 4 and
  element 8q + 2(s - 4) + 1 for s >= 4 (even elements in the low half-word,
  odd ones in the high half-word, so a shift and a mask put elements 2j and
  2j+1 into the two 16-bit lanes of a word). Planes are stored back to back:
  plane 0, 1, 2, each plane_bytes(rows, cols) long.
"""
import numpy as np

# element (within a group of 8) held by nibble slot s = 0 .. 7 of a plane word
SLOT_ELEMENT = np.array([0, 2, 4, 6, 1, 3, 5, 7])


class NotRepresentable(ValueError):
    pass


TILE_ROWS, TILE_COLS, TILE_BYTES = 64, 128, 4096


def plane_bytes(rows, cols):
    """Bytes of one plane: whole 64 x 128 tiles."""
    return -(-rows // TILE_ROWS) * -(-cols // TILE_COLS) * TILE_BYTES


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
    return code_planes(code, rows, cols), base


def code_planes(code, rows, cols):
    """The three tiled planes of a [rows, cols] array of 12-bit codes."""
    rt, kt = -(-rows // TILE_ROWS), -(-cols // TILE_COLS)
    padded = np.zeros((rt * TILE_ROWS, kt * TILE_COLS), dtype=np.int64)
    padded[:rows, :cols] = code
    # nibble slot t of a row holds element (t // 8) * 8 + SLOT_ELEMENT[t % 8]
    slot_elem = (np.arange(kt * TILE_COLS) // 8) * 8 + SLOT_ELEMENT[np.arange(kt * TILE_COLS) % 8]
    planes = np.zeros((3, plane_bytes(rows, cols)), dtype=np.uint8)
    for p in range(3):
        slots = ((padded >> (4 * p)) & 0xF)[:, slot_elem]
        rowbytes = slots[:, 0::2] | (slots[:, 1::2] << 4)                # [rows_pad, cols_pad / 2]
        tiles = rowbytes.reshape(rt, TILE_ROWS, kt, TILE_COLS // 2).transpose(0, 2, 1, 3)
        planes[p] = tiles.reshape(-1).astype(np.uint8)
    return planes


def unpack(planes, base, rows, cols):
    """Inverse of pack: uint16 bf16 patterns [rows, cols]."""
    code = plane_codes(planes, rows, cols)
    s = code >> 11
    e = ((code >> 7) & 0xF) + base
    m = code & 0x7F
    return ((s << 15) | (e << 7) | m).astype(np.uint16)


def plane_codes(planes, rows, cols):
    """Inverse of code_planes: the 12-bit codes [rows, cols]."""
    planes = np.asarray(planes, dtype=np.uint8)
    rt, kt = -(-rows // TILE_ROWS), -(-cols // TILE_COLS)
    slot_elem = (np.arange(kt * TILE_COLS) // 8) * 8 + SLOT_ELEMENT[np.arange(kt * TILE_COLS) % 8]
    code = np.zeros((rt * TILE_ROWS, kt * TILE_COLS), dtype=np.int64)    # element order
    for p in range(3):
        tiles = planes[p].astype(np.int64).reshape(rt, kt, TILE_ROWS, TILE_COLS // 2)
        rowbytes = tiles.transpose(0, 2, 1, 3).reshape(rt * TILE_ROWS, kt * TILE_COLS // 2)
        slots = np.empty_like(code)
        slots[:, 0::2] = rowbytes & 0xF
        slots[:, 1::2] = rowbytes >> 4
        nib = np.empty_like(code)
        nib[:, slot_elem] = slots
        code |= nib << (4 * p)
    return code[:rows, :cols]


# ---------------------------------------------------------------- grouped W12
# The per-tensor window fails on real weights (zeros, or tails that span more
# than 16 binades). The grouped form keeps the planes above and adds, per block
# of 64 rows (a plane tile's rows), its own base, and a list of escapes:
#   base[rb] = max(1, (max E over the block's normal elements) - 15), or 1 for
#   a block without normal elements; an element escapes when it is not a
#   normal number or E < base[rb]; its code is 0 and the escape list holds
#   its exact pattern. Escapes are grouped by plane tile (rb, kt), tiles in
#   order rb * KT + kt, and within a tile in row-major order; entry =
#   row in block << 23 | column in tile << 16 | bf16 pattern, and tile i's
#   entries are esc[esc_off[i] .. esc_off[i + 1]].

def pack_grouped(bits):
    """Returns (planes, bases uint8 [row blocks], esc_off int32 [tiles + 1], esc uint32 [escapes])."""
    bits = np.asarray(bits, dtype=np.uint16)
    rows, cols = bits.shape
    s, e, m = fields(bits)
    normal = representable_mask(bits)
    rb_n, kt_n = -(-rows // TILE_ROWS), -(-cols // TILE_COLS)
    bases = np.ones(rb_n, dtype=np.int64)
    for rb in range(rb_n):
        blk_e, blk_n = e[rb * TILE_ROWS:(rb + 1) * TILE_ROWS], normal[rb * TILE_ROWS:(rb + 1) * TILE_ROWS]
        if blk_n.any():
            bases[rb] = max(1, int(blk_e[blk_n].max()) - 15)
    base_el = bases[np.arange(rows) // TILE_ROWS][:, None]
    esc = ~normal | (e < base_el)
    code = np.where(esc, 0, (s << 11) | ((e - base_el) << 7) | m)
    planes = code_planes(code, rows, cols)
    counts, entries = [], []
    for rb in range(rb_n):
        for kt in range(kt_n):
            r0, c0 = rb * TILE_ROWS, kt * TILE_COLS
            rr, cc = np.nonzero(esc[r0:r0 + TILE_ROWS, c0:c0 + TILE_COLS])   # row-major order
            counts.append(len(rr))
            entries += [(int(r) << 23) | (int(c) << 16) | int(bits[r0 + r, c0 + c]) for r, c in zip(rr, cc)]
    esc_off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return planes, bases.astype(np.uint8), esc_off, np.asarray(entries, dtype=np.uint32)


def unpack_grouped(planes, bases, esc_off, esc, rows, cols):
    """Inverse of pack_grouped."""
    code = plane_codes(planes, rows, cols)
    base_el = np.asarray(bases, dtype=np.int64)[np.arange(rows) // TILE_ROWS][:, None]
    out = ((code >> 11) << 15) | ((((code >> 7) & 0xF) + base_el) << 7) | (code & 0x7F)
    kt_n = -(-cols // TILE_COLS)
    for i in range(len(esc_off) - 1):
        rb, kt = divmod(i, kt_n)
        for ent in np.asarray(esc[esc_off[i]:esc_off[i + 1]], dtype=np.int64):
            out[rb * TILE_ROWS + ((ent >> 23) & 63), kt * TILE_COLS + ((ent >> 16) & 127)] = ent & 0xFFFF
    return out.astype(np.uint16)
