"""Philox4x32-10 counter-based RNG, written from its published definition.

Test infrastructure (see the package docstring). Source: J. K. Salmon,
M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel random numbers: as easy as
1, 2, 3", SC'11, section 3.3 (the Philox S-box: two 32x32->64 multiplies per
round, a Weyl-sequence key schedule, ten rounds for Philox4x32-10).

The verify step draws its uniforms from this generator (the DSpark summary,
"Problem", says acceptance is by rejection sampling; the pages fix no RNG).
Keying, as this library defines it:
  key     = (seed & 0xffffffff, seed >> 32)
  counter = (position, stream, request_id & 0xffffffff, request_id >> 32)
  u       = (word0 >> 8) * 2**-24, exactly representable in float32, in [0, 1)
stream 0 drives the accept test of a draft, stream 1 the resample/bonus draw.
"""
import numpy as np

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)


def philox4x32_10(counter, key):
    """Apply ten Philox rounds.

    counter: uint32-compatible array [..., 4]; key: [..., 2]. Returns uint32 [..., 4].
    Each round multiplies words 0 and 2 by the two round constants, keeps the
    high and low halves, and mixes the high halves with words 1 and 3 and the
    round key; the key advances by the Weyl constants between rounds.
    """
    counter = np.asarray(counter, dtype=np.uint64)
    key = np.asarray(key, dtype=np.uint64)
    c0, c1, c2, c3 = (counter[..., i] & _MASK32 for i in range(4))
    k0, k1 = key[..., 0] & _MASK32, key[..., 1] & _MASK32
    for rnd in range(10):
        if rnd:
            k0 = (k0 + np.uint64(PHILOX_W0)) & _MASK32
            k1 = (k1 + np.uint64(PHILOX_W1)) & _MASK32
        prod0 = np.uint64(PHILOX_M0) * c0
        prod1 = np.uint64(PHILOX_M1) * c2
        hi0, lo0 = prod0 >> np.uint64(32), prod0 & _MASK32
        hi1, lo1 = prod1 >> np.uint64(32), prod1 & _MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def uniform(seed, request_id, position, stream):
    """u in [0,1) for (seed, request, absolute position, stream); broadcasts."""
    seed = np.uint64(seed)
    req = np.asarray(request_id, dtype=np.int64).astype(np.uint64)
    pos = np.asarray(position, dtype=np.int64).astype(np.uint64)
    stm = np.asarray(stream, dtype=np.int64).astype(np.uint64)
    req, pos, stm = np.broadcast_arrays(req, pos, stm)
    ctr = np.stack([pos & _MASK32, stm & _MASK32, req & _MASK32, req >> np.uint64(32)], axis=-1)
    key = np.broadcast_to(np.array([int(seed) & 0xFFFFFFFF, int(seed) >> 32], dtype=np.uint64),
                          ctr.shape[:-1] + (2,))
    word0 = philox4x32_10(ctr, key)[..., 0]
    return (word0 >> np.uint32(8)).astype(np.float64) * 2.0 ** -24
