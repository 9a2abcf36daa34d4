"""Philox4x32-10, the counter-based generator of Salmon, Moraes, Dror and Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11), section 4.

A Philox round maps a 4-word counter (c0, c1, c2, c3) and a 2-word key (k0, k1)
to (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0)) with the
multipliers M0 = 0xD2511F53 and M1 = 0xCD9E8D57; between rounds the key is
bumped by the Weyl constants (0x9E3779B9, 0xBB67AE85).  Ten rounds are applied.
The published known-answer vectors are pinned in tests/golden/philox_kat.txt.
"""

import numpy as np

_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85
_MASK = np.uint64(0xFFFFFFFF)
_SH = np.uint64(32)


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox4x32-10.

    c0..c3: broadcastable uint32 arrays (the counter); k0, k1: python ints (the key).
    Returns four uint32 arrays of the broadcast shape.
    """
    c0, c1, c2, c3 = np.broadcast_arrays(
        np.asarray(c0, dtype=np.uint32), np.asarray(c1, dtype=np.uint32),
        np.asarray(c2, dtype=np.uint32), np.asarray(c3, dtype=np.uint32))
    x0 = c0.astype(np.uint64)
    x1 = c1.astype(np.uint64)
    x2 = c2.astype(np.uint64)
    x3 = c3.astype(np.uint64)
    key0 = int(k0) & 0xFFFFFFFF
    key1 = int(k1) & 0xFFFFFFFF
    for _ in range(10):
        p0 = _M0 * x0
        p1 = _M1 * x2
        hi0, lo0 = p0 >> _SH, p0 & _MASK
        hi1, lo1 = p1 >> _SH, p1 & _MASK
        x0, x1, x2, x3 = (hi1 ^ x1 ^ np.uint64(key0), lo1,
                          hi0 ^ x3 ^ np.uint64(key1), lo0)
        key0 = (key0 + _W0) & 0xFFFFFFFF
        key1 = (key1 + _W1) & 0xFFFFFFFF
    return (x0.astype(np.uint32), x1.astype(np.uint32),
            x2.astype(np.uint32), x3.astype(np.uint32))
