"""Philox4x32-10 counter-based generator, written from [Random123].

Test infrastructure only (see the package docstring).

The generator: a 128-bit counter (c0, c1, c2, c3) and a 64-bit key (k0, k1)
go through 10 rounds.  One round multiplies c0 and c2 by two fixed odd
constants into 64-bit products, and produces
    (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0)).
Between rounds the key is bumped by the two Weyl constants (mod 2^32).

Uniform contract of this library (the pages specify no RNG):
    key     = (seed mod 2^32, seed >> 32)
    counter = (req_id, position, draw, trial)
    u       = (out0 >> 8) * 2^-24   in [0, 1), exact in fp32 and fp64
Draw ids: 0 draft sample at position k, 1 accept test at k, 2 residual at the
rejecting k, 3 bonus at l+1, 4 the acceptance test of a residual proposal;
trial numbers the proposals of the rejection-sampled residual (0 otherwise);
ids >= 16 are free for synthetic data.
"""
import numpy as np

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
MASK32 = 0xFFFFFFFF

DRAW_DRAFT = 0
DRAW_ACCEPT = 1
DRAW_RESIDUAL = 2
DRAW_BONUS = 3
DRAW_RESID_ACCEPT = 4


def philox4x32_10(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox4x32-10; all arguments broadcastable integer arrays < 2^32.

    Returns four uint64 arrays holding the 32-bit output words."""
    c0, c1, c2, c3, k0, k1 = np.broadcast_arrays(*[np.asarray(x, dtype=np.uint64) & np.uint64(MASK32)
                                                   for x in (c0, c1, c2, c3, k0, k1)])
    c0, c1, c2, c3, k0, k1 = (a.copy() for a in (c0, c1, c2, c3, k0, k1))
    m0 = np.uint64(PHILOX_M0)
    m1 = np.uint64(PHILOX_M1)
    w0 = np.uint64(PHILOX_W0)
    w1 = np.uint64(PHILOX_W1)
    mask = np.uint64(MASK32)
    s32 = np.uint64(32)
    for rnd in range(10):
        if rnd > 0:
            k0 = (k0 + w0) & mask
            k1 = (k1 + w1) & mask
        p0 = m0 * c0  # < 2^64: exact in uint64
        p1 = m1 * c2
        hi0, lo0 = p0 >> s32, p0 & mask
        hi1, lo1 = p1 >> s32, p1 & mask
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def uniform(seed: int, req_id, position, draw, trial=0):
    """u in [0,1) for (seed, request id, position, draw id, trial); fp64 array (exact 24-bit values)."""
    seed = int(seed)
    k0 = seed & MASK32
    k1 = (seed >> 32) & MASK32
    out0, _, _, _ = philox4x32_10(req_id, position, draw, trial, k0, k1)
    return (out0 >> np.uint64(8)).astype(np.float64) * (2.0 ** -24)
