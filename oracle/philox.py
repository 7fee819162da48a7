"""Philox4x32-10 counter-based generator, written from its published definition.

TEST INFRASTRUCTURE: part of the CPU oracle.  Only tests/, the smoke check and
the benchmark's CPU-baseline leg may import it.

Definition (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
1, 2, 3", SC'11, section on the Philox family): a 4-word counter (c0..c3) and
a 2-word key (k0, k1), all 32-bit.  One round replaces the counter by
    (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0))
with multipliers M0 = 0xD2511F53, M1 = 0xCD9E8D57; between rounds the key is
bumped by the Weyl constants (0x9E3779B9, 0xBB67AE85).  Ten rounds.

The method's pages give no random-number layout; the draws here follow one
fixed layout keyed by (seed, request, position) so that a GPU implementation
written independently draws the same numbers:
    key     = (seed mod 2^32, seed >> 32)
    counter = (v >> 2, position, request, stream)    output word = v & 3
    u       = ((word >> 9) + 1/2) * 2^-23            exact in float32, in (0, 1)
    Gumbel  = -log(-log u)
Streams: 0 draft Gumbel, 1 accept uniform (v = 0), 2 residual Gumbel, 3 bonus Gumbel;
the block-level Gumbels of a draw in stream s use stream s + 4 (4 draft,
6 residual, 7 bonus; v = the block index; see oracle.dspark.gumbel_max).
Residual trial q (q = 0, 1, ...; see oracle.dspark.verify) uses stream 16 + 8q
for its proposal's id Gumbels, 16 + 8q + 4 for its block Gumbels, 16 + 8q + 5
for its super-block Gumbels (oracle.dspark.gumbel_max_trial) and 16 + 8q + 1
for its acceptance uniform (v = 0).
"""
from __future__ import annotations

import numpy as np

M0 = np.uint64(0xD2511F53)
M1 = np.uint64(0xCD9E8D57)
W0 = 0x9E3779B9
W1 = 0xBB67AE85
MASK = np.uint64(0xFFFFFFFF)

STREAM_DRAFT = 0
STREAM_ACCEPT = 1
STREAM_RESIDUAL = 2
STREAM_BONUS = 3
BLOCK_STREAM_OFFSET = 4   # block-level draws of stream s use stream s + 4
STREAM_TRIAL0 = 16        # residual trial q: streams 16 + 8q (+1 uniform, +4 blocks, +5 super-blocks)


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Return the four 32-bit output words (as uint64 arrays) for broadcastable counters."""
    x0, x1, x2, x3 = (np.asarray(c, dtype=np.uint64) & MASK for c in (c0, c1, c2, c3))
    x0, x1, x2, x3 = np.broadcast_arrays(x0, x1, x2, x3)
    key0, key1 = int(k0) & 0xFFFFFFFF, int(k1) & 0xFFFFFFFF
    for _ in range(10):
        p0 = M0 * x0                      # exact: both factors < 2^32
        p1 = M1 * x2
        hi0, lo0 = p0 >> np.uint64(32), p0 & MASK
        hi1, lo1 = p1 >> np.uint64(32), p1 & MASK
        x0, x1, x2, x3 = (hi1 ^ x1 ^ np.uint64(key0), lo1,
                          hi0 ^ x3 ^ np.uint64(key1), lo0)
        key0 = (key0 + W0) & 0xFFFFFFFF
        key1 = (key1 + W1) & 0xFFFFFFFF
    return x0, x1, x2, x3


def words(seed: int, position, request, stream: int, v) -> np.ndarray:
    """The 32-bit word drawn for vocabulary slot v (layout in the module docstring)."""
    v = np.asarray(v, dtype=np.uint64)
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    out = philox4x32_10(v >> np.uint64(2), position, request, stream,
                        seed & 0xFFFFFFFF, seed >> 32)
    lane = (v & np.uint64(3)).astype(np.int64)
    stacked = np.stack(out, axis=0)
    lane_b = np.broadcast_to(lane, stacked.shape[1:])
    return np.take_along_axis(stacked, lane_b[None], axis=0)[0]


def uniform(seed: int, position, request, stream: int, v) -> np.ndarray:
    """u = ((w >> 9) + 1/2) / 2^23 in (0, 1), returned in float64 (exact)."""
    w = words(seed, position, request, stream, v)
    return ((w >> np.uint64(9)).astype(np.float64) + 0.5) * (2.0 ** -23)


def gumbel(seed: int, position, request, stream: int, v) -> np.ndarray:
    u = uniform(seed, position, request, stream, v)
    return -np.log(-np.log(u))
