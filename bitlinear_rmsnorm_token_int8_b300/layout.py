"""Host-side index helpers for the packed weight layout (numpy only).

``bitlinear_pack_weights`` writes the 2-bit codes in the tile-major layout that
the contraction kernels stream (``include/bitlinear.h``): rows padded to a
multiple of 16 (Np) and grouped in tiles of 128 (the last tile holds the
remaining Np % 128 rows, if any), K in segments of 512 codes (128 bytes per
row); tiles one after another, and within a tile of R rows one contiguous block
of R x 128 bytes per segment, in which the 16-byte chunk c of row r sits at
chunk position c ^ (r % 8).  Rows past N and codes past K are zero.  The canonical form is the row-major [N, K/4] byte matrix of the
code table (weight k of row n in byte k/4, bits 2(k%4)..2(k%4)+1).

These functions only move bytes; they hold none of the method's arithmetic.
"""
from __future__ import annotations

import numpy as np

SEG_K = 512
ROW_PAD = 16
TILE_N = 128
ROW_BYTES = 128          # one row of one segment


def packed_bytes(N: int, K: int) -> int:
    """Size of the tiled layout for an N x K weight matrix."""
    return -(-N // ROW_PAD) * ROW_PAD * -(-K // SEG_K) * ROW_BYTES


def packed_index(N: int, K: int) -> np.ndarray:
    """int64 [N, K/4]: offset in the tiled layout of each canonical packed byte."""
    nseg = -(-K // SEG_K)
    Np = -(-N // ROW_PAD) * ROW_PAD
    n = np.arange(N, dtype=np.int64)[:, None]
    b = np.arange(K // 4, dtype=np.int64)[None, :]
    t = n // TILE_N
    rows = np.minimum(TILE_N, Np - t * TILE_N)           # rows of this tile
    return (t * TILE_N * nseg * ROW_BYTES + (b // 128) * rows * ROW_BYTES + (n % TILE_N) * ROW_BYTES
            + (((b % 128) // 16) ^ (n % 8)) * 16 + b % 16)


def canonical_from_tiled(tiled: np.ndarray, N: int, K: int) -> np.ndarray:
    """Tiled layout (flat uint8) -> canonical [N, K/4] uint8."""
    tiled = np.ascontiguousarray(tiled, dtype=np.uint8).reshape(-1)
    assert tiled.size >= packed_bytes(N, K)
    return tiled[packed_index(N, K)]


def tiled_from_canonical(canon: np.ndarray, K: int) -> np.ndarray:
    """Canonical [N, K/4] uint8 -> tiled layout (flat uint8, zero padding)."""
    canon = np.ascontiguousarray(canon, dtype=np.uint8)
    N = canon.shape[0]
    assert canon.shape[1] * 4 == K
    out = np.zeros(packed_bytes(N, K), dtype=np.uint8)
    out[packed_index(N, K)] = canon
    return out
