"""5D TCGEN scale-factor layout (oracle; test infrastructure only).

The block_scaled_quantization module page (function list,
block_scales_interleave) names a 5D TCGEN layout that rank-2 scales are
rearranged into, without giving it.  Reading: the block-scale layout the tcgen05 block-scaled MMA
consumes, tiles of 128 rows x 4 scale columns (512 bytes) stored tile-row
major, shape (Mt, Kt, 32, 4, 4) with Mt = ceil(rows/128), Kt = ceil(S/4);
inside a tile, row r and column c sit at (r%32)*16 + (r/32)*4 + c.
"""
from __future__ import annotations

import numpy as np

TILE_ROWS = 128
TILE_COLS = 4
TILE_BYTES = 512


def _tiles(rows: int, S: int) -> tuple[int, int]:
    return -(-rows // TILE_ROWS), -(-S // TILE_COLS)


def scales5d_bytes(rows: int, S: int) -> int:
    """Bytes of the 5D buffer for ``rows`` x ``S`` scales (tiles fully padded)."""
    Mt, Kt = _tiles(rows, S)
    return Mt * Kt * TILE_BYTES


def offset_5d(m, s, Kt: int):
    """Byte offset of scale (row m, scale column s) in the 5D layout."""
    m = np.asarray(m, dtype=np.int64)
    s = np.asarray(s, dtype=np.int64)
    return (((m // 128) * Kt + s // 4) * 512 + (m % 32) * 16
            + ((m % 128) // 32) * 4 + (s % 4))


def scales_to_5d(scales2d: np.ndarray) -> np.ndarray:
    """Place an (M, S) uint8 scale matrix into a zero-filled 5D buffer."""
    scales2d = np.asarray(scales2d, dtype=np.uint8)
    M, S = scales2d.shape
    Mt, Kt = _tiles(M, S)
    out = np.zeros(Mt * Kt * TILE_BYTES, dtype=np.uint8)
    m, s = np.meshgrid(np.arange(M), np.arange(S), indexing="ij")
    out[offset_5d(m, s, Kt)] = scales2d
    return out


def scales_interleave(scales_bytes: np.ndarray, M: int, S: int, ld: int) -> np.ndarray:
    """Rank-2 -> 5D reinterleave: ``scales_bytes`` holds M rows of S scale
    bytes with a row stride of ``ld`` bytes; the output is the zero-padded 5D
    buffer."""
    flat = np.asarray(scales_bytes, dtype=np.uint8).reshape(-1)
    rows = np.stack([flat[m * ld: m * ld + S] for m in range(M)]) if M else \
        np.zeros((0, S), dtype=np.uint8)
    return scales_to_5d(rows)


def scales_from_5d_view(buf: np.ndarray, rows: int, S: int) -> np.ndarray:
    """Read a 5D buffer back as a (Mt*128, Kt*4) matrix by viewing it as
    (Mt, Kt, r32, r4, c) and permuting to (Mt, r4, r32, Kt, c): a statement of
    the layout independent of ``offset_5d``, used by the checks."""
    Mt, Kt = _tiles(rows, S)
    v = np.asarray(buf, dtype=np.uint8)[: Mt * Kt * TILE_BYTES].reshape(Mt, Kt, 32, 4, 4)
    return v.transpose(0, 3, 2, 1, 4).reshape(Mt * TILE_ROWS, Kt * TILE_COLS)
