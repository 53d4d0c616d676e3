"""Pins of the oracle's tiled scale-factor layout (reading R23: the layout of
the grouped NVFP4 tensor with GEMM-swizzled scales of TE PR #3753, commit
"... under NVFP4 autocast", taken as the 128-row x 4-column tiles that Blackwell block-scaled
matrix multiplies read).

The checks do not re-type the oracle's formula: positions worked out by hand
from the tile description (one 512-byte tile per 128 rows x 4 scale columns,
tiles along the scale columns contiguous; in a tile, 16-byte chunk i holds the
4 scale bytes of rows i, i+32, i+64, i+96 in that order), the permutation
property, the chunk structure itself, and the grouping of the per-expert
matrices.
"""
import numpy as np
import pytest

import oracle


def position_of(M, Kb, m, kb):
    lin = np.zeros((M, Kb), np.uint8)
    lin[m, kb] = 1
    out = oracle.scale_swizzle(lin)
    where = np.nonzero(out)[0]
    assert len(where) == 1
    return int(where[0])


# (M, Kb, m, kb, byte offset), each derived by hand:
HAND = [
    (256, 8, 0, 0, 0),          # first byte of the first tile
    (256, 8, 0, 3, 3),          # row 0's four bytes are contiguous
    (256, 8, 1, 0, 16),         # row 1 starts the second 16-byte chunk
    (256, 8, 32, 0, 4),         # row 32 shares row 0's chunk, second word
    (256, 8, 96, 2, 14),        # row 96: fourth word of chunk 0, byte 2
    (256, 8, 31, 3, 499),       # chunk 31 (496), word 0, byte 3
    (256, 8, 127, 3, 511),      # last byte of the first tile
    (256, 8, 0, 4, 512),        # scale column 4 opens the next tile along Kb
    (256, 8, 128, 0, 1024),     # row 128: tile (1, 0) = third tile (Kb/4 = 2 per row of tiles)
    (256, 8, 200, 5, 1673),     # tile (1, 1) = 1536; row 200: chunk 8 (128), word 2 (8), byte 1
    (128, 12, 65, 9, 1049),     # tile (0, 2) = 1024; row 65: chunk 1 (16), word 2 (8), byte 1
]


@pytest.mark.parametrize("M,Kb,m,kb,want", HAND)
def test_hand_worked_positions(M, Kb, m, kb, want):
    assert position_of(M, Kb, m, kb) == want


@pytest.mark.parametrize("M,Kb", [(128, 4), (256, 8), (384, 12), (128, 64)])
def test_is_a_permutation(M, Kb):
    idx = np.arange(M * Kb, dtype=np.int64).reshape(M, Kb)
    lo = oracle.scale_swizzle((idx & 0xFF).astype(np.uint8)).astype(np.int64)
    hi = oracle.scale_swizzle((idx >> 8).astype(np.uint8)).astype(np.int64)
    moved = hi * 256 + lo
    assert sorted(moved.tolist()) == list(range(M * Kb))


def test_chunk_structure_of_one_tile():
    rng = np.random.default_rng(3)
    lin = rng.integers(0, 256, (128, 4), dtype=np.uint8)
    out = oracle.scale_swizzle(lin)
    for i in range(32):
        chunk = out[16 * i:16 * i + 16]
        want = np.concatenate([lin[i], lin[i + 32], lin[i + 64], lin[i + 96]])
        assert np.array_equal(chunk, want), i


def test_rejects_partial_tiles():
    with pytest.raises(ValueError):
        oracle.scale_swizzle(np.zeros((100, 4), np.uint8))
    with pytest.raises(ValueError):
        oracle.scale_swizzle(np.zeros((128, 6), np.uint8))


def test_grouped_scales_follow_the_expert_slots():
    """Each expert's columnwise block [H, n_e/16] is tiled on its own, at its
    own byte offset; the rowwise [R, H/16] matrix is tiled once; bytes past R
    rows keep their values."""
    H, E = 256, 3
    offsets = np.array([0, 128, 128, 384], np.int32)   # expert 1 empty
    R_cap = 400
    rng = np.random.default_rng(5)
    dr = dict(rw_scales=rng.integers(0, 256, (R_cap, H // 16), dtype=np.uint8),
              cw_scales=rng.integers(0, 256, R_cap * H // 16, dtype=np.uint8))
    sw = oracle.swizzle_grouped_scales(dr, H, offsets, E)
    R = 384
    assert np.array_equal(sw["rw_scales"].reshape(-1)[: R * H // 16], oracle.scale_swizzle(dr["rw_scales"][:R]))
    assert np.array_equal(sw["rw_scales"][R:], dr["rw_scales"][R:])
    for e, (a, n) in enumerate([(0, 128), (128, 256)]):
        blk = dr["cw_scales"][a * H // 16:(a + n) * H // 16].reshape(H, n // 16)
        got = sw["cw_scales"][a * H // 16:(a + n) * H // 16]
        # row h of the expert's matrix, scale column kb, by the tile description
        for h, kb in [(0, 0), (5, 3), (200, 7), (255, n // 16 - 1)]:
            t = (h // 128) * (n // 64) + kb // 4
            pos = t * 512 + (h % 32) * 16 + ((h % 128) // 32) * 4 + kb % 4
            assert got[pos] == blk[h, kb], (e, h, kb)
    assert np.array_equal(sw["cw_scales"][R * H // 16:], dr["cw_scales"][R * H // 16:])
