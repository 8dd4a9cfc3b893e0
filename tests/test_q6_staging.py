"""Host-side check of the production q6_K GEMM's raw-weight staging arithmetic.

The kernel (mmq_prod_q6K.cuh) views the 210-byte q6_K blocks of W as
[O/8][8*nsb*210] bytes: eight consecutive rows span 1680*nsb bytes, a
multiple of 16, so the blocks of super-block sb in rows 8g + i (phase i fixed,
g = 0..15 of a 128-row tile) are one 2-D TMA box of 16 x 224 bytes starting at
byte x = floor((i*nsb*210 + sb*210) / 16) * 16 of each group row; a tile that
holds an incomplete group of eight rows is copied row by row instead.  The
unpack thread of row o reads its block at offset lead = ((o*nsb + sb)*210) % 16
of the copied window.  These tests restate that arithmetic and check, for many
shapes, that every block lies inside its window at that offset, that no box
starts off a 16-byte boundary, and that the box path is never taken for a row
of an incomplete group.
"""
import pytest

BLOCK = 210
WINDOW = 224
BN = 128


def box_window(o0, rho, sb, nsb):
    """Global byte range [start, end) the box of tile row rho copies, and the
    end of the group row it reads (bytes past it arrive zero-filled)."""
    i, g = rho & 7, (o0 // 8) + (rho >> 3)
    group_bytes = 8 * nsb * BLOCK
    x = ((i * nsb + sb) * BLOCK) & ~15
    start = g * group_bytes + x
    return start, start + WINDOW, (g + 1) * group_bytes, x


def uses_boxes(O, o0):
    return O % 8 == 0 or o0 + BN <= 8 * (O // 8)


@pytest.mark.parametrize("O", [8, 16, 128, 136, 200, 256, 300, 4096, 11008])
@pytest.mark.parametrize("K", [256, 512, 768, 1280, 2048, 4096, 11008])
def test_blocks_inside_box_windows(O, K):
    nsb = K // 256
    for o0 in range(0, O, BN):
        boxes = uses_boxes(O, o0)
        for rho in range(BN):
            o = o0 + rho
            if o >= O:
                continue
            if boxes:
                # a row handled by a box belongs to a complete group of eight
                assert (o // 8) < O // 8
            for sb in range(nsb):
                block = (o * nsb + sb) * BLOCK
                lead = block % 16
                if boxes:
                    start, end, row_end, x = box_window(o0, rho, sb, nsb)
                    assert x % 16 == 0                      # TMA x coordinate on a 16-byte boundary
                    assert start + lead == block            # the kernel's lead finds the block
                    assert block + BLOCK <= end             # the whole block is in the window
                    assert block + BLOCK <= row_end         # and none of it is zero fill
                else:
                    a = block & ~15                         # the row's bulk-copy window
                    assert a + lead == block and block + BLOCK <= a + WINDOW


def test_box_rows_are_the_groups_rows():
    # phase i, group row g of a tile: rows 8g + i, each row exactly once per tile
    seen = set()
    for rho in range(BN):
        i, g = rho & 7, rho >> 3
        seen.add(8 * g + i)
    assert seen == set(range(BN))


@pytest.mark.parametrize("O", [1, 7, 9, 129, 300, 4097])
def test_incomplete_group_tile_takes_bulk_copies(O):
    # the tile that holds rows of an incomplete group of eight uses the per-row path
    last = ((O - 1) // BN) * BN
    if O % 8:
        assert not uses_boxes(O, last)
    for o0 in range(0, last, BN):
        assert uses_boxes(O, o0)
