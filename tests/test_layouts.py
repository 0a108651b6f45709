"""The test-side statements of the tiled operand layouts (used by the GPU tests
to pack and unpack operands) cover every byte of a buffer exactly once when the
rows and K fill whole tiles, and agree with the library's size rule."""
import numpy as np
import pytest

from tests.nvf_testutil import ensure_built, row_tiles, tiled_index, weight_index


@pytest.mark.parametrize("groups,group_rows,K", [(1, 256, 256), (3, 384, 512), (2, 128, 768), (1, 640, 256)])
def test_weight_layout_is_a_bijection(groups, group_rows, K):
    rows = groups * group_rows
    code, sf = weight_index(rows, K, group_rows)
    nbytes = rows // 128 * ((K + 255) // 256) * 18432
    idx = np.concatenate([code.ravel(), sf.ravel()])
    assert idx.min() >= 0 and idx.max() < nbytes
    assert np.array_equal(np.sort(idx), np.arange(nbytes))


def test_weight_layout_pairs_tiles():
    """In a pair's unit both halves' codes come first, then both halves' atoms;
    an odd last tile has [codes][atoms] units."""
    K = 512
    code, sf = weight_index(384, K, 384)          # tiles 0, 1 paired; tile 2 alone
    unit = 2 * 18432
    assert code[0, 0] == 0 and code[128, 0] == 16384        # tile 1's codes follow tile 0's
    assert sf[0].min() == 32768 and sf[128].min() == 32768 + 2048
    assert code[0, 128] == unit                             # K tile 1 of the pair: next unit
    base2 = 2 * 2 * 18432                                   # after the pair's 2 K tiles
    assert code[256, 0] == base2 and sf[256].min() == base2 + 16384
    assert code[256, 128] == base2 + 18432


def test_grouped_layout_is_a_bijection():
    sizes = np.array([128, 256, 0, 384])
    offs = np.concatenate([[0], np.cumsum(sizes)])
    tiles = np.concatenate([[0], np.cumsum((sizes + 127) // 128)])
    K = 512
    code, sf = tiled_index(*row_tiles(int(offs[-1]), offs, tiles), K)
    nbytes = int(tiles[-1]) * 2 * 18432
    idx = np.concatenate([code.ravel(), sf.ravel()])
    assert np.array_equal(np.sort(idx), np.arange(nbytes))


def test_library_size_rule_matches():
    ensure_built()
    import nvfp4_moe_grouped_router_gb300 as nvf
    assert nvf.tiled_bytes(3 * 384, 0, 512) == 3 * 3 * 2 * 18432
