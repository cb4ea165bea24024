"""The tile-list checker the GPU tests apply to the library's tile list, checked here on CPU: it accepts the tile
lists that tile_list() builds and rejects each plausible mistake (a dropped row, an overlap, a tile across two
experts, an oversized tile, experts out of order, a wasted extra tile).  The library's maximum tile rows in the
binding equals the one in include/smoe.h."""
import os
import re

import numpy as np
import pytest

from helpers import check_tile_list, tile_list

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _case():
    counts = np.array([0, 5, 13, 0, 1, 8], np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return offsets


def test_checker_accepts_built_lists():
    offsets = _case()
    for R in (1, 2, 4, 8, 13, 64):
        tl = tile_list(offsets, R)
        check_tile_list(tl, offsets, R, max_tiles=10 ** 6)
        assert tl[:, 2].sum() == offsets[-1]
    check_tile_list(tile_list(np.zeros(5, np.int32), 4), np.zeros(5, np.int32), 4, 0)


@pytest.mark.parametrize("mistake", ["drop", "overlap", "cross", "oversize", "order", "extra", "count"])
def test_checker_rejects_mistakes(mistake):
    offsets = _case()
    R = 4
    tl = tile_list(offsets, R).copy()
    if mistake == "drop":        # a routed row in no tile
        tl[1, 2] -= 1
    elif mistake == "overlap":   # a row in two tiles
        tl[2, 1] -= 1
        tl[2, 2] += 1
    elif mistake == "cross":     # expert 1's last tile reaching into expert 2's first row
        last = int(np.nonzero(tl[:, 0] == 1)[0][-1])
        tl[last, 2] += 1
        tl[last + 1, 1] += 1
        tl[last + 1, 2] -= 1
    elif mistake == "oversize":  # more rows than the maximum
        tl = tile_list(offsets, 8)
    elif mistake == "order":     # experts out of order
        tl = np.concatenate([tl[-2:], tl[:-2]])
    elif mistake == "extra":     # an expert split into more tiles than it needs
        tl = tile_list(offsets, 2)
        R = 3
    elif mistake == "count":     # more tiles than the buffer holds
        with pytest.raises(AssertionError):
            check_tile_list(tl, offsets, R, max_tiles=len(tl) - 1)
        return
    with pytest.raises(AssertionError):
        check_tile_list(tl, offsets, R, max_tiles=10 ** 6)


def test_binding_tile_rows_match_header():
    text = open(os.path.join(ROOT, "include", "smoe.h")).read()
    from quantized_routed_expert_smoe_gb300 import binding
    assert int(re.search(r"#define SMOE_TILE_ROWS (\d+)", text).group(1)) == binding.TILE_ROWS
