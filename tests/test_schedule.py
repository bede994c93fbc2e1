"""The GEMM work split every block computes on its own (a closed form of
tiles, super-blocks, rows and grid), checked on the host through the
library's host-only hook: every unit of a phase belongs to exactly one math
warp, each block's reduction slice fits its shared-memory activation
region, and every split tile's completion ticket waits for exactly the warp
ranges that hold its units (a wrong count would leave a tile unsummed or
never finished)."""
import itertools

import numpy as np
import pytest

ACT_BYTES = 44 * 1024  # the kernel's activation region


@pytest.fixture(scope="module")
def mk():
    from speculative_decode_persistent_gb300 import mk
    return mk


# (n_tiles, nsb): the 27B phases (input GDN/FA, o_proj, gate/up, down,
# lm_head), the tiny model's, and ragged shapes
SHAPES = [(515, 20), (448, 20), (160, 24), (1088, 20), (160, 68), (7760, 20),
          (25, 1), (8, 1), (48, 1), (64, 3), (1, 1), (3, 7), (997, 13)]


@pytest.mark.parametrize("rows", [1, 2, 5, 9, 12])
@pytest.mark.parametrize("grid", [152, 148, 37])
def test_every_unit_once_and_tickets_match(mk, rows, grid):
    for n_tiles, nsb in SHAPES:
        info, arrivals = mk.gemm_schedule(n_tiles, nsb, rows, grid)
        nw = info.shape[1]
        owner = -np.ones((n_tiles, nsb), np.int64)
        segs = np.zeros(n_tiles, np.int64)
        for cta, w in itertools.product(range(grid), range(nw)):
            sb0, nsb_s, u0, u1 = (int(x) for x in info[cta, w])
            assert 1 <= nsb_s and sb0 + nsb_s <= nsb
            assert mk.lib.mk_debug_act_bytes(nsb_s, rows) <= ACT_BYTES
            tiles = set()
            for u in range(u0, u1):
                t, sbl = divmod(u, nsb_s)
                assert t < n_tiles
                assert owner[t, sb0 + sbl] == -1, (n_tiles, nsb, rows, grid, t, sb0 + sbl)
                owner[t, sb0 + sbl] = cta * nw + w
                tiles.add(t)
            for t in tiles:
                segs[t] += 1
        assert (owner >= 0).all(), (n_tiles, nsb, rows, grid)
        assert np.array_equal(segs, arrivals), (n_tiles, nsb, rows, grid)


def test_invalid_arguments(mk):
    from speculative_decode_persistent_gb300.mk import MkError
    with pytest.raises(MkError):
        mk.gemm_schedule(0, 1, 1, 152)
    with pytest.raises(MkError):
        mk.gemm_schedule(4, 1, 13, 152)
