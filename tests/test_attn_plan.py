"""The attention plan mk_step_prepare makes for every step (query n-tiles,
head-dim blocks per warp, warp groups, staging slots, shared-memory exchange
areas), checked on the host through the library's host-only hook for every
head dim the layout accepts, both pool kinds and every query-row count:
the plan names a kernel variant that exists, the warps of a group cover the
head dim exactly once, the groups fit the block's math warps, the staging
slots and the page list fit the weight ring, the exchange areas fit the
phase region after Q and the new-rows slot, and every group has at least
two slots (one being filled while one is read)."""
import pytest

# (n-tiles, 32-dim blocks per warp) of the attention variants the kernel is
# compiled with (its dispatch on the plan)
VARIANTS = {(1, 4), (1, 2), (2, 2), (3, 2), (4, 1), (5, 1), (6, 1)}
MATH_WARPS = 8
MAX_SLOTS = 16
MAX_GROUPS = 8


@pytest.fixture(scope="module")
def mk():
    from speculative_decode_persistent_gb300 import mk
    return mk


@pytest.mark.parametrize("q8", [0, 1])
@pytest.mark.parametrize("dh", [64, 128, 192, 256])
def test_plan_invariants(mk, dh, q8):
    for q_rows in range(1, 49):
        rc, p = mk.attn_plan(q_rows, dh, q8)
        assert rc == 0, (q_rows, dh, q8, p)
        nq = (q_rows + 7) // 8
        assert p["nq"] == nq
        assert (p["nq"], p["jw"]) in VARIANTS, p
        assert p["wpg"] * p["jw"] * 32 == dh, p  # the group's warps cover the head dim once
        assert 1 <= p["ng"] <= MAX_GROUPS and p["ng"] * p["wpg"] <= MATH_WARPS, p
        assert p["spg"] >= 2 and p["nslots"] == p["spg"] * p["ng"] <= MAX_SLOTS, p
        # slots (first one aligned to 1024 bytes) and the page list inside the weight ring
        assert 1024 + p["nslots"] * p["slot_bytes"] + p["page_list_bytes"] <= p["ring_bytes"], p
        # Q (8 nq rows of dh + 8 halves) and the new-rows slot come before the exchange areas
        q_bytes = nq * 8 * (dh + 8) * 2
        row_bytes = dh if q8 else 2 * dh
        new_bytes = 2 * 16 * row_bytes + (2 * 16 * (dh // 32) * 2 if q8 else 0)
        assert p["xoff"] >= q_bytes + new_bytes, p
        assert p["xoff"] + p["ng"] * p["xslab"] + 16 <= p["phase_bytes"], p  # the flag word at the end


def test_headline_plans(mk):
    # 27B attention (24 query heads, 4 kv heads, dh 256): T = 1 and T = 5 on
    # fp16, 4 x T = 3 on q8
    for args, want in [((6, 256, 0), (1, 4, 2, 4, 2)), ((18, 256, 1), (3, 2, 4, 2, 7)),
                       ((30, 256, 0), (4, 1, 8, 1, 8))]:
        rc, p = mk.attn_plan(*args)
        assert rc == 0 and (p["nq"], p["jw"], p["wpg"], p["ng"], p["spg"]) == want, (args, p)


def test_plan_rejects_bad_arguments(mk):
    for args in [(0, 256, 0), (49, 256, 0), (8, 96, 0), (8, 320, 1), (8, 0, 0)]:
        assert mk.attn_plan(*args)[0] == -1, args  # MK_ERR_INVALID
