"""The C ABI: libfo.so loads on a machine without a GPU and exports every
function include/fo.h declares; argument errors come back synchronously."""
import ctypes
import os
import re

import pytest

from communication_overlap_gb300 import fo

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "fo.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fo_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("fo_plan_groups", "fo_signaled_gemm", "fo_consume_group",
                     "fo_reorder_back"):
        assert required in names


def test_library_exports_every_declared_symbol():
    L = ctypes.CDLL(fo.LIB_PATH)
    missing = [n for n in _declared() if not hasattr(L, n)]
    assert not missing, missing
    # the binding exposes the same names
    for n in _declared():
        assert hasattr(fo, n), n


def test_status_strings():
    assert fo.fo_status_string(fo.FO_OK) == "ok"
    assert "timed out" in fo.fo_status_string(fo.FO_ERR_TIMEOUT)


@pytest.mark.parametrize("bad", [
    dict(N=500),                       # N not a multiple of tile_n
    dict(K=100),                       # K not a multiple of 64
    dict(tile_n=64),                   # unsupported tile
    dict(swizzle=0),
    dict(group_waves=(1, 2)),          # does not sum to T = 4
    dict(group_waves=(0, 4)),          # empty group
    dict(layout=fo.FO_LAYOUT_RS_SUBTILE, n_dest=3),   # R does not divide 128
    dict(layout=fo.FO_LAYOUT_A2A_SUBTOKEN, n_dest=8,  # a routed row without a slot
         row_token=[0] * 256, row_slot=[-1] * 256),
    dict(layout=fo.FO_LAYOUT_A2A_SUBTOKEN, n_dest=2,  # (token 0, slot 0) twice: rank
         row_token=[0, 0] + [-1] * 254, row_slot=[0] * 256),  # 0 outgrows its buffer
    dict(wave_width=0),                # host-only plan needs an explicit W
    dict(M=0), dict(N=0), dict(K=0),   # empty operands
    dict(M=-128), dict(K=-64),
    dict(swizzle=-1), dict(wave_width=-3),
    dict(group_waves=(-1, 5)),         # a negative group
    dict(band_order=5),                # unknown band order
    dict(pad_expert_tile_rows=True),   # padding is an All-to-All option
    dict(tile_m=64),                   # unsupported tile height
])
def test_bad_descriptions_are_rejected(bad):
    args = dict(M=256, N=512, K=256, tile_n=128, swizzle=2, wave_width=2,
                group_waves=(1, 2, 1), host_only=True)
    args.update(bad)
    d = fo.make_desc(**args)
    with pytest.raises(fo.FoError) as e:
        fo.fo_plan_groups(d)
    assert e.value.status in (fo.FO_ERR_ARG, fo.FO_ERR_UNSUPPORTED)


def test_host_only_plan_refuses_launches():
    d = fo.make_desc(M=256, N=512, K=256, tile_n=128, swizzle=2, wave_width=2,
                     group_waves=(1, 2, 1), host_only=True)
    plan = fo.fo_plan_groups(d)
    try:
        with pytest.raises(fo.FoError) as e:
            fo.fo_signaled_gemm(plan, 16, [16], 16, 16, 16, 1, 0)
        assert e.value.status == fo.FO_ERR_ARG
        with pytest.raises(fo.FoError):
            fo.fo_reorder_back(plan, 0, 3, [16], [16], 0)
        with pytest.raises(fo.FoError):
            fo.fo_consume_group(plan, -1, fo.FO_CONS_COPY, 16, [], [16], 16, 1, 0, 16, 0)
        for comm in ([16], None):    # with communication buffers, and direct
            with pytest.raises(fo.FoError) as e:
                fo.fo_consume_reorder(plan, -1, fo.FO_CONS_COPY, 16, [], comm, [16], 0,
                                      fo.FO_ACT_NONE, 16, 1, 0, 16, 0)
            assert e.value.status == fo.FO_ERR_ARG
    finally:
        fo.fo_plan_destroy(plan)


def test_unit_place_table():
    """Every unit's final place, as k << 28 | 16-byte vector index; a plan
    whose output holds 2^28 vectors or more cannot name them."""
    d = fo.make_desc(M=256, N=512, K=256, tile_n=128, swizzle=2, wave_width=2,
                     group_waves=(1, 2, 1), host_only=True)
    plan = fo.fo_plan_groups(d)
    try:
        place = fo.fo_plan_table(plan, fo.FO_TAB_UNIT_PLACE)
        unit = fo.fo_plan_table(plan, fo.FO_TAB_UNIT)
        tile_of_slot = fo.fo_plan_table(plan, fo.FO_TAB_SLOT_TILE)
        assert sorted(place) == list(range(0, 256 * 512 // 8, 128 // 8))
        for s, t in enumerate(tile_of_slot):   # tile t = tm * 4 + tn (row-major)
            for r in range(128):
                row, col = 128 * (t // 4) + r, 128 * (t % 4)
                assert place[unit[128 * s + r]] == row * 512 // 8 + col // 8
    finally:
        fo.fo_plan_destroy(plan)
    big = dict(M=65536, N=32768, K=64, tile_n=256, swizzle=8, wave_width=148, host_only=True)
    _, T = fo.fo_wave_count(fo.make_desc(**big))
    plan = fo.fo_plan_groups(fo.make_desc(**big, group_waves=(T,)))
    try:
        with pytest.raises(fo.FoError) as e:
            fo.fo_plan_table(plan, fo.FO_TAB_UNIT_PLACE)
        assert e.value.status == fo.FO_ERR_UNSUPPORTED
    finally:
        fo.fo_plan_destroy(plan)


def test_a2a_plan_without_routing_starts_empty():
    """An All-to-All plan given no routing has every row empty: no units, no
    output rows; fo_plan_route fills it later (it needs a device plan)."""
    d = fo.make_desc(M=300, N=512, K=64, tile_n=256, swizzle=2, wave_width=3,
                     group_waves=(1, 1), layout=fo.FO_LAYOUT_A2A_SUBTOKEN, n_dest=4,
                     expert_rows=[200, 100], host_only=True)
    plan = fo.fo_plan_groups(d)
    try:
        assert fo.fo_plan_table(plan, fo.FO_TAB_DEST_UNITS) == [0] * 4
        assert fo.fo_plan_table(plan, fo.FO_TAB_FINAL_ROWS) == [0] * 4
        assert fo.fo_plan_table(plan, fo.FO_TAB_DEST_CAPACITY) == [0] * 4
        assert set(fo.fo_plan_table(plan, fo.FO_TAB_UNIT)) == {-1}
        assert fo.fo_plan_table(plan, fo.FO_TAB_UNIT_PLACE) == []
        with pytest.raises(fo.FoError) as e:   # host-only: nothing on a device to route
            fo.fo_plan_route(plan, 16, 16, 10, 2, 16, 0)
        assert e.value.status == fo.FO_ERR_ARG
    finally:
        fo.fo_plan_destroy(plan)


def test_consumer_placement_arguments():
    """fo_plan_set_consumer_placement: a null plan or an unknown placement is
    an argument error; a host-only plan (no device, so no SM is known to be
    free) cannot reserve SMs; the shared placement is always accepted."""
    assert fo.lib().fo_plan_set_consumer_placement(None, fo.FO_CONSUMER_SHARED) == fo.FO_ERR_ARG
    d = fo.make_desc(M=256, N=512, K=256, tile_n=128, swizzle=2, wave_width=2,
                     group_waves=(1, 2, 1), host_only=True)
    plan = fo.fo_plan_groups(d)
    try:
        with pytest.raises(fo.FoError) as e:
            fo.fo_plan_set_consumer_placement(plan, 7)
        assert e.value.status == fo.FO_ERR_ARG
        with pytest.raises(fo.FoError) as e:
            fo.fo_plan_set_consumer_placement(plan, fo.FO_CONSUMER_RESERVED)
        assert e.value.status == fo.FO_ERR_UNSUPPORTED
        fo.fo_plan_set_consumer_placement(plan, fo.FO_CONSUMER_SHARED)
    finally:
        fo.fo_plan_destroy(plan)


def test_smallest_plans():
    """One row (a ragged tile row of 1) and a single group covering every
    wave are valid plans."""
    for args, tiles, waves in ((dict(M=1, group_waves=(1, 1)), 4, 2),
                               (dict(M=256, group_waves=(4,)), 8, 4)):
        a = dict(M=256, N=512, K=256, tile_n=128, swizzle=2, wave_width=2, host_only=True)
        a.update(args)
        plan = fo.fo_plan_groups(fo.make_desc(**a))
        try:
            t, w, g, _ = fo.fo_plan_info(plan)
            assert (t, w) == (tiles, waves)
            assert sum(g) == tiles
        finally:
            fo.fo_plan_destroy(plan)
