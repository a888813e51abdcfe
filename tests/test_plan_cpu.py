"""The automatic table-merging plan (mt_plan_merge, host code) against hand-worked groupings (no GPU)."""
import pytest

import update_merged_table_gb300 as mt
from update_merged_table_gb300 import build_lib


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_lib.build()
    mt.load_library()


def test_groups_by_row_shape_in_order_of_first_appearance():
    feats = [(16, "f32", 1000), (32, "f32", 500), (16, "bf16", 10), (64, "bf16", 100000), (32, "f32", 700),
             (16, "f32", 3000)]
    placement, groups = mt.plan_merge(feats, max_load=0.5)
    # worked by hand: (16, f32) takes features 0 and 5, (32, f32) features 1 and 4, then (16, bf16), (64, bf16)
    assert placement == [(0, 0), (1, 0), (2, 0), (3, 0), (1, 1), (0, 1)]
    assert [(g["dim"], g["row_dtype"], g["num_features"], g["capacity"]) for g in groups] == [
        (16, "f32", 2, 4000), (32, "f32", 2, 1200), (16, "bf16", 1, 10), (64, "bf16", 1, 100000)]
    # slots: the smallest 2^n with capacity <= 0.5 * 2^n: 8000 -> 2^13, 2400 -> 2^12, 20 -> 2^5, 200000 -> 2^18
    assert [g["log2_slots"] for g in groups] == [13, 12, 5, 18]


def test_load_factor_and_tiny_capacity():
    _, groups = mt.plan_merge([(8, "bf16", 0), (8, "bf16", 0)], max_load=1.0)
    assert len(groups) == 1 and groups[0]["log2_slots"] == 1  # at least two slots
    _, groups = mt.plan_merge([(4, "f32", 1024)], max_load=1.0)
    assert groups[0]["log2_slots"] == 10
    _, groups = mt.plan_merge([(4, "f32", 1025)], max_load=1.0)
    assert groups[0]["log2_slots"] == 11


def test_more_than_255_features_of_one_shape_open_a_second_table():
    placement, groups = mt.plan_merge([(16, "f32", 10)] * 256, max_load=0.5)
    assert [g["num_features"] for g in groups] == [255, 1]
    assert placement[254] == (0, 254) and placement[255] == (1, 0)  # table id 255 stays reserved


@pytest.mark.parametrize("feats, load", [
    ([(12, "bf16", 10)], 0.5),           # bf16 rows need dim % 8 == 0
    ([(6, "f32", 10)], 0.5),             # fp32 rows need dim % 4 == 0
    ([(16, "f32", -1)], 0.5),            # negative capacity
    ([(16, "f32", 10)], 0.0),            # load factor out of (0, 1]
    ([(16, "f32", 10)], 1.5),
    ([(16, "f32", 1 << 40)], 0.5),       # more than 2^31 slots
])
def test_invalid_plans_rejected(feats, load):
    with pytest.raises(mt.MTError):
        mt.plan_merge(feats, max_load=load)
