"""The plan selector as pure host code, on a described GB300 (no GPU).

Mirrors the page's planner tests ("TIRx Metal reduction lowering" §6 and §8):
legality before cost, every selected plan covers the row exactly, ordered
requests always get the fixed tree, and the choice is deterministic."""
import math

import pytest

import fp32_row_reduction_gb300 as trlib
from fp32_row_reduction_gb300 import build as trbuild

DEV = trlib.gb300_device_desc()
SHAPES = [(37, 1537), (256, 3072), (64, 12289), (768, 6144), (4096, 50257), (16, 65536), (16, 262144),
          (16, 1048576), (65536, 128), (17, 257), (3, 4096), (7, 1024), (1, 1), (5, 3), (1000, 96)]


@pytest.fixture(scope="module", autouse=True)
def lib():
    trbuild.build()
    return trlib.load()


def select(op, rows, cols, order=0, align=1):
    return trlib.tr_plan_select_for(DEV, op, rows, cols, order, align)


def covers(p, cols):
    n4 = math.ceil(cols / 4)
    if p.kind == trlib.TR_PLAN_ROWS:
        w = p.lanes_per_row if p.lanes_per_row < 32 else 32 * p.warps_per_row
        return w * p.vec_slots >= n4
    if p.kind == trlib.TR_PLAN_CLUSTER:
        return p.block_threads * p.vec_slots >= math.ceil(n4 / p.cluster_ctas)
    if p.kind == trlib.TR_PLAN_ORDERED:
        return p.vec_slots == 0 or 1024 * p.vec_slots >= cols
    return True  # streaming plans cover any row


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("op", [0, 1, 2])
def test_unordered_plans_are_legal_and_cover(op, rows, cols):
    p = select(op, rows, cols)
    assert p.kind in (trlib.TR_PLAN_ROWS, trlib.TR_PLAN_CLUSTER, trlib.TR_PLAN_STREAM)
    assert covers(p, cols)
    assert p.block_threads % 32 == 0 and 32 <= p.block_threads <= 1024
    assert p.candidates >= 1 and p.est_us > 0 and p.ctas_per_sm >= 1
    if p.kind == trlib.TR_PLAN_ROWS:
        assert p.grid_ctas == math.ceil(rows / p.rows_per_cta)
    else:
        assert p.grid_ctas == rows * p.cluster_ctas


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_cross_entropy_uses_the_streaming_plan(rows, cols):
    p = select(3, rows, cols)
    assert p.kind == trlib.TR_PLAN_XENT
    assert p.vec_slots in (2, 4, 8)


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("op", [0, 1, 2, 3])
def test_ordered_requests_get_the_fixed_tree(op, rows, cols):
    p = select(op, rows, cols, order=1)
    assert p.kind == trlib.TR_PLAN_ORDERED
    assert p.block_threads == 256 and p.rows_per_cta == 1 and p.cluster_ctas == 1
    assert covers(p, cols)
    assert p.grid_ctas == rows


def test_selection_is_deterministic():
    for op in range(4):
        a = select(op, 768, 6144).as_dict()
        b = select(op, 768, 6144).as_dict()
        assert a == b


def test_768x6144_fits_one_wave():
    # the model must keep every row of the 768 x 6144 case resident at once
    for op in (0, 1, 2):
        p = select(op, 768, 6144)
        assert p.grid_ctas <= p.ctas_per_sm * DEV.sm_count, p.as_dict()


def test_long_rows_split_across_ctas():
    # 16 rows cannot fill 152 SMs one CTA per row: the rows must be split
    for cols in (262144, 1048576):
        p = select(0, 16, cols)
        assert p.cluster_ctas >= 2, p.as_dict()


def test_short_rows_pack_several_per_cta():
    p = select(0, 65536, 128)
    assert p.kind == trlib.TR_PLAN_ROWS and p.rows_per_cta >= 2


def test_packing_example_from_the_page():
    # "TIRx Metal reduction lowering" §4.1: P=17 rows of N=257 use one subgroup
    # per row with several rows packed in a group; here too a 257-wide row
    # never needs more than one warp.
    p = select(0, 17, 257)
    assert p.kind == trlib.TR_PLAN_ROWS
    assert p.lanes_per_row < 32 or p.warps_per_row == 1


def test_host_planner_rejects_malformed_device():
    bad = trlib.gb300_device_desc()
    bad.sm_count = 0
    with pytest.raises(trlib.TrError):
        trlib.tr_plan_select_for(bad, 0, 4, 8, 0, 1)
    with pytest.raises(trlib.TrError):
        trlib.tr_plan_select_for(DEV, 7, 4, 8, 0, 1)


def test_fewer_sms_never_gives_a_cheaper_estimate():
    small = trlib.gb300_device_desc()
    small.sm_count = 38
    for op in (0, 2):
        assert select(op, 768, 6144).est_us <= trlib.tr_plan_select_for(small, op, 768, 6144, 0, 1).est_us
