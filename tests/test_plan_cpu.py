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
    if p.kind == trlib.TR_PLAN_ORDERED_STAGED:
        return 1024 * p.vec_slots >= cols
    if p.kind == trlib.TR_PLAN_STAGED:
        ring = p.rows_per_cta * (4 * math.ceil(cols / 4) + 8) * 4
        return p.block_threads * p.vec_slots >= n4 and ring <= 225 * 1024
    if p.kind == trlib.TR_PLAN_WAVE:
        return cols % 4 == 0 and 1024 * p.vec_slots >= cols
    if p.kind == trlib.TR_PLAN_SEGMENTS:  # one segment of every row per CTA, one CTA per SM
        return cols % 4 == 0 and p.block_threads * p.vec_slots * p.grid_ctas >= n4
    return True  # streaming plans cover any row


def check_wave(p, rows, cols, op):
    """A wave plan: 256 threads (8 warps) per CTA on 1 or 2 aligned rows of >= 1024
    columns, vec_slots the smallest of 2/4/6/8 that covers the row, one CTA per rows_per_cta rows
    (two-row plans whose rows outnumber the resident CTAs, not twice over: every resident CTA)."""
    assert op in (0, 1, 2) and cols % 4 == 0 and cols >= 1024
    assert p.block_threads == 256 and p.warps_per_row == 8 and p.lanes_per_row == 32 and p.cluster_ctas == 1
    assert p.rows_per_cta in (1, 2) and p.flags == 0
    assert p.vec_slots == min(k for k in (2, 4, 6, 8) if 1024 * k >= cols)
    if p.rows_per_cta == 2 and p.resident_ctas < rows < 2 * p.resident_ctas:
        assert p.grid_ctas == p.resident_ctas   # every resident CTA, rows - res of them with two rows
    else:
        assert p.grid_ctas == math.ceil(rows / p.rows_per_cta)


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("op", [0, 1, 2])
def test_unordered_plans_are_legal_and_cover(op, rows, cols):
    p = select(op, rows, cols)
    assert p.kind in (trlib.TR_PLAN_ROWS, trlib.TR_PLAN_CLUSTER, trlib.TR_PLAN_STREAM, trlib.TR_PLAN_STAGED,
                      trlib.TR_PLAN_SPLIT, trlib.TR_PLAN_WAVE, trlib.TR_PLAN_SEGMENTS)
    assert covers(p, cols)
    assert p.block_threads % 32 == 0 and 32 <= p.block_threads <= 1024
    assert p.candidates >= 1 and p.est_us > 0 and p.ctas_per_sm >= 1
    if p.kind == trlib.TR_PLAN_ROWS:
        pair = 2 if p.flags & trlib.TR_PLAN_FLAG_TWO_ROWS else 1
        assert p.grid_ctas == math.ceil(rows / (p.rows_per_cta * pair))
    elif p.kind == trlib.TR_PLAN_STAGED:
        assert p.grid_ctas == min(rows, p.ctas_per_sm * DEV.sm_count)  # persistent CTAs
    elif p.kind == trlib.TR_PLAN_SPLIT:
        assert p.grid_ctas == rows * p.cluster_ctas <= p.ctas_per_sm * DEV.sm_count  # all resident
        assert 2 <= p.cluster_ctas <= 32 and p.vec_slots * p.block_threads * 16 <= 225 * 1024
    elif p.kind == trlib.TR_PLAN_WAVE:
        check_wave(p, rows, cols, op)
    elif p.kind == trlib.TR_PLAN_SEGMENTS:
        assert p.grid_ctas == DEV.sm_count and p.rows_per_cta == rows and p.block_threads == 1024
    else:
        assert p.grid_ctas == rows * p.cluster_ctas
    if p.flags == trlib.TR_PLAN_FLAG_PARAMS_IN_REGISTERS:
        assert p.kind == trlib.TR_PLAN_STAGED and op in (1, 2) and cols % 4 == 0
    else:
        if p.flags & trlib.TR_PLAN_FLAG_PARAMS_IN_SHARED:
            assert p.kind == trlib.TR_PLAN_ROWS and p.lanes_per_row == 32 and op in (1, 2) and cols % 4 == 0
        if p.flags & trlib.TR_PLAN_FLAG_TWO_ROWS:
            assert p.kind == trlib.TR_PLAN_ROWS and p.lanes_per_row == 32 and p.vec_slots in (2, 4, 6)
        assert p.flags & ~(trlib.TR_PLAN_FLAG_PARAMS_IN_SHARED | trlib.TR_PLAN_FLAG_TWO_ROWS) == 0


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_cross_entropy_uses_the_streaming_plan(rows, cols):
    p = select(3, rows, cols)
    assert p.kind == trlib.TR_PLAN_XENT
    assert p.vec_slots in (2, 4, 8)


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("op", [0, 1, 2, 3])
def test_ordered_requests_get_the_fixed_tree(op, rows, cols):
    p = select(op, rows, cols, order=1)
    assert p.kind in (trlib.TR_PLAN_ORDERED, trlib.TR_PLAN_ORDERED_STAGED, trlib.TR_PLAN_WAVE)
    assert p.block_threads == 256
    assert covers(p, cols)
    if p.kind == trlib.TR_PLAN_WAVE:
        check_wave(p, rows, cols, op)
    elif p.kind == trlib.TR_PLAN_ORDERED and p.cluster_ctas == 8:
        # few long rows: a cluster per row, one CTA per group of the tree
        assert p.vec_slots == 0 and cols > 16 * 1024 and rows < 2 * DEV.sm_count
        assert p.grid_ctas == 8 * rows and math.ceil(cols / 1024) * 512 <= 200 * 1024
    elif p.kind == trlib.TR_PLAN_ORDERED:
        assert p.cluster_ctas == 1 and p.rows_per_cta == 1 and p.grid_ctas == rows
    else:
        assert p.cluster_ctas == 1
        assert 1 <= p.rows_per_cta <= 8 and p.grid_ctas == min(rows, p.ctas_per_sm * DEV.sm_count)


def test_selection_is_deterministic():
    for op in range(4):
        a = select(op, 768, 6144).as_dict()
        b = select(op, 768, 6144).as_dict()
        assert a == b


def test_staged_plans_only_for_aligned_norms():
    # staged CTAs win only when their weights stay in registers across rows
    for rows, cols in SHAPES:
        assert select(0, rows, cols).kind != trlib.TR_PLAN_STAGED
        for op in (1, 2):
            p = select(op, rows, cols, align=0)
            assert p.kind != trlib.TR_PLAN_STAGED
            q = select(op, rows, cols, align=1)
            if q.kind == trlib.TR_PLAN_STAGED:
                assert q.flags == trlib.TR_PLAN_FLAG_PARAMS_IN_REGISTERS


def test_short_rows_never_split_or_stage():
    for rows, cols in [(65536, 128), (32768, 64), (4096, 256)]:
        for op in (0, 1, 2):
            p = select(op, rows, cols)
            assert p.kind == trlib.TR_PLAN_ROWS, p.as_dict()


def test_params_in_registers_only_when_aligned():
    staged = trlib.TR_PLAN_FLAG_PARAMS_IN_REGISTERS | trlib.TR_PLAN_FLAG_PARAMS_IN_SHARED
    for op in (1, 2):
        assert select(op, 768, 6144, align=0).flags & staged == 0


def test_long_rows_split_across_ctas():
    # 16 rows cannot fill 152 SMs one CTA per row: the rows must be split
    # (several CTAs per row, or every CTA holding a segment of every row)
    for op in (0, 1, 2):
        for cols in (262144, 1048576):
            p = select(op, 16, cols)
            assert p.cluster_ctas >= 2 or p.kind == trlib.TR_PLAN_SEGMENTS, p.as_dict()


def test_short_rows_pack_several_per_cta():
    p = select(0, 65536, 128)
    assert p.kind == trlib.TR_PLAN_ROWS and p.rows_per_cta >= 2


def test_packing_example_from_the_page():
    # "TIRx Metal reduction lowering" §4.1: P=17 rows of N=257. The page's Metal
    # planner packs one 32-lane group per row; on GB300 the fitted model may
    # spread the row over more lanes, but it stays a plain row plan whose
    # workers cover the row (no split across CTAs, no staging).
    p = select(0, 17, 257)
    assert p.kind == trlib.TR_PLAN_ROWS and p.cluster_ctas == 1
    assert covers(p, 257) and p.grid_ctas == math.ceil(17 / p.rows_per_cta)


def test_host_planner_rejects_malformed_device():
    bad = trlib.gb300_device_desc()
    bad.sm_count = 0
    with pytest.raises(trlib.TrError):
        trlib.tr_plan_select_for(bad, 0, 4, 8, 0, 1)
    with pytest.raises(trlib.TrError):
        trlib.tr_plan_select_for(DEV, 10, 4, 8, 0, 1)   # one past the last operator


def test_fewer_sms_never_gives_a_cheaper_estimate():
    small = trlib.gb300_device_desc()
    small.sm_count = 38
    for op in (0, 2):
        assert select(op, 768, 6144).est_us <= trlib.tr_plan_select_for(small, op, 768, 6144, 0, 1).est_us


def split_plan(rows, cols, C=4, T=512, K=2, op=0):
    return trlib.tr_plan(op=op, order=0, kind=trlib.TR_PLAN_SPLIT, lanes_per_row=32, warps_per_row=T // 32,
                         rows_per_cta=1, cluster_ctas=C, vec_slots=K, block_threads=T)


def test_split_plan_limits():
    # legal: co-resident grid, 2..32 CTAs per row, cache within the shared-memory budget
    for C, T, K, ok in [(2, 512, 2, True), (32, 256, 1, True), (33, 256, 1, False), (1, 256, 1, False),
                        (8, 1024, 14, True), (8, 1024, 15, False), (8, 512, 0, True)]:
        p = split_plan(4, 100000, C, T, K)
        st, why = trlib.check_plan_for(DEV, p, 4, 100000, 1)
        assert (st == trlib.TR_OK) == ok, (C, T, K, why)
    # the grid must fit the device at once: 200 rows x 2 CTAs of 1024 threads cannot
    st, why = trlib.check_plan_for(DEV, split_plan(200, 4096, 2, 1024, 1), 200, 4096, 1)
    assert st == trlib.TR_ERR_UNSUPPORTED and "resident" in why
    # the ordered policy is never split
    p = split_plan(4, 100000)
    p.order = 1
    st, _ = trlib.check_plan_for(DEV, p, 4, 100000, 1)
    assert st == trlib.TR_ERR_UNSUPPORTED


def seg_plan(op, rows, cols, K=None):
    sq = math.ceil(cols // 4 / DEV.sm_count)
    K = K if K is not None else math.ceil(sq / 1024)
    return trlib.tr_plan(op=op, order=0, kind=trlib.TR_PLAN_SEGMENTS, lanes_per_row=32, warps_per_row=32,
                         rows_per_cta=rows, cluster_ctas=1, vec_slots=K, block_threads=1024)


def test_segments_plan_limits_and_selection():
    # legal when forced: aligned rows, one 1024-thread CTA per SM holding a
    # segment of every row (rows <= 32, rows x SMs partials), 512..2048 quads per CTA
    for op, rows, cols, K, ok in [(0, 16, 1048576, 2, True), (1, 4, 1245184, 2, True), (2, 26, 400000, 1, True),
                                  (2, 27, 400000, 1, False),   # 27 x 152 partials > the workspace
                                  (0, 16, 1048576, 1, False),  # 1725 quads per CTA > 1 x 1024
                                  (0, 16, 262144, 1, False),   # 432 quads per CTA: too short
                                  (0, 4, 1253376, 2, False),   # 2062 quads per CTA > 2 x 1024
                                  (3, 16, 1048576, 2, False)]:  # cross-entropy is not served
        st, why = trlib.check_plan_for(DEV, seg_plan(op, rows, cols, K), rows, cols, 1)
        assert (st == trlib.TR_OK) == ok, (op, rows, cols, K, why)
    st, _ = trlib.check_plan_for(DEV, seg_plan(0, 16, 1048576), 16, 1048576, 0)  # unaligned
    assert st == trlib.TR_ERR_UNSUPPORTED
    p = seg_plan(0, 16, 1048576)
    p.rows_per_cta = 8                                 # a CTA holds every row
    assert trlib.check_plan_for(DEV, p, 16, 1048576, 1)[0] == trlib.TR_ERR_UNSUPPORTED
    # chosen for the norms' long rows (measured at 16 x 1048576: LayerNorm 33.4 us
    # against 40.0 for the best split plan; one row of 1048576: 9.5 against 18.1),
    # for softmax only with fewer rows than SMs / 32 (the split plans fill the
    # GPU from there and measured faster: 26.9 against 31.5 us at 16 x 1048576)
    for op in (1, 2):
        for rows, cols in [(16, 1048576), (1, 400000), (2, 1048576), (8, 1245184)]:
            assert select(op, rows, cols).kind == trlib.TR_PLAN_SEGMENTS, (op, rows, cols)
    assert select(0, 2, 1048576).kind == trlib.TR_PLAN_SEGMENTS
    for rows in (5, 8, 16, 24):
        assert select(0, rows, 1048576).kind != trlib.TR_PLAN_SEGMENTS
    # never for rows too short for it, an unaligned row, the ordered policy or cross-entropy
    for op in (0, 1, 2):
        for rows, cols in SHAPES:
            if cols < 4 * 512 * DEV.sm_count:
                assert select(op, rows, cols).kind != trlib.TR_PLAN_SEGMENTS
        assert select(op, 16, 1048576, align=0).kind != trlib.TR_PLAN_SEGMENTS
        assert select(op, 16, 1048576, order=1).kind != trlib.TR_PLAN_SEGMENTS
    assert select(3, 2, 1048576).kind != trlib.TR_PLAN_SEGMENTS


@pytest.mark.parametrize("op", [trlib.TR_OP_ROW_SUM, trlib.TR_OP_ROW_MAX, trlib.TR_OP_ROW_MIN, trlib.TR_OP_ROW_MINMAX])
def test_row_reductions_stream_once(op):
    # standalone reductions: the streaming kind unordered, the streaming OT-1024 ordered
    for rows, cols in SHAPES:
        p = select(op, rows, cols)
        assert p.kind == trlib.TR_PLAN_XENT
        q = select(op, rows, cols, order=1)
        assert q.kind == trlib.TR_PLAN_ORDERED and q.vec_slots == 0 and q.grid_ctas == rows


@pytest.mark.parametrize("order", [trlib.TR_ORDER_FOLD_LEFT, trlib.TR_ORDER_FOLD_RIGHT])
def test_fold_orders_get_the_warp_per_row_plan(order):
    for op in (0, 1, 2, 3, trlib.TR_OP_ROW_SUM, trlib.TR_OP_ROW_MINMAX):
        for rows, cols in [(768, 6144), (5, 3), (4096, 50257)]:
            p = select(op, rows, cols, order=order)
            assert p.kind == trlib.TR_PLAN_FOLD and p.block_threads == 64 and p.rows_per_cta == 2
            assert p.grid_ctas == math.ceil(rows / 2)
    with pytest.raises(trlib.TrError) as e:
        select(trlib.TR_OP_ADD_LAYERNORM, 4, 8, order=order)
    assert e.value.status == trlib.TR_ERR_UNSUPPORTED


def test_few_long_ordered_rows_spread_over_a_cluster():
    for op in (0, 1, 2, 3):
        p = select(op, 16, 262144, order=1)
        assert p.kind == trlib.TR_PLAN_ORDERED and p.cluster_ctas == 8 and p.grid_ctas == 128
        assert select(op, 16, 1048576, order=1).cluster_ctas == 1      # a group's share exceeds shared memory
        assert select(op, 4096, 50257, order=1).cluster_ctas == 1      # enough rows for a CTA each
    assert select(trlib.TR_OP_ROW_SUM, 16, 262144, order=1).cluster_ctas == 1
