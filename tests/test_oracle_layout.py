"""Pins for the oracle's shape:stride layout evaluator.

Every expected value below is printed on the pages (typed into tests/golden
with its page and section); none is produced by the evaluator itself.
"""
import itertools

import pytest

import oracle
from golden_io import lines, nested, tup


def test_sm80_tv_layouts_match_printed_lane_tables():
    layouts = {}
    checked = 0
    for f in lines("sm80_tv_layouts.txt"):
        if f[0] == "layout":
            layouts[f[1]] = (nested(f[2]), nested(f[3]), int(f[4]))
        elif f[0] == "lane":
            shape, stride, rows = layouts[f[1]]
            lane = int(f[2])
            for v, want in enumerate(f[3:]):
                q = oracle.layout_offset(shape, stride, (lane, v))
                assert (q % rows, q // rows) == tup(want), (f[1], lane, v)
                checked += 1
    assert checked == 4 * 4 + 8 + 4 + 4


def test_thread_layouts_and_warp_origins():
    for f in lines("tiled_mma_threads.txt"):
        if f[0] == "map":
            assert oracle.layout_offset(nested(f[1]), nested(f[2]), tup(f[3])) == int(f[4])


def _c_coord(lane, v, wm, wn):
    """C coordinate of (lane, value) in warp (wm, wn): CLayout plus the warp's
    block origin, read through the evaluator only."""
    q = oracle.layout_offset(((4, 8), (2, 2)), ((32, 1), (16, 8)), (lane, v))
    return (q % 16 + 16 * wm, q // 16 + 8 * wn)


def test_get_slice_warp_origins():
    n = 0
    for f in lines("tiled_mma_threads.txt"):
        if f[0] != "warp":
            continue
        t, wm, wn = int(f[1]), int(f[2]), int(f[3])
        # (lane, wm, wn, wk) recovered from t through the thread layout
        found = [c for c in itertools.product(range(32), range(2), range(2), range(1))
                 if oracle.layout_offset((32, 2, 2, 1), (1, 32, 64, 0), c) == t]
        assert found == [(0, wm, wn, 0)]
        got = [_c_coord(0, v, wm, wn) for v in range(4)]
        assert got == [tup(s) for s in f[4:8]]
        n += 1
    assert n == 4


def test_four_warp_multiplicity():
    """A/B/C coverage multiplicities of the 2x2x1 four-warp tiling (32x16x16)."""
    want = {f[1]: int(f[2]) for f in lines("tiled_mma_threads.txt") if f[0] == "multiplicity"}
    a_lay = (((4, 8), (2, 2, 2)), ((32, 1), (16, 8, 128)))
    b_lay = (((4, 8), (2, 2)), ((16, 1), (8, 64)))
    c_lay = (((4, 8), (2, 2)), ((32, 1), (16, 8)))
    cnt = {"A": {}, "B": {}, "C": {}}
    for t in range(128):
        lane, wm, wn = None, None, None
        for c in itertools.product(range(32), range(2), range(2)):
            if oracle.layout_offset((32, 2, 2, 1), (1, 32, 64, 0), c + (0,)) == t:
                lane, wm, wn = c
        for v in range(8):
            q = oracle.layout_offset(*a_lay, (lane, v))
            key = (q % 16 + 16 * wm, q // 16)
            cnt["A"][key] = cnt["A"].get(key, 0) + 1
        for v in range(4):
            q = oracle.layout_offset(*b_lay, (lane, v))
            key = (q % 8 + 8 * wn, q // 8)
            cnt["B"][key] = cnt["B"].get(key, 0) + 1
            q = oracle.layout_offset(*c_lay, (lane, v))
            key = (q % 16 + 16 * wm, q // 16 + 8 * wn)
            cnt["C"][key] = cnt["C"].get(key, 0) + 1
    assert len(cnt["A"]) == 32 * 16 and len(cnt["B"]) == 16 * 16 and len(cnt["C"]) == 32 * 16
    for op in "ABC":
        assert set(cnt[op].values()) == {want[op]}, op


def test_perm_m_table():
    it = lines("perm_m.txt")
    head = next(it)
    shape, stride = nested(head[1]), nested(head[2])
    seen = 0
    for f in it:
        assert oracle.layout_offset(shape, stride, int(f[0])) == int(f[1])
        seen += 1
    assert seen == 8
    # a bijection on 0..31 (stated in the same section)
    assert sorted(oracle.layout_offset(shape, stride, i) for i in range(32)) == list(range(32))


def test_partition_c_offsets_on_row_major_c():
    cur = None
    n = 0
    for f in lines("partition_c.txt"):
        if f[0] == "offsets":
            cur = (nested(f[1]), nested(f[2]), int(f[3]))
            continue
        shape, stride, ld = cur
        off = oracle.layout_offset(shape, stride, tup(f[0]))
        assert (off // ld, off % ld) == (int(f[1]), int(f[2]))
        n += 1
    assert n == 4 + 16


def test_simple_gemm_thread0_a_positions():
    it = lines("simple_gemm_tAgA.txt")
    head = next(it)
    shape, stride, ld = nested(head[1]), nested(head[2]), int(head[3])
    n = 0
    for f in it:
        ik, mm = int(f[0]), int(f[1])
        for v, want in enumerate(f[2:10]):
            off = oracle.layout_offset(shape, stride, (v, mm, 0, ik))
            assert (off // ld, off % ld) == tup(want)
            n += 1
    assert n == 128  # "thread 0 reads 8 x 4 x 1 x 4 = 128 A elements"


def test_ldmatrix_route_values_and_packing():
    packed = {}
    for f in lines("ldmatrix_route.txt"):
        if f[0] == "eval":
            assert oracle.layout_offset(nested(f[1]), nested(f[2]), tup(f[3])) == int(f[4])
        elif f[0] == "packed":
            packed[int(f[1])] = (int(f[2]), int(f[3]))
    # labels A(m,k) = 16 m + k in a (16,16):(16,1) tile, A(0,9) overwritten with 37
    label = {}
    for m in range(16):
        for k in range(16):
            label[oracle.layout_offset((16, 16), (16, 1), (m, k))] = 16 * m + k
    label[oracle.layout_offset((16, 16), (16, 1), (0, 9))] = 37
    a_lay = (((4, 8), (2, 2, 2)), ((32, 1), (16, 8, 128)))
    vals = []
    for v in range(8):
        q = oracle.layout_offset(*a_lay, (0, v))
        m, k = q % 16, q // 16
        vals.append(label[oracle.layout_offset((16, 16), (16, 1), (m, k))])
    for i in range(4):
        assert (vals[2 * i], vals[2 * i + 1]) == packed[i]


def test_size_one_mode_stride_is_irrelevant():
    # "a size-1 mode can only take coordinate 0, its stride does not matter"
    for s in (0, 4, 12345):
        assert oracle.layout_offset((2, 2, 1), (1, 2, s), (1, 1, 0)) == 3


def test_out_of_range_coordinate_is_rejected():
    with pytest.raises(ValueError):
        oracle.layout_offset((2, 2), (1, 2), (2, 0))
    with pytest.raises(ValueError):
        oracle.layout_offset((8, 4), (4, 1), 32)
