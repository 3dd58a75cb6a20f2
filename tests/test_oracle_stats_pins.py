"""Pins for the oracle's region statistics (CPU only).

Region statistics are the step after labelling on three of the pages: the
lpnh.cn CUDA segmentation page (§1.1: regions are labelled so that their area
and position can be measured), "GPU Connected Component Labeling"
(mcclanahoochie.com, closing section: statistics on every labelled region)
and bendabir.com (Prologue: each area's bounding box).  The oracle computes
area, inclusive bounding box, first pixel in reading order and the sums of
the row and column indices.  It is checked against:
* a small example worked by hand;
* scipy.ndimage (sum_labels, find_objects, minimum): library routines that
  compute the same quantities by other means;
* closed forms (constant image, row stripes, checkerboard);
* the batch layout (entries of image b follow those of images 0..b-1);
* planted mistakes in a copy of the oracle source, each caught by these pins.
"""
import ctypes
import subprocess

import numpy as np
import pytest

import oracle

scipy_ndimage = pytest.importorskip("scipy.ndimage")


def stats_by_scipy(lab, n):
    """The same statistics from scipy.ndimage, one image."""
    H, W = lab.shape
    idx = np.arange(1, n + 1)
    ones = np.ones_like(lab, dtype=np.float64)
    yy, xx = np.indices((H, W), dtype=np.float64)
    raster = yy * W + xx
    area = scipy_ndimage.sum_labels(ones, lab, idx)
    sum_y = scipy_ndimage.sum_labels(yy, lab, idx)
    sum_x = scipy_ndimage.sum_labels(xx, lab, idx)
    first = scipy_ndimage.minimum(raster, lab, idx)
    boxes = scipy_ndimage.find_objects(lab, max_label=n)
    out = np.zeros(n, dtype=oracle.STAT_DTYPE)
    out["area"] = np.asarray(area).astype(np.int64)
    out["sum_y"] = np.asarray(sum_y).astype(np.int64)
    out["sum_x"] = np.asarray(sum_x).astype(np.int64)
    out["first"] = np.asarray(first).astype(np.int64)
    for k, sl in enumerate(boxes):
        ys, xs = sl
        out["y_min"][k], out["y_max"][k] = ys.start, ys.stop - 1
        out["x_min"][k], out["x_max"][k] = xs.start, xs.stop - 1
    return out


def test_hand_worked_example():
    # 4-connectivity, binary:     1 1 0 2      labels  1 1 0 2
    #                             0 1 0 2              0 1 0 2
    #                             3 0 0 2              3 0 0 2
    # region 1 = (0,0) (0,1) (1,1): area 3, rows 0-1, cols 0-1, first 0,
    #   sum_y 0+0+1 = 1, sum_x 0+1+1 = 2
    # region 2 = (0,3) (1,3) (2,3): area 3, rows 0-2, col 3, first 3, sums 3 and 9
    # region 3 = (2,0): area 1, row 2, col 0, first 2*4+0 = 8, sums 2 and 0
    img = np.array([[1, 1, 0, 2], [0, 1, 0, 2], [3, 0, 0, 2]], np.uint8)
    lab, n = oracle.label(img, 4, oracle.MODE_BINARY)
    st = oracle.region_stats(lab, [n])
    expect = [(3, 0, 0, 1, 1, 0, 1, 2), (3, 0, 3, 2, 3, 3, 3, 9), (1, 2, 0, 2, 0, 8, 2, 0)]
    assert [tuple(int(v) for v in e) for e in st] == expect


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("conn", [4, 8])
def test_against_scipy(seed, conn):
    rng = np.random.default_rng(seed)
    H, W = int(rng.integers(1, 40)), int(rng.integers(1, 40))
    img = rng.integers(0, 3, size=(H, W)).astype(np.uint8)
    for mode in (oracle.MODE_ALL, oracle.MODE_BINARY):
        lab, n = oracle.label(img, conn, mode)
        st = oracle.region_stats(lab, [n])
        ref = stats_by_scipy(lab, int(n))
        assert st.dtype == ref.dtype
        for f in oracle.STAT_DTYPE.names:
            np.testing.assert_array_equal(st[f], ref[f], err_msg=f)


def test_constant_image_closed_form():
    H, W = 7, 11
    lab, n = oracle.label(np.full((H, W), 5, np.uint8), 8, oracle.MODE_ALL)
    (s,) = oracle.region_stats(lab, [n])
    assert (s["area"], s["y_min"], s["x_min"], s["y_max"], s["x_max"], s["first"]) == \
        (H * W, 0, 0, H - 1, W - 1, 0)
    assert s["sum_y"] == W * H * (H - 1) // 2
    assert s["sum_x"] == H * W * (W - 1) // 2


def test_row_stripes_closed_form():
    H, W = 6, 9
    img = (np.arange(H)[:, None] % 2 * np.ones((1, W), np.int64)).astype(np.uint8)
    lab, n = oracle.label(img, 4, oracle.MODE_ALL)
    assert n == H
    st = oracle.region_stats(lab, [n])
    for r in range(H):
        s = st[r]
        assert (s["area"], s["y_min"], s["y_max"], s["x_min"], s["x_max"]) == (W, r, r, 0, W - 1)
        assert s["first"] == r * W
        assert s["sum_y"] == r * W and s["sum_x"] == W * (W - 1) // 2


def test_checkerboard_8conn_closed_form():
    H, W = 5, 8
    r, c = np.indices((H, W))
    lab, n = oracle.label(((r + c) & 1).astype(np.uint8), 8, oracle.MODE_ALL)
    assert n == 2
    st = oracle.region_stats(lab, [n])
    # even cells (label 1, first pixel 0) and odd cells (label 2, first pixel 1)
    assert st["area"].tolist() == [H * W // 2, H * W // 2]
    assert st["first"].tolist() == [0, 1]
    assert st["y_min"].tolist() == [0, 0] and st["y_max"].tolist() == [H - 1, H - 1]
    assert st["x_min"].tolist() == [0, 0] and st["x_max"].tolist() == [W - 1, W - 1]
    # each row holds W/2 cells of each parity; even cells of row y sit at
    # columns of y's parity
    assert st["sum_y"].tolist() == [W // 2 * H * (H - 1) // 2] * 2
    even_x = sum(sum(range(y % 2, W, 2)) for y in range(H))
    assert st["sum_x"].tolist() == [even_x, H * W * (W - 1) // 2 - even_x]


def test_batch_layout_and_background():
    a = np.array([[1, 0, 1]], np.uint8)          # two regions
    b = np.array([[0, 0, 0]], np.uint8)          # none
    c = np.array([[1, 1, 1]], np.uint8)          # one
    imgs = np.stack([a, b, c])
    lab, n = oracle.label(imgs, 8, oracle.MODE_BINARY)
    assert n.tolist() == [2, 0, 1]
    st = oracle.region_stats(lab, n)
    assert len(st) == 3
    assert st["first"].tolist() == [0, 2, 0]      # image 2's region follows image 0's two
    assert st["area"].tolist() == [1, 1, 3]


def test_invalid_labels_rejected():
    lab = np.array([[1, 3]], np.int32)
    with pytest.raises(RuntimeError):
        oracle.region_stats(lab, [2])             # label 3 > n
    with pytest.raises(RuntimeError):
        oracle.region_stats(np.array([[-1]], np.int32), [1])


# ------------------------------------------------------ planted mistakes

MUTATIONS = {
    "x_for_y": ("if (y < s->y_min) s->y_min = (int32_t)y;", "if (y < s->y_min) s->y_min = (int32_t)x;"),
    "last_not_first": ("if (s->area == 0) s->first = (int32_t)(y * W + x);", "s->first = (int32_t)(y * W + x);"),
    "no_batch_offset": ("    base += n_regions[b];\n", "\n"),
    "open_box": ("if (x > s->x_max) s->x_max = (int32_t)x;", "if (x + 1 > s->x_max) s->x_max = (int32_t)(x + 1);"),
    "swapped_sums": ("        s->sum_x += x;", "        s->sum_x += y;"),
}


@pytest.mark.parametrize("key", sorted(MUTATIONS))
def test_pins_catch_planted_mistakes(tmp_path, key):
    src = open(oracle._SRC).read()
    old, new = MUTATIONS[key]
    assert old in src, key
    path = tmp_path / ("m_%s.c" % key)
    path.write_text(src.replace(old, new, 1))
    so = tmp_path / ("m_%s.so" % key)
    subprocess.check_call(["gcc", "-O1", "-std=c99", "-shared", "-fPIC", "-o", str(so), str(path)])
    lib = ctypes.CDLL(str(so))
    lib.oracle_region_stats.restype = ctypes.c_int
    lib.oracle_region_stats.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
    rng = np.random.default_rng(7)
    imgs = rng.integers(0, 3, size=(3, 9, 13)).astype(np.uint8)
    lab, n = oracle.label(imgs, 8, oracle.MODE_ALL)    # the oracle's labelling is pinned elsewhere
    lab = np.ascontiguousarray(lab)
    n = np.ascontiguousarray(n.astype(np.int32))
    total = int(n.sum())
    out = np.empty(total, dtype=oracle.STAT_DTYPE)
    lib.oracle_region_stats(lab.ctypes.data, 3, 9, 13, n.ctypes.data, out.ctypes.data, total)
    ref = np.concatenate([stats_by_scipy(lab[b], int(n[b])) for b in range(3)])
    assert any(not np.array_equal(out[f], ref[f]) for f in oracle.STAT_DTYPE.names), key
