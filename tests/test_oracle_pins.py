"""Pins for the oracle (CPU only).

The oracle is checked against things other than itself:
* the worked examples the pages print (tests/golden/, each with its citation);
* brute force: every binary 4x4 image and every 3-valued 3x3 image, under both
  connectivities and both modes, against a transitive-closure labelling that
  uses neither union-find nor flood fill;
* closed forms (checkerboard, serpentine, stripes, constant, all-distinct);
* scipy.ndimage.label, the library routine the binary case reduces to;
* mutation checks: plausible mistakes planted in a copy of the oracle source
  (a dropped diagonal, a row wrap-around, a byte left out of the compare,
  background not ignored, numbering that does not restart per image, seeds
  taken in reverse raster order) are caught by these pins.
"""
import itertools
import os
import subprocess

import numpy as np
import pytest

import oracle
from tests.helpers import (canonicalize, check_invariants, closure_labels,
                           read_golden, scipy_labels)

GOLDENS = sorted(f for f in os.listdir(os.path.join(os.path.dirname(__file__), "golden"))
                 if f.endswith(".txt"))


@pytest.mark.parametrize("name", [g for g in GOLDENS if g.startswith(("p1_", "p2_"))])
def test_golden_worked_examples(name):
    g = read_golden(name)
    mode = oracle.MODE_BINARY if g["mode"] == "binary" else oracle.MODE_ALL
    lab, n = oracle.label(g["image"].astype(np.uint8), g["connectivity"], mode)
    np.testing.assert_array_equal(lab, g["labels"])
    assert n == g["n"]
    # the brute force agrees with the same fixtures (pins the pin)
    bl, bn = closure_labels(g["image"][None], g["connectivity"], mode == oracle.MODE_BINARY)
    np.testing.assert_array_equal(bl[0], g["labels"])
    assert bn[0] == g["n"]


def test_p2_printed_roots():
    # bendabir.com, "The basic approach": after the scan the roots are 0, 12, 15.
    g = read_golden("p2_4x4_binary_8conn.txt")
    lab, n = oracle.label(g["image"].astype(np.uint8), 8, oracle.MODE_BINARY)
    flat = lab.reshape(-1)
    firsts = [int(np.flatnonzero(flat == k)[0]) for k in range(1, n + 1)]
    assert firsts == [0, 12, 15]


def _all_binary_4x4():
    k = np.arange(1 << 16, dtype=np.int64)
    bits = (k[:, None] >> np.arange(16)[None, :]) & 1
    return bits.reshape(-1, 4, 4).astype(np.uint8)


@pytest.mark.parametrize("conn", [4, 8])
@pytest.mark.parametrize("binary", [False, True])
def test_bruteforce_all_binary_4x4(conn, binary):
    imgs = _all_binary_4x4()
    mode = oracle.MODE_BINARY if binary else oracle.MODE_ALL
    lab, n = oracle.label(imgs, conn, mode)
    bl, bn = closure_labels(imgs, conn, binary)
    np.testing.assert_array_equal(lab, bl)
    np.testing.assert_array_equal(n, bn)


@pytest.mark.parametrize("conn", [4, 8])
@pytest.mark.parametrize("binary", [False, True])
def test_bruteforce_all_3colour_3x3(conn, binary):
    imgs = np.array(list(itertools.product(range(3), repeat=9)), dtype=np.uint8).reshape(-1, 3, 3)
    mode = oracle.MODE_BINARY if binary else oracle.MODE_ALL
    lab, n = oracle.label(imgs, conn, mode)
    bl, bn = closure_labels(imgs, conn, binary)
    np.testing.assert_array_equal(lab, bl)
    np.testing.assert_array_equal(n, bn)


# ---------------------------------------------------------------- closed forms

def checkerboard(H, W):
    r, c = np.indices((H, W))
    return ((r + c) & 1).astype(np.uint8)


def serpentine(H, W):
    img = np.zeros((H, W), np.uint8)
    img[0::2, :] = 1
    img[1::4, W - 1] = 1
    img[3::4, 0] = 1
    return img


@pytest.mark.parametrize("H,W", [(2, 2), (8, 8), (7, 10), (64, 48), (5, 3)])
def test_checkerboard_closed_form(H, W):
    img = checkerboard(H, W)
    r, c = np.indices((H, W))
    lab, n = oracle.label(img, 8, oracle.MODE_ALL)
    assert n == 2
    np.testing.assert_array_equal(lab, 1 + ((r + c) & 1))
    lab, n = oracle.label(img, 4, oracle.MODE_ALL)
    assert n == H * W
    np.testing.assert_array_equal(lab, r * W + c + 1)
    lab, n = oracle.label(img, 8, oracle.MODE_BINARY)
    assert n == 1
    np.testing.assert_array_equal(lab, (r + c) & 1)
    lab, n = oracle.label(img, 4, oracle.MODE_BINARY)
    assert n == (H * W) // 2
    ones = ((r + c) & 1).reshape(-1) == 1
    expect = np.zeros(H * W, np.int64)
    expect[ones] = np.arange(1, ones.sum() + 1)
    np.testing.assert_array_equal(lab.reshape(-1), expect)


@pytest.mark.parametrize("n_side", [4, 8, 64, 256])
@pytest.mark.parametrize("conn", [4, 8])
def test_serpentine_closed_form(n_side, conn):
    H = W = n_side
    img = serpentine(H, W)
    lab, n = oracle.label(img, conn, oracle.MODE_BINARY)
    assert n == 1
    np.testing.assert_array_equal(lab, img)
    lab, n = oracle.label(img, conn, oracle.MODE_ALL)
    assert n == 1 + H // 2
    r = np.arange(H)
    # zeros of odd row r form region 1 + (r + 1) / 2; the ones are region 1
    expect = np.where(img == 1, 1, (1 + (r + 1) // 2)[:, None])
    np.testing.assert_array_equal(lab, expect)
    # the single ones-region is H/2*W + H/2 pixels long
    assert (lab == 1).sum() == (H // 2) * W + H // 2


@pytest.mark.parametrize("conn", [4, 8])
def test_stripes_constant_distinct(conn):
    H, W = 10, 13
    stripes = np.zeros((H, W), np.uint8)
    stripes[0::2] = 1
    lab, n = oracle.label(stripes, conn, oracle.MODE_ALL)
    assert n == H
    np.testing.assert_array_equal(lab, np.repeat(np.arange(1, H + 1)[:, None], W, 1))
    lab, n = oracle.label(stripes, conn, oracle.MODE_BINARY)
    assert n == H // 2
    const = np.full((H, W), 7, np.uint32)
    lab, n = oracle.label(const, conn, oracle.MODE_ALL)
    assert n == 1 and (lab == 1).all()
    lab, n = oracle.label(np.zeros((H, W), np.uint32), conn, oracle.MODE_BINARY)
    assert n == 0 and (lab == 0).all()
    distinct = np.arange(H * W, dtype=np.uint32).reshape(H, W)
    lab, n = oracle.label(distinct, conn, oracle.MODE_ALL)
    assert n == H * W
    np.testing.assert_array_equal(lab, distinct.astype(np.int64) + 1)
    lab, n = oracle.label(distinct, conn, oracle.MODE_BINARY)
    assert n == H * W - 1
    np.testing.assert_array_equal(lab, distinct.astype(np.int64))


def test_rgba_alpha_counts():
    # equality covers all four bytes: two pixels differing only in alpha differ
    img = np.full((3, 4), 0xFFFFFFFF, np.uint32)
    img[1, 1] = 0x7FFFFFFF
    lab, n = oracle.label(img, 8, oracle.MODE_ALL)
    assert n == 2 and lab[1, 1] == 2


@pytest.mark.parametrize("conn", [4, 8])
def test_rgb_three_byte_pixels(conn):
    """Packed 24-bit RGB ("every-colour", ch. 08 "Tried and dropped": RGB read
    as is): labelling the [H, W, 3] bytes gives the labels of the same colours
    packed into one 32-bit word with an opaque alpha, and two pixels that
    differ only in their third byte are different colours."""
    rng = np.random.default_rng(11)
    rgb = rng.integers(0, 2, size=(37, 53, 3)).astype(np.uint8) * np.array([0, 7, 200], np.uint8)
    packed = (rgb[..., 0].astype(np.uint32) | (rgb[..., 1].astype(np.uint32) << 8)
              | (rgb[..., 2].astype(np.uint32) << 16) | np.uint32(0xFF000000))
    lab3, n3 = oracle.label(rgb[None], conn, oracle.MODE_ALL)
    lab4, n4 = oracle.label(packed, conn, oracle.MODE_ALL)
    np.testing.assert_array_equal(lab3[0], lab4)
    assert n3[0] == n4
    two = np.zeros((1, 1, 2, 3), np.uint8)
    two[0, 0, 1, 2] = 1                               # only the blue byte differs
    lab, n = oracle.label(two, conn, oracle.MODE_ALL)
    assert n[0] == 2 and lab[0, 0].tolist() == [1, 2]


def test_empty_and_degenerate_shapes():
    for shape in [(0, 5), (5, 0), (0, 0)]:
        lab, n = oracle.label(np.zeros(shape, np.uint8), 8, oracle.MODE_ALL)
        assert n == 0 and lab.shape == shape
    lab, n = oracle.label(np.zeros((0, 3, 3), np.uint8), 8, oracle.MODE_ALL)
    assert lab.shape == (0, 3, 3) and n.shape == (0,)
    lab, n = oracle.label(np.array([[5]], np.uint8), 4, oracle.MODE_ALL)
    assert n == 1 and lab[0, 0] == 1
    row = np.array([[1, 1, 0, 2, 2, 2, 0, 1]], np.uint8)
    lab, n = oracle.label(row, 8, oracle.MODE_BINARY)
    np.testing.assert_array_equal(lab, [[1, 1, 0, 2, 2, 2, 0, 3]])
    lab, n = oracle.label(row.T.copy(), 4, oracle.MODE_ALL)
    np.testing.assert_array_equal(lab.T, [[1, 1, 2, 3, 3, 3, 4, 5]])


def test_batch_numbering_restarts_per_image():
    rng = np.random.default_rng(5)
    imgs = (rng.random((6, 17, 23)) < 0.5).astype(np.uint8)
    lab, n = oracle.label(imgs, 8, oracle.MODE_BINARY)
    for b in range(6):
        lb, nb = oracle.label(imgs[b], 8, oracle.MODE_BINARY)
        np.testing.assert_array_equal(lab[b], lb)
        assert n[b] == nb


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("conn", [4, 8])
@pytest.mark.parametrize("binary", [False, True])
def test_against_scipy_random(seed, conn, binary):
    rng = np.random.default_rng(seed)
    H, W = rng.integers(20, 90, size=2)
    for dtype, k in [(np.uint8, 4), (np.uint32, 3)]:
        img = rng.integers(0, k, size=(H, W)).astype(dtype)
        mode = oracle.MODE_BINARY if binary else oracle.MODE_ALL
        lab, n = oracle.label(img, conn, mode)
        sl, sn = scipy_labels(img, conn, binary)
        np.testing.assert_array_equal(lab, sl)
        assert n == sn
        assert check_invariants(img, lab, n, conn, binary) == []


def test_invariant_checker_catches_errors():
    rng = np.random.default_rng(0)
    img = rng.integers(0, 3, size=(30, 30)).astype(np.uint8)
    lab, n = oracle.label(img, 8, oracle.MODE_ALL)
    assert check_invariants(img, lab, n, 8, False) == []
    bad = lab.copy()
    bad[bad == 3], bad[bad == 4] = 4, 3          # swapped numbering
    assert check_invariants(img, bad, n, 8, False)
    bad = lab.copy()
    bad[0, 0] = bad[0, 0] + 1 if bad[0, 0] < n else 1  # one pixel moved
    assert check_invariants(img, bad, n, 8, False)


# ------------------------------------------------------------ mutation checks

MUTATIONS = {
    # 8-connectivity that forgets the corner-sharing neighbours
    "no_diagonals": ("const int nn = (conn == 8) ? 8 : 4;", "const int nn = 4;"),
    # neighbours found by flat index +-1, so rows wrap around
    "row_wrap": ("const int64_t rr = r + dr[k], cc = c + dc[k];",
                 "int64_t rr = r + dr[k], cc = c + dc[k]; "
                 "if (cc < 0) { rr -= 1; cc += W; } if (cc >= W) { rr += 1; cc -= W; }"),
    # compare only the first byte of a pixel
    "short_compare": ("return memcmp(a, b, (size_t)pb) == 0;", "return a[0] == b[0];"),
    # binary background not ignored
    "no_background": ("if (mode == ORACLE_MODE_BINARY && is_zero(v, pb))", "if (0)"),
    # seeds taken from the last pixel backwards (numbering not in raster order)
    "reverse_scan": ("for (int64_t seed = 0; seed < N; ++seed)",
                     "for (int64_t seed = N - 1; seed >= 0; --seed)"),
    # numbering restarts are dropped (labels continue across the batch)
    "global_numbering": ("int64_t n = 0;\n  for (int64_t seed", "static int64_t n = 0;\n  for (int64_t seed"),
}


def _build_mutant(tmp_path, key):
    src = open(oracle._SRC).read()
    old, new = MUTATIONS[key]
    assert old in src, key
    path = tmp_path / ("m_%s.c" % key)
    path.write_text(src.replace(old, new, 1))
    so = tmp_path / ("m_%s.so" % key)
    subprocess.check_call(["gcc", "-O1", "-std=c99", "-shared", "-fPIC", "-o", str(so), str(path)])
    import ctypes
    lib = ctypes.CDLL(str(so))
    lib.oracle_label.restype = ctypes.c_int
    lib.oracle_label.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_void_p, ctypes.c_void_p]
    return lib


def _run(lib, imgs, conn, mode):
    imgs = np.ascontiguousarray(imgs)
    B, H, W = imgs.shape
    lab = np.empty((B, H, W), np.int32)
    n = np.empty(B, np.int32)
    lib.oracle_label(imgs.ctypes.data, B, H, W, imgs.dtype.itemsize, conn, mode,
                     lab.ctypes.data, n.ctypes.data)
    return lab, n


@pytest.mark.parametrize("key", sorted(MUTATIONS))
def test_pins_catch_planted_mistakes(tmp_path, key):
    lib = _build_mutant(tmp_path, key)
    caught = False
    imgs = _all_binary_4x4()
    for conn, binary in [(8, False), (8, True), (4, True)]:
        lab, n = _run(lib, imgs, conn, int(binary))
        bl, bn = closure_labels(imgs, conn, binary)
        caught |= not (np.array_equal(lab, bl) and np.array_equal(n, bn))
    img = np.full((1, 3, 4), 0xFFFFFFFF, np.uint32)
    img[0, 1, 1] = 0x7FFFFFFF                      # differs only in the top byte
    lab, n = _run(lib, img, 8, 0)
    caught |= int(n[0]) != 2
    assert caught, key


# ------------------------------------------------------ ignoring one value
# "every-colour", ch. 08 switch 4 "Ignore the paper": pixels of the named
# value get label 0 and take part in nothing.

@pytest.mark.parametrize("conn", [4, 8])
@pytest.mark.parametrize("ignore", [0, 1, 2])
def test_ignore_bruteforce_all_3colour_3x3(conn, ignore):
    imgs = np.array(list(itertools.product(range(3), repeat=9)), dtype=np.uint8).reshape(-1, 3, 3)
    lab, n = oracle.label_ignore(imgs, ignore, conn)
    bl, bn = closure_labels(imgs, conn, False, ignore=ignore)
    np.testing.assert_array_equal(lab, bl)
    np.testing.assert_array_equal(n, bn)


@pytest.mark.parametrize("conn", [4, 8])
def test_ignore_zero_is_binary_mode(conn):
    rng = np.random.default_rng(7)
    imgs = rng.integers(0, 4, size=(3, 41, 67)).astype(np.uint8)
    a, na = oracle.label_ignore(imgs, 0, conn)
    b, nb = oracle.label(imgs, conn, oracle.MODE_BINARY)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(na, nb)


@pytest.mark.parametrize("conn", [4, 8])
def test_ignore_white_on_rgba_against_scipy(conn):
    import workloads
    img = workloads.drawing(150, 230, seed=3, n_segments=40, n_rects=5, levels=16,
                            hatched=False).numpy().view(np.uint32)
    lab, n = oracle.label_ignore(img, 0xFFFFFFFF, conn)
    sl, sn = scipy_labels(img, conn, False, ignore=0xFFFFFFFF)
    np.testing.assert_array_equal(lab, sl)
    assert n == sn
    assert (lab[img == 0xFFFFFFFF] == 0).all()


def test_ignore_compares_every_byte(tmp_path):
    # a copy that compares only the first byte against the ignored value
    # must fail this pin: 0x7FFFFFFF differs from white only in alpha
    img = np.full((2, 3), 0x7FFFFFFF, np.uint32)
    lab, n = oracle.label_ignore(img, 0xFFFFFFFF, 8)
    assert n == 1 and (lab == 1).all()
    src = open(oracle._SRC).read()
    old = "else if (ign && same_value(v, ign, pb))"
    assert old in src
    path = tmp_path / "m_ign.c"
    path.write_text(src.replace(old, "else if (ign && v[0] == ign[0])", 1))
    so = tmp_path / "m_ign.so"
    subprocess.check_call(["gcc", "-O1", "-std=c99", "-shared", "-fPIC", "-o", str(so), str(path)])
    import ctypes
    lib = ctypes.CDLL(str(so))
    ign = np.frombuffer((0xFFFFFFFF).to_bytes(4, "little"), np.uint8).copy()
    out = np.empty((1, 2, 3), np.int32)
    cnt = np.empty(1, np.int32)
    lib.oracle_label_ignore(ctypes.c_void_p(img.ctypes.data), ctypes.c_int64(1), ctypes.c_int64(2),
                            ctypes.c_int64(3), 4, 8, ctypes.c_void_p(ign.ctypes.data),
                            ctypes.c_void_p(out.ctypes.data), ctypes.c_void_p(cnt.ctypes.data))
    assert cnt[0] != 1          # the planted mistake is caught


def _free_memory_bytes():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def test_image_beyond_2_31_pixels():
    """"every-colour" ch. 11 names images of more than 2^31 pixels as the case
    it never ran; the oracle indexes in 64 bits and accepts up to 2^32 - 1
    pixels.  One row of 2^31 + 3000 pixels in runs of 2^20 of alternating
    value (4-connectivity): run k is region k + 1, so the last pixels carry
    a label past 2^11 with raster indices past 2^31.  Needs about 28 GB of
    host memory (image, labels, the flood fill's queue)."""
    W = (1 << 31) + 3000
    if _free_memory_bytes() < 34 * (1 << 30):
        pytest.skip("needs about 28 GB of free host memory")
    x = np.arange(W, dtype=np.int64)
    img = ((x >> 20) & 1).astype(np.uint8).reshape(1, W)
    del x
    lab, n = oracle.label(img, 4, oracle.MODE_ALL)
    del img
    assert int(n) == (W + (1 << 20) - 1) >> 20
    step = 1 << 27
    for x0 in range(0, W, step):
        xs = np.arange(x0, min(W, x0 + step), dtype=np.int64)
        np.testing.assert_array_equal(lab[0, x0:x0 + len(xs)], ((xs >> 20) + 1).astype(np.int32))


def test_images_of_2_32_pixels_refused():
    """Images of 2^32 pixels or more are refused (status 2), as by the
    library; nothing is read (the pointers are never touched)."""
    import ctypes
    n = (ctypes.c_int32 * 1)()
    rc = oracle._load().oracle_label(ctypes.c_void_p(16), 1, 1 << 16, 1 << 16, 1, 4, 0,
                                     ctypes.c_void_p(16), n)
    assert rc == 2
