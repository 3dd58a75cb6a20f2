"""GPU labelling at the largest images: just below 2^31 pixels (labels near
the top of the int32 range), past 2^31 ("every-colour" ch. 11: images of
more than 2^31 pixels are the case it never ran) and just below 2^32, the
largest the library accepts (raster keys inside an image are 32-bit).  The
images have closed-form labels, checked chunk by chunk on the device (an
oracle pass at this size would take minutes; the closed forms are pinned
against the oracle at small sizes in tests/test_oracle_pins.py, and the
oracle itself past 2^31 there too)."""
import pytest
import torch

import connected_component_labelling_gb300 as ccl

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
N = 46340                      # N * N = 2,147,395,600 < 2^31 - 1
N2 = 46341                     # N2 * N2 = 2,147,488,281 > 2^31
N3 = 65535                     # N3 * N3 = 4,294,836,225 < 2^32
W1 = (1 << 31) - 1             # the widest one-row image
CHUNK = 2048                   # rows compared at a time


@pytest.fixture(scope="module", autouse=True)
def built():
    ccl.build()
    yield
    torch.cuda.empty_cache()


MODES = {"all": ccl.CCL_MODE_ALL, "binary": ccl.CCL_MODE_BINARY}


def label_ws(img, conn, mode):
    B, H, W, pb, squeeze = ccl.image_geometry(img)
    need = ccl.ccl_workspace_bytes(B, H, W, pb, conn, MODES[mode])
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    lab, n = ccl.label(img, conn, mode, workspace=ws)
    ccl.check_status()
    del ws
    return lab, n


def checkerboard(n=N):
    r = torch.arange(n, device=DEV, dtype=torch.int32)
    return ((r[:, None] + r[None, :]) & 1).to(torch.uint8)


def test_checkerboard_8conn_all_at_max_size():
    """Two regions: even cells (first pixel 0) and odd cells (first pixel 1)."""
    img = checkerboard()
    lab, n = label_ws(img, 8, "all")
    assert int(n) == 2
    c = torch.arange(N, device=DEV, dtype=torch.int32)
    for r0 in range(0, N, CHUNK):
        r = torch.arange(r0, min(N, r0 + CHUNK), device=DEV, dtype=torch.int32)
        exp = 1 + ((r[:, None] + c[None, :]) & 1)
        assert torch.equal(lab[r0:r0 + len(r)], exp), r0
    del lab, img


def test_checkerboard_4conn_all_at_max_size():
    """Every pixel its own region: label = raster index + 1, up to N² =
    2,147,395,600, the largest label an accepted image can have."""
    img = checkerboard()
    lab, n = label_ws(img, 4, "all")
    assert int(n) == N * N
    c = torch.arange(N, device=DEV, dtype=torch.int64)
    for r0 in range(0, N, CHUNK):
        r = torch.arange(r0, min(N, r0 + CHUNK), device=DEV, dtype=torch.int64)
        exp = (r[:, None] * N + c[None, :] + 1).to(torch.int32)
        assert torch.equal(lab[r0:r0 + len(r)], exp), r0
    del lab, img


def test_checkerboard_4conn_binary_at_max_size():
    """Every 1 its own region, numbered in raster order: a row holds N/2 ones,
    so the one at (r, c) is number r·N/2 + c//2 + 1; zeros are 0."""
    img = checkerboard()
    lab, n = label_ws(img, 4, "binary")
    assert int(n) == N * N // 2
    c = torch.arange(N, device=DEV, dtype=torch.int64)
    for r0 in range(0, N, CHUNK):
        r = torch.arange(r0, min(N, r0 + CHUNK), device=DEV, dtype=torch.int64)
        one = ((r[:, None] + c[None, :]) & 1) == 1
        exp = torch.where(one, r[:, None] * (N // 2) + c[None, :] // 2 + 1, 0).to(torch.int32)
        assert torch.equal(lab[r0:r0 + len(r)], exp), r0
    del lab, img


def test_one_row_of_max_width():
    """One row of 2^31 - 1 pixels in runs of 1024 of alternating value: the
    run index + 1 is the label (8.4 M tiles in one tile row)."""
    x = torch.arange(W1, device=DEV, dtype=torch.int64)
    img = ((x >> 10) & 1).to(torch.uint8).view(1, W1)
    del x
    lab, n = label_ws(img, 8, "all")
    assert int(n) == (W1 + 1023) // 1024
    step = 1 << 28
    for x0 in range(0, W1, step):
        xs = torch.arange(x0, min(W1, x0 + step), device=DEV, dtype=torch.int64)
        assert torch.equal(lab[0, x0:x0 + len(xs)], ((xs >> 10) + 1).to(torch.int32)), x0
    del img, xs
    # region statistics of the same labels: run k covers columns 1024k ..
    # min(W, 1024(k+1)) - 1 of row 0
    raw, f = ccl.region_stats(lab, n)
    ccl.check_status()
    k = torch.arange(int(n), device=DEV, dtype=torch.int64)
    x_min = k * 1024
    x_max = torch.clamp((k + 1) * 1024, max=W1) - 1
    area = x_max - x_min + 1
    assert torch.equal(f["area"].to(torch.int64), area)
    assert torch.equal(f["x_min"].to(torch.int64), x_min)
    assert torch.equal(f["x_max"].to(torch.int64), x_max)
    assert torch.equal(f["first"].to(torch.int64), x_min)
    assert int(f["y_min"].abs().sum()) == 0 and int(f["y_max"].abs().sum()) == 0
    assert int(f["sum_y"].abs().sum()) == 0
    assert torch.equal(f["sum_x"], (x_min + x_max) * area // 2)
    del lab, raw, f


def test_checkerboard_8conn_all_beyond_2_31():
    """Past 2^31 pixels: still the two diagonal families."""
    img = checkerboard(N2)
    assert N2 * N2 > (1 << 31)
    lab, n = label_ws(img, 8, "all")
    assert int(n) == 2
    c = torch.arange(N2, device=DEV, dtype=torch.int32)
    for r0 in range(0, N2, CHUNK):
        r = torch.arange(r0, min(N2, r0 + CHUNK), device=DEV, dtype=torch.int32)
        assert torch.equal(lab[r0:r0 + len(r)], 1 + ((r[:, None] + c[None, :]) & 1)), r0
    del lab, img


def test_checkerboard_4conn_binary_beyond_2_31():
    """Every 1 its own region past 2^31 pixels (N2 odd): rows hold 23170 and
    23171 ones alternately, so the one at (r, c) is number
    r*23170 + r//2 + c//2 + 1, the last one (N2*N2 - 1) / 2."""
    img = checkerboard(N2)
    lab, n = label_ws(img, 4, "binary")
    assert int(n) == (N2 * N2 - 1) // 2
    c = torch.arange(N2, device=DEV, dtype=torch.int64)
    for r0 in range(0, N2, CHUNK):
        r = torch.arange(r0, min(N2, r0 + CHUNK), device=DEV, dtype=torch.int64)
        one = ((r[:, None] + c[None, :]) & 1) == 1
        exp = torch.where(one, r[:, None] * ((N2 - 1) // 2) + r[:, None] // 2 + c[None, :] // 2 + 1, 0)
        assert torch.equal(lab[r0:r0 + len(r)], exp.to(torch.int32)), r0
    del lab, img


def test_more_regions_than_int32_labels_reported():
    """The 4-connected all-pixels checkerboard past 2^31 pixels has N2*N2 >
    2^31 - 1 regions: more than int32 labels hold.  The call completes and
    the device status reports CCL_ERR_TOO_LARGE (the counts are clamped)."""
    img = checkerboard(N2)
    B, H, W, pb, _ = ccl.image_geometry(img)
    ws = torch.empty(ccl.ccl_workspace_bytes(B, H, W, pb, 4, 0), dtype=torch.uint8, device=DEV)
    lab, n = ccl.label(img, 4, "all", workspace=ws)
    with pytest.raises(ccl.CCLError) as e:
        ccl.check_status()
    assert e.value.status == ccl.CCL_ERR_TOO_LARGE
    assert int(n) == (1 << 31) - 1
    del lab, ws, img


def test_checkerboard_8conn_all_near_2_32():
    """The largest square accepted, 65535^2 = 2^32 - 2^17 + 1 pixels."""
    img = checkerboard(N3)
    lab, n = label_ws(img, 8, "all")
    assert int(n) == 2
    c = torch.arange(N3, device=DEV, dtype=torch.int32)
    for r0 in range(0, N3, CHUNK):
        r = torch.arange(r0, min(N3, r0 + CHUNK), device=DEV, dtype=torch.int32)
        assert torch.equal(lab[r0:r0 + len(r)], 1 + ((r[:, None] + c[None, :]) & 1)), r0
    del lab, img


def test_serpentine_binary_near_2_32():
    """One serpentine of 1s through 65535^2 pixels (even rows all 1, odd rows
    a single 1 at alternate ends): one region of 2^31 + 2^15 pixels whose
    joins chain through every tile seam of the image; label 1 on the 1s."""
    r = torch.arange(N3, device=DEV, dtype=torch.int64)
    c = torch.arange(N3, device=DEV, dtype=torch.int64)
    img = torch.zeros((N3, N3), dtype=torch.uint8, device=DEV)
    img[0::2] = 1
    img[1::4, N3 - 1] = 1
    img[3::4, 0] = 1
    lab, n = label_ws(img, 8, "binary")
    assert int(n) == 1
    for r0 in range(0, N3, CHUNK):
        assert torch.equal(lab[r0:r0 + CHUNK], img[r0:r0 + CHUNK].to(torch.int32)), r0
    del lab, img, r, c
