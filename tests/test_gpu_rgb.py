"""GPU parity for packed 24-bit RGB input (pixel_bytes 3): three bytes a
pixel, no padding, compared as one 24-bit value ("every-colour", ch. 08
"Tried and dropped": the drawings are read as RGB, not packed to 32 bits).
Bit-exact against the oracle (which compares the three bytes with memcmp).
Covers the vector path (row length a multiple of 8, 8-byte aligned base),
the scalar path (other row lengths, a base 3 bytes off), the three modes and
colours that differ in one byte only."""
import numpy as np
import pytest
import torch

import connected_component_labelling_gb300 as ccl
import oracle
import workloads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def built():
    ccl.build()
    oracle.build()


def rgb_from_levels(B, H, W, levels, seed, byte=None):
    """uint8 [B,H,W,3]: colours drawn from `levels` fixed RGB triples; with
    `byte`, the triples differ only in that byte."""
    rng = np.random.default_rng(seed)
    if byte is None:
        pal = rng.integers(0, 256, size=(levels, 3), dtype=np.uint8)
    else:
        pal = np.tile(np.array([[10, 20, 30]], np.uint8), (levels, 1))
        pal[:, byte] = np.arange(levels, dtype=np.uint8) * 7
    idx = rng.integers(0, levels, size=(B, H, W))
    return pal[idx]


def check(host, conn, mode, dev_img=None):
    img = dev_img if dev_img is not None else torch.from_numpy(host).to(DEV)
    lab, n = ccl.label(img, conn, mode)
    ccl.check_status()
    olab, on = oracle.label(host, conn, mode)
    np.testing.assert_array_equal(n.cpu().numpy().reshape(-1), np.asarray(on).reshape(-1))
    assert np.array_equal(lab.cpu().numpy().reshape(olab.shape), olab)


@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 5, 7), (1, 16, 256), (2, 17, 264), (1, 40, 250),
                                   (3, 33, 517)])
@pytest.mark.parametrize("conn", [4, 8])
@pytest.mark.parametrize("mode", [ccl.CCL_MODE_ALL, ccl.CCL_MODE_BINARY])
def test_random_colours(shape, conn, mode):
    B, H, W = shape
    host = rgb_from_levels(B, H, W, 3, seed=H * 131 + W)
    host[..., :][host.sum(axis=-1) < 200] = 0           # some all-zero (background) pixels
    check(host, conn, mode)


@pytest.mark.parametrize("byte", [0, 1, 2])
def test_colours_differing_in_one_byte(byte):
    host = rgb_from_levels(1, 48, 264, 2, seed=byte, byte=byte)
    check(host, 8, ccl.CCL_MODE_ALL)


def test_unaligned_base():
    host = rgb_from_levels(1, 37, 272, 3, seed=11)
    buf = torch.zeros(host.size + 8, dtype=torch.uint8, device=DEV)
    view = buf[3:3 + host.size].view(1, 37, 272, 3)     # 3 bytes past an aligned start
    view.copy_(torch.from_numpy(host).to(DEV))
    check(host, 8, ccl.CCL_MODE_ALL, dev_img=view)


def test_drawing_as_rgb_matches_rgba_and_oracle():
    rgba = workloads.c0_drawing(device=DEV)
    rgb = rgba.view(torch.uint8).reshape(1024, 1024, 4)[:, :, :3].contiguous().reshape(1, 1024, 1024, 3)
    la, na = ccl.label(rgba, 8, ccl.CCL_MODE_ALL)
    lb, nb = ccl.label(rgb, 8, ccl.CCL_MODE_ALL)
    assert int(na) == int(nb[0])                          # alpha is 255 everywhere
    assert torch.equal(la.reshape(-1), lb.reshape(-1))
    check(rgb.cpu().numpy(), 8, ccl.CCL_MODE_ALL, dev_img=rgb)


def test_ignore_white_rgb():
    rgba = workloads.c0_drawing(device=DEV)
    rgb = rgba.view(torch.uint8).reshape(1024, 1024, 4)[:, :, :3].contiguous().reshape(1, 1024, 1024, 3)
    lab, n = ccl.label_ignore(rgb, 0xFFFFFF, connectivity=8)
    ccl.check_status()
    olab, on = oracle.label_ignore(rgb.cpu().numpy(), 0xFFFFFF, 8)
    assert int(n[0]) == int(on[0])
    assert np.array_equal(lab.cpu().numpy(), olab)


def test_sheet_rgb_full_size():
    rgb = workloads.c4_sheet_rgb(device=DEV)
    assert rgb.shape == (1, 24000, 33600, 3)
    lab, n = ccl.label(rgb, 8, ccl.CCL_MODE_ALL)
    ccl.check_status()
    host = rgb.cpu().numpy()
    del rgb
    olab, on = oracle.label(host, 8, oracle.MODE_ALL)
    assert int(n[0]) == int(on[0])
    assert np.array_equal(lab.cpu().numpy(), olab)
