"""CPU checks of the seeded input generators against the recipes they state:
a band of a drawing rendered alone equals the same rows of the whole picture
(the CPU baseline labels such a band of the sheet), the RGB sheet is the RGBA
sheet without its alpha byte, alpha is opaque, the sheet is mostly paper, the
slide's foreground is exactly the part above its 55th-percentile value, the
masks' foreground fractions follow their p, and every generator is
deterministic in its seed."""
import math

import numpy as np
import torch

import workloads as wl

H, W = 1200, 1680          # the sheet generator at 1/400 of its full area


def test_sheet_band_equals_the_rows_of_the_whole_sheet():
    full = wl.c4_sheet(H=H, W=W)
    for r0, r1 in ((0, 16), (300, 777), (1184, 1200)):
        assert torch.equal(wl.c4_sheet(H=H, W=W, rows=(r0, r1)), full[r0:r1]), (r0, r1)


def test_drawing_band_equals_the_rows_of_the_whole_drawing():
    full = wl.c0_drawing()
    assert torch.equal(wl.c0_drawing(rows=(511, 600)), full[511:600])


def test_sheet_pixels_are_opaque_and_mostly_paper():
    full = wl.c4_sheet(H=H, W=W)
    px = full.numpy().view(np.uint32)
    assert ((px >> 24) == 255).all()                      # alpha 255 everywhere
    paper = float((px == 0xFFFFFFFF).mean())
    assert 0.80 < paper < 0.92, paper                     # about 86 % white paper
    assert len(np.unique(px)) > 64                        # anti-aliased shades: many colours


def test_rgb_sheet_is_the_rgba_sheet_without_alpha():
    rgba = wl.c4_sheet(H=H, W=W)
    rgb = wl.c4_sheet_rgb(H=H, W=W)
    assert rgb.shape == (1, H, W, 3) and rgb.dtype == torch.uint8
    assert torch.equal(rgb[0], rgba.view(torch.uint8).reshape(H, W, 4)[:, :, :3])


def test_slide_foreground_is_above_the_55th_percentile():
    s = wl.tissue_slide(512, 512, seed=5)
    n = 512 * 512
    assert s.dtype == torch.uint8 and set(s.unique().tolist()) == {0, 1}
    assert int(s.sum()) == n - math.ceil(0.55 * n)        # continuous values: no ties


def test_mask_foreground_fractions_follow_p():
    m = wl.bernoulli_masks(8, 256, 256, (0.2, 0.4, 0.6, 0.8), seed=1)
    for b in range(8):
        p = (0.2, 0.4, 0.6, 0.8)[b * 4 // 8]
        assert abs(float(m[b].float().mean()) - p) < 0.01, (b, p)


def test_generators_are_deterministic_in_their_seed():
    a = wl.drawing(200, 300, seed=9, n_segments=30, n_rects=4, levels=16, hatched=True)
    b = wl.drawing(200, 300, seed=9, n_segments=30, n_rects=4, levels=16, hatched=True)
    c = wl.drawing(200, 300, seed=10, n_segments=30, n_rects=4, levels=16, hatched=True)
    assert torch.equal(a, b) and not torch.equal(a, c)
    assert torch.equal(wl.random_levels(64, 64, 4, seed=3), wl.random_levels(64, 64, 4, seed=3))
    assert torch.equal(wl.tissue_slide(128, 128, seed=2), wl.tissue_slide(128, 128, seed=2))
