"""Seeded synthetic inputs for connected-component labelling.

This module only draws pictures; it holds none of the labelling arithmetic and
is shared by the tests, the benchmark and the smoke check (both the oracle and
the CUDA library are fed the very same arrays).

The pages label real construction drawings, NVIDIA sample images, YACCLAB sets
and tissue scans, none of which exist here; these generators stand in for them
with the same structure:

* ``drawing``        -- RGBA line drawing on white paper: palette-coloured
                        rectangles (solid, or outlined and hatched), black
                        anti-aliased segments whose coverage is quantised to a
                        fixed number of grey levels, so every shade is its own
                        colour ("every-colour", ch. 01, Fig. 2);
* ``bernoulli_masks``-- batches of i.i.d. binary masks;
* ``tissue_slide``   -- Gaussian-smoothed white noise thresholded at a
                        percentile (blob-like regions, as in the tissue scans of
                        the lpnh.cn page, section 1.1);
* ``serpentine``, ``checkerboard``, ``random_levels`` -- adversarial structures.

Rendering model used by ``drawing`` (a stated reading of "Wu-style
anti-aliasing"): a pixel's coverage by a stroke of width w is
clamp(w/2 + 0.5 - d, 0, 1), d the distance from the pixel centre to the
segment; it is quantised to L levels; where strokes overlap the pixel takes
the largest coverage (a union of strokes), rectangles drawn later lie on top,
and a covered pixel's channel is round(base * (1 - q) + ink * q).
"""
from __future__ import annotations

import math

import numpy as np
import torch

WHITE = 0xFFFFFFFF

# 8 opaque palette colours (R, G, B)
PALETTE = np.array([
    (220, 30, 30), (30, 150, 40), (30, 60, 210), (230, 160, 20),
    (150, 40, 170), (20, 170, 180), (120, 80, 40), (240, 90, 160),
], dtype=np.int64)


def pack_rgba(r, g, b, a=None):
    """Pack uint8-valued channels into little-endian RGBA uint32 (as int64
    tensors; callers cast)."""
    if a is None:
        a = torch.full_like(r, 255)
    return r | (g << 8) | (b << 16) | (a << 24)


# --------------------------------------------------------------- rasteriser

def _raster_segments(x0, y0, x1, y1, w, levels, H, W, row0, row1, device,
                     out_flat, key=None, chunk=40_000_000):
    """Scatter-max the quantised coverage of every segment into ``out_flat``
    (int32, rows [row0, row1) of a W-wide image, flattened).  ``key``: an
    optional int32 per segment; the stored value is key*levels + level so that
    the largest key wins and, within a key, the largest coverage."""
    S = len(x0)
    if S == 0:
        return
    x0 = np.asarray(x0, np.float64); y0 = np.asarray(y0, np.float64)
    x1 = np.asarray(x1, np.float64); y1 = np.asarray(y1, np.float64)
    w = np.asarray(w, np.float64)
    pad = w / 2.0 + 1.0
    horiz = np.abs(x1 - x0) >= np.abs(y1 - y0)
    a0 = np.where(horiz, x0, y0); a1 = np.where(horiz, x1, y1)
    b0 = np.where(horiz, y0, x0); b1 = np.where(horiz, y1, x1)
    da = a1 - a0
    slope = np.where(np.abs(da) > 0, (b1 - b0) / np.where(da == 0, 1, da), 0.0)
    lo = np.floor(np.minimum(a0, a1) - pad).astype(np.int64)
    hi = np.ceil(np.maximum(a0, a1) + pad).astype(np.int64)
    # clip the major range to the picture (plus nothing: outside pixels drop)
    amax = np.where(horiz, W - 1, H - 1)
    lo = np.maximum(lo, 0); hi = np.minimum(hi, amax)
    hm = (np.ceil(pad * np.sqrt(1.0 + slope * slope)) + 1).astype(np.int64)
    # drop segments that miss the row window
    ymin = np.minimum(y0, y1) - pad - 1; ymax = np.maximum(y0, y1) + pad + 1
    keep = (hi >= lo) & (ymax >= row0) & (ymin < row1)
    idx = np.flatnonzero(keep)
    if idx.size == 0:
        return
    counts = (hi - lo + 1)[idx] * (2 * hm[idx] + 1)
    # split into chunks of at most `chunk` candidates
    cum = np.cumsum(counts)
    starts = [0]
    while starts[-1] < idx.size:
        base = cum[starts[-1] - 1] if starts[-1] > 0 else 0
        nxt = int(np.searchsorted(cum, base + chunk, side="right"))
        starts.append(max(nxt, starts[-1] + 1))
    starts[-1] = idx.size
    f32 = torch.float32
    for s0, s1 in zip(starts[:-1], starts[1:]):
        sel = idx[s0:s1]
        cnt = torch.as_tensor(counts[s0:s1], device=device)
        T = int(counts[s0:s1].sum())
        sid = torch.repeat_interleave(torch.arange(len(sel), device=device), cnt, output_size=T)
        off = torch.cumsum(cnt, 0) - cnt
        local = torch.arange(T, device=device) - off[sid]
        P = lambda arr, dt=f32: torch.as_tensor(arr[sel], device=device, dtype=dt)[sid]
        span = 2 * P(hm, torch.int64) + 1
        m = P(lo, torch.int64) + torch.div(local, span, rounding_mode="floor")
        k = local % span - P(hm, torch.int64)
        A0, A1, B0 = P(a0), P(a1), P(b0)
        mf = m.to(f32)
        mc = torch.minimum(torch.maximum(mf, torch.minimum(A0, A1)), torch.maximum(A0, A1))
        bc = torch.round(B0 + (mc - A0) * P(slope)).to(torch.int64)
        b = bc + k
        hz = P(horiz, torch.bool)
        xx = torch.where(hz, m, b); yy = torch.where(hz, b, m)
        X0, Y0, X1, Y1, Wd = P(x0), P(y0), P(x1), P(y1), P(w)
        dx, dy = X1 - X0, Y1 - Y0
        L2 = dx * dx + dy * dy
        px, py = xx.to(f32) - X0, yy.to(f32) - Y0
        t = torch.where(L2 > 0, (px * dx + py * dy) / torch.where(L2 > 0, L2, 1), 0)
        t = t.clamp(0, 1)
        ex, ey = px - t * dx, py - t * dy
        d = torch.sqrt(ex * ex + ey * ey)
        cov = (Wd * 0.5 + 0.5 - d).clamp(0, 1)
        lvl = torch.round(cov * (levels - 1)).to(torch.int32)
        ok = (lvl > 0) & (xx >= 0) & (xx < W) & (yy >= row0) & (yy < row1)
        lin = ((yy - row0) * W + xx)[ok]
        val = lvl[ok]
        if key is not None:
            val = P(np.asarray(key, np.int64), torch.int32)[ok] * levels + val
        out_flat.scatter_reduce_(0, lin, val, reduce="amax", include_self=True)


def _hatched_rect_segments(rx0, ry0, rx1, ry1, spacing, outline_w):
    """Outline (4 segments) and 45-degree hatch lines clipped to the box."""
    segs = [(rx0, ry0, rx1, ry0, outline_w), (rx1, ry0, rx1, ry1, outline_w),
            (rx1, ry1, rx0, ry1, outline_w), (rx0, ry1, rx0, ry0, outline_w)]
    # lines x - y = c, c from rx0 - ry1 to rx1 - ry0
    c = rx0 - ry1 + spacing
    while c < rx1 - ry0:
        # intersection with the box: x in [rx0, rx1], y = x - c in [ry0, ry1]
        xa = max(rx0, ry0 + c); xb = min(rx1, ry1 + c)
        if xb > xa:
            segs.append((xa, xa - c, xb, xb - c, 1.0))
        c += spacing
    return segs


def drawing(H, W, *, seed, n_segments, n_rects, levels, hatched, n_walls=0,
            seg_len=None, device="cpu", rows=None):
    """RGBA line drawing [H, W] as int32 holding the little-endian R,G,B,A
    bytes of each pixel (or rows [r0, r1) of it when ``rows`` is
    given: the same pixels the full picture has there).

    n_rects rectangles from the 8-colour palette: solid (hatched=False) or a
    1-2 px outline with 45-degree hatch lines every 8-24 px (hatched=True),
    anti-aliased in the palette colour.  Then n_segments black segments, width
    1-3: with seg_len=None their endpoints are uniform over the picture;
    otherwise n_walls of them are full-width / full-height wall lines 4-8 px
    wide and the rest start uniformly with a length uniform in seg_len, their
    angle snapped to 0/45/90/135 degrees 80% of the time.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    r0, r1 = (0, H) if rows is None else rows
    h = r1 - r0
    dev = torch.device(device)
    # ---- rectangles
    rw = rng.integers(16, max(17, min(W, 400)), size=n_rects) if hatched else \
        rng.integers(max(1, W // 32), max(2, W // 4), size=n_rects)
    rh = rng.integers(16, max(17, min(H, 400)), size=n_rects) if hatched else \
        rng.integers(max(1, H // 32), max(2, H // 4), size=n_rects)
    rx = rng.integers(0, max(1, W - 8), size=n_rects)
    ry = rng.integers(0, max(1, H - 8), size=n_rects)
    rcol = rng.integers(0, len(PALETTE), size=n_rects)
    rspace = rng.integers(8, 25, size=n_rects)
    rout = rng.integers(1, 3, size=n_rects).astype(np.float64)
    base_r = torch.full((h, W), 255, dtype=torch.int64, device=dev)
    base_g = base_r.clone(); base_b = base_r.clone()
    if not hatched:
        for i in range(n_rects):
            ya, yb = int(ry[i]), int(min(H, ry[i] + rh[i]))
            xa, xb = int(rx[i]), int(min(W, rx[i] + rw[i]))
            ya, yb = max(ya, r0) - r0, min(yb, r1) - r0
            if yb <= ya:
                continue
            cr, cg, cb = (int(v) for v in PALETTE[rcol[i]])
            base_r[ya:yb, xa:xb] = cr; base_g[ya:yb, xa:xb] = cg; base_b[ya:yb, xa:xb] = cb
    else:
        sx0, sy0, sx1, sy1, sw, sk = [], [], [], [], [], []
        for i in range(n_rects):
            bx0, by0 = float(rx[i]), float(ry[i])
            bx1 = float(min(W - 1, rx[i] + rw[i])); by1 = float(min(H - 1, ry[i] + rh[i]))
            for (a, b, c, d, ww) in _hatched_rect_segments(bx0, by0, bx1, by1, int(rspace[i]),
                                                           float(rout[i])):
                sx0.append(a); sy0.append(b); sx1.append(c); sy1.append(d); sw.append(ww)
                sk.append(i + 1)
        keyed = torch.zeros(h * W, dtype=torch.int32, device=dev)
        _raster_segments(sx0, sy0, sx1, sy1, sw, levels, H, W, r0, r1, dev, keyed, key=sk)
        keyed = keyed.view(h, W).to(torch.int64)
        lvl = keyed % levels
        rid = keyed // levels - 1
        hit = lvl > 0
        pal = torch.as_tensor(PALETTE, device=dev)[torch.as_tensor(rcol, device=dev)[rid.clamp(min=0)]]
        q = lvl.to(torch.float32) / (levels - 1)
        for ch, base in enumerate((base_r, base_g, base_b)):
            mixed = torch.round(255.0 * (1 - q) + pal[..., ch].to(torch.float32) * q).to(torch.int64)
            base.copy_(torch.where(hit, mixed, base))
    # ---- black segments
    if seg_len is None:
        x0 = rng.uniform(0, W - 1, n_segments); y0 = rng.uniform(0, H - 1, n_segments)
        x1 = rng.uniform(0, W - 1, n_segments); y1 = rng.uniform(0, H - 1, n_segments)
        sw = rng.integers(1, 4, n_segments).astype(np.float64)
    else:
        nw = min(n_walls, n_segments)
        ns = n_segments - nw
        horiz = np.arange(nw) % 2 == 0
        pos = np.where(horiz, rng.uniform(0, H - 1, nw), rng.uniform(0, W - 1, nw))
        wx0 = np.where(horiz, -8.0, pos); wx1 = np.where(horiz, W + 8.0, pos)
        wy0 = np.where(horiz, pos, -8.0); wy1 = np.where(horiz, pos, H + 8.0)
        ww = rng.integers(4, 9, nw).astype(np.float64)
        sx = rng.uniform(0, W - 1, ns); sy = rng.uniform(0, H - 1, ns)
        ang = rng.uniform(0, math.pi, ns)
        snap = rng.random(ns) < 0.8
        ang = np.where(snap, np.round(ang / (math.pi / 4)) * (math.pi / 4), ang)
        ln = rng.uniform(seg_len[0], seg_len[1], ns)
        ex = sx + ln * np.cos(ang); ey = sy + ln * np.sin(ang)
        x0 = np.concatenate([wx0, sx]); y0 = np.concatenate([wy0, sy])
        x1 = np.concatenate([wx1, ex]); y1 = np.concatenate([wy1, ey])
        sw = np.concatenate([ww, rng.integers(1, 4, ns).astype(np.float64)])
    lv = torch.zeros(h * W, dtype=torch.int32, device=dev)
    _raster_segments(x0, y0, x1, y1, sw, levels, H, W, r0, r1, dev, lv)
    q = lv.view(h, W).to(torch.float32) / (levels - 1)
    chans = [torch.round(b.to(torch.float32) * (1 - q)).to(torch.int64) for b in (base_r, base_g, base_b)]
    px = pack_rgba(*chans)
    # int32 tensor holding the RGBA bytes (the bit pattern of the uint32 pixel)
    return (px - torch.where(px >= (1 << 31), 1 << 32, 0)).to(torch.int32)


# ------------------------------------------------------------ binary inputs

def bernoulli_masks(B, H, W, ps, *, seed, device="cpu"):
    """uint8 [B, H, W] masks; image b has foreground probability
    ps[b * len(ps) // B]."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    u = torch.rand((B, H, W), generator=g)
    p = torch.as_tensor([ps[b * len(ps) // B] for b in range(B)], dtype=torch.float32)
    return (u < p[:, None, None]).to(torch.uint8).to(device)


def tissue_slide(H, W, *, seed, sigma=8.0, radius=32, percentile=0.55, device="cpu"):
    """uint8 [H, W]: white noise N(0,1), separable Gaussian blur (sigma,
    radius, reflect padding), foreground = value above the exact
    ceil(percentile*N)-th smallest value."""
    import torch.nn.functional as F
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn((H, W), generator=g, dtype=torch.float32).to(device)
    t = torch.arange(-radius, radius + 1, dtype=torch.float32, device=device)
    k = torch.exp(-0.5 * (t / sigma) ** 2)
    k = k / k.sum()
    y = x[None, None]
    y = F.conv2d(F.pad(y, (radius, radius, 0, 0), mode="reflect"), k.view(1, 1, 1, -1))
    y = F.conv2d(F.pad(y, (0, 0, radius, radius), mode="reflect"), k.view(1, 1, -1, 1))
    y = y[0, 0]
    N = H * W
    kth = int(math.ceil(percentile * N))
    thr = torch.sort(y.reshape(-1)).values[kth - 1]
    return (y > thr).to(torch.uint8)


def serpentine(H, W, device="cpu"):
    """uint8: even rows all 1; odd row r has a single 1 at column W-1 when
    r = 1 (mod 4) and at column 0 when r = 3 (mod 4): one 1-px-wide path of
    H/2*W + H/2 pixels."""
    img = torch.zeros((H, W), dtype=torch.uint8, device=device)
    img[0::2, :] = 1
    img[1::4, W - 1] = 1
    img[3::4, 0] = 1
    return img


def checkerboard(H, W, device="cpu"):
    r = torch.arange(H, device=device)[:, None]
    c = torch.arange(W, device=device)[None, :]
    return ((r + c) & 1).to(torch.uint8)


def random_levels(H, W, k, *, seed, device="cpu"):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randint(0, k, (H, W), generator=g, dtype=torch.uint8).to(device)


# ------------------------------------------------------------ named workloads

MODE_ALL, MODE_BINARY = 0, 1


def c0_drawing(device="cpu", rows=None):
    """1024 x 1024 RGBA drawing: 20 solid palette rectangles, 200 black
    segments with uniform endpoints, widths 1-3, 16 coverage levels."""
    return drawing(1024, 1024, seed=1000, n_segments=200, n_rects=20, levels=16,
                   hatched=False, device=device, rows=rows)


C4_H, C4_W = 24000, 33600


def c4_sheet(device="cpu", rows=None, H=C4_H, W=C4_W):
    """The construction-sheet analogue, 24000 rows x 33600 columns RGBA
    (33,600 x 24,000 = 806.4 Mpx, a 42 x 30 in sheet at 800 dpi): 5000 hatched
    palette rectangles; 400,000 black segments with 64 coverage levels, of which
    64 are full-width / full-height wall lines 4-8 px wide and the rest short
    strokes 16-80 px long.  Smaller H, W scale the counts by area."""
    scale = (H * W) / float(C4_H * C4_W)
    n_seg = max(8, int(round(400_000 * scale)))
    n_rect = max(2, int(round(5_000 * scale)))
    n_walls = max(2, int(round(64 * math.sqrt(scale))))
    return drawing(H, W, seed=4000, n_segments=n_seg, n_rects=n_rect, levels=64,
                   hatched=True, n_walls=n_walls, seg_len=(16.0, 80.0), device=device,
                   rows=rows)


def c1_masks(device="cpu"):
    """64 binary 1024 x 1024 masks, p = 0.2 / 0.4 / 0.6 / 0.8 (16 each)."""
    return bernoulli_masks(64, 1024, 1024, (0.2, 0.4, 0.6, 0.8), seed=1001, device=device)


def c2_slide(device="cpu", H=20000, W=20000):
    return tissue_slide(H, W, seed=1002, device=device)


def c3_structures(device="cpu", H=8192, W=8192):
    return {
        "serpentine": serpentine(H, W, device),
        "checkerboard": checkerboard(H, W, device),
        "random4": random_levels(H, W, 4, seed=1003, device=device),
    }


# name -> (connectivity, mode, pixel_bytes)
CONFIGS = {
    "c0_drawing_1024_rgba": (8, MODE_ALL, 4),
    "c1_masks_64x1024": (8, MODE_BINARY, 1),
    "c2_slide_20000": (4, MODE_BINARY, 1),
    "c3_structures_8192": (None, None, 1),      # every structure x {4,8} x {all,binary}
    "c4_sheet_24000x33600_rgba": (8, MODE_ALL, 4),
}


def c4_sheet_rgb(device="cpu", H=C4_H, W=C4_W):
    """The construction sheet as packed 24-bit RGB, uint8 [1, H, W, 3] (2.4 GB
    at full size): the RGBA sheet without its alpha byte, which is 255
    everywhere, so its regions are the RGBA sheet's."""
    rgba = c4_sheet(device=device, H=H, W=W)
    return rgba.view(torch.uint8).reshape(H, W, 4)[:, :, :3].contiguous().reshape(1, H, W, 3)
