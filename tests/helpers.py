"""Test-side helpers that are independent of both the oracle and the CUDA path.

* ``read_golden``      -- parse a fixture under tests/golden/.
* ``canonicalize``     -- renumber any partition 1..n by first pixel in raster
                          order (background 0 stays 0).
* ``closure_labels``   -- brute-force labelling of tiny images by transitive
                          closure of the neighbour relation (no union-find, no
                          flood fill): the pin the oracle is checked against.
* ``scipy_labels``     -- the same partition through scipy.ndimage.label, one
                          call per distinct value (the library routine the
                          binary case reduces to).
* ``check_invariants`` -- O(N) properties every correct labelling has.
"""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name):
    """Returns dict(image=int array, labels=int32 array, n=int,
    connectivity=int, mode='all'|'binary')."""
    out = {}
    section = None
    rows = {"image": [], "labels": []}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.endswith(":") and line[:-1] in rows:
                section = line[:-1]
                continue
            if ":" in line:
                k, v = [s.strip() for s in line.split(":", 1)]
                out[k] = v
                section = None
                continue
            rows[section].append([int(t) for t in line.split()])
    return dict(image=np.array(rows["image"]),
                labels=np.array(rows["labels"], dtype=np.int32),
                n=int(out["n"]), connectivity=int(out["connectivity"]),
                mode=out["mode"])


def canonicalize(lab, background=None):
    """Renumber a labelling so that regions get 1..n in the raster order of
    their first pixel.  ``background``: boolean mask of pixels that keep 0."""
    lab = np.asarray(lab)
    flat = lab.reshape(-1)
    out = np.zeros(flat.shape, dtype=np.int64)
    keep = np.ones(flat.shape, bool) if background is None else ~np.asarray(background).reshape(-1)
    vals = flat[keep]
    uniq, first = np.unique(vals, return_index=True)
    order = np.argsort(first, kind="stable")
    rank = np.empty(len(uniq), np.int64)
    rank[order] = np.arange(1, len(uniq) + 1)
    out[keep] = rank[np.searchsorted(uniq, vals)]
    return out.reshape(lab.shape), len(uniq)


def _neighbour_offsets(conn):
    if conn == 4:
        return [(-1, 0), (0, -1), (0, 1), (1, 0)]
    return [(dr, dc) for dr in (-1, 0, 1) for dc in (-1, 0, 1) if (dr, dc) != (0, 0)]


def closure_labels(imgs, conn, binary, ignore=None):
    """Brute force for a batch of tiny images [B,H,W] (H*W <= 64).

    Builds the adjacency matrix of the pixel graph (neighbours of equal value,
    neither ignored in binary mode), takes its reflexive-transitive closure by
    repeated boolean squaring, represents each pixel by the smallest pixel it
    reaches and numbers those representatives in raster order.
    Returns (labels [B,H,W] int64, n [B])."""
    imgs = np.asarray(imgs)
    B, H, W = imgs.shape
    N = H * W
    flat = imgs.reshape(B, N)
    if binary:
        ignore = 0
    active = (flat != ignore) if ignore is not None else np.ones_like(flat, dtype=bool)
    A = np.zeros((B, N, N), dtype=np.float32)
    idx = np.arange(N)
    A[:, idx, idx] = active
    for r in range(H):
        for c in range(W):
            p = r * W + c
            for dr, dc in _neighbour_offsets(conn):
                rr, cc = r + dr, c + dc
                if 0 <= rr < H and 0 <= cc < W:
                    q = rr * W + cc
                    A[:, p, q] = (flat[:, p] == flat[:, q]) & active[:, p] & active[:, q]
    R = A
    steps = 1
    while steps < N:
        R = np.minimum(np.matmul(R, R), 1.0)
        steps *= 2
    reach = R > 0
    # smallest reachable pixel (first pixel of the region in raster order)
    rep = np.where(reach.any(axis=2), reach.argmax(axis=2), -1)
    is_first = (rep == idx[None, :]) & active
    cum = np.cumsum(is_first, axis=1)
    lab = np.where(active, np.take_along_axis(cum, np.maximum(rep, 0), axis=1), 0)
    return lab.reshape(B, H, W), is_first.sum(axis=1)


def scipy_labels(img, conn, binary, ignore=None):
    """Partition via scipy.ndimage.label run once per distinct value,
    then renumbered canonically.  Returns (labels, n)."""
    from scipy import ndimage
    img = np.asarray(img)
    structure = ndimage.generate_binary_structure(2, 1 if conn == 4 else 2)
    out = np.zeros(img.shape, dtype=np.int64)
    nxt = 0
    if binary:
        ignore = 0
    for v in np.unique(img):
        if ignore is not None and v == ignore:
            continue
        lab, k = ndimage.label(img == v, structure=structure)
        m = lab > 0
        out[m] = lab[m] + nxt
        nxt += k
    bg = (img == ignore) if ignore is not None else None
    return canonicalize(out, bg)


def check_invariants(img, lab, n, conn, binary):
    """O(N) checks of a labelling of one image (numpy arrays H x W):
    (i) labels are 0..n, 0 exactly on background, and each label's first
        pixel comes after the previous label's first pixel (canonical order);
    (ii) every pair of equal-valued (non-background) neighbours has equal
        labels;
    (iii) every label is value-homogeneous.
    Returns a list of failure strings (empty when all hold)."""
    fails = []
    img = np.asarray(img)
    lab = np.asarray(lab).astype(np.int64)
    H, W = img.shape
    bg = (img == 0) if binary else np.zeros(img.shape, bool)
    if (lab[bg] != 0).any():
        fails.append("background pixel with a non-zero label")
    if (lab[~bg] <= 0).any():
        fails.append("foreground pixel with label <= 0")
    if lab.max(initial=0) != n:
        fails.append("max label %d != n %d" % (lab.max(initial=0), n))
    flat = lab.reshape(-1)
    fg = flat[flat > 0]
    if fg.size:
        uniq, first = np.unique(fg, return_index=True)
        if len(uniq) != n or uniq[0] != 1 or uniq[-1] != n:
            fails.append("labels are not exactly 1..n")
        pos = np.flatnonzero(flat > 0)[first]
        if (np.diff(pos) <= 0).any():
            fails.append("first pixels not in increasing raster order")
    elif n != 0:
        fails.append("no foreground but n != 0")
    offs = [(0, 1), (1, 0)] + ([(1, 1), (1, -1)] if conn == 8 else [])
    for dr, dc in offs:
        r0, r1 = 0, H - dr
        c0, c1 = max(0, -dc), W - max(0, dc)
        a = img[r0:r1, c0:c1]
        b = img[r0 + dr:r1 + dr, c0 + dc:c1 + dc]
        la = lab[r0:r1, c0:c1]
        lb = lab[r0 + dr:r1 + dr, c0 + dc:c1 + dc]
        eq = (a == b) & ~bg[r0:r1, c0:c1]
        if (la[eq] != lb[eq]).any():
            fails.append("equal neighbours (%d,%d) with different labels" % (dr, dc))
    if fg.size:
        fv = img.reshape(-1)[flat > 0]
        order = np.argsort(fg, kind="stable")
        sl, sv = fg[order], fv[order]
        same = sl[1:] == sl[:-1]
        if (sv[1:][same] != sv[:-1][same]).any():
            fails.append("a label covers two values")
    return fails
