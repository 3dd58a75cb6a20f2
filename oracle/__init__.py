"""The oracle: a plain single-threaded CPU labeller (breadth-first flood fill).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  It shares no code with
the CUDA library and the CUDA library never calls it.

What it computes (the plain definition; see ``ccl_oracle.c`` for citations):
two pixels share a label exactly when a path of 4- or 8-neighbours of exactly
equal value joins them ("every-colour", ch. 01-02); regions are numbered
1..n in the raster order of their first pixel ("every-colour", ch. 04 and
ch. 11); in binary mode value 0 is background and keeps label 0
("every-colour", ch. 08 switch 4; bendabir.com, "The basic approach").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ccl_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libccl_oracle.so")

MODE_ALL = 0
MODE_BINARY = 1

# one region's statistics, the layout of the oracle's C struct (40 bytes)
STAT_DTYPE = np.dtype([("area", np.int32), ("y_min", np.int32), ("x_min", np.int32),
                       ("y_max", np.int32), ("x_max", np.int32), ("first", np.int32),
                       ("sum_y", np.int64), ("sum_x", np.int64)])
assert STAT_DTYPE.itemsize == 40

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler; returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-shared", "-fPIC",
                           "-o", tmp, _SRC])
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_label.restype = ctypes.c_int
            lib.oracle_label.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_label_ignore.restype = ctypes.c_int
            lib.oracle_label_ignore.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_region_stats.restype = ctypes.c_int
            lib.oracle_region_stats.argtypes = [
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
            _lib = lib
    return _lib


def _shape(a):
    if a.dtype == np.uint8 and a.ndim == 4:      # [B,H,W,pixel_bytes]
        B, H, W, pb = a.shape
        return B, H, W, pb, False
    if a.ndim == 3:
        B, H, W = a.shape
        return B, H, W, a.dtype.itemsize, False
    if a.ndim == 2:
        H, W = a.shape
        return 1, H, W, a.dtype.itemsize, True
    raise ValueError("expected a [B,]H,W array")


def label_ignore(img: np.ndarray, ignore_value: int, connectivity: int = 8):
    """Like ``label`` in the all-pixels mode, but pixels equal to
    ``ignore_value`` (an integer holding the pixel's bytes, little-endian)
    are background: label 0, joining nothing ("every-colour", ch. 08
    switch 4)."""
    a = np.ascontiguousarray(img)
    B, H, W, pb, squeeze = _shape(a)
    ign = np.frombuffer(int(ignore_value).to_bytes(8, "little")[:pb], dtype=np.uint8).copy()
    labels = np.empty((B, H, W), dtype=np.int32)
    n = np.empty((B,), dtype=np.int32)
    rc = _load().oracle_label_ignore(a.ctypes.data, B, H, W, pb, connectivity, ign.ctypes.data,
                                     labels.ctypes.data, n.ctypes.data)
    if rc != 0:
        raise RuntimeError("oracle_label_ignore failed with status %d" % rc)
    if squeeze:
        return labels[0], n[0]
    return labels, n


def label(img: np.ndarray, connectivity: int = 8, mode: int = MODE_ALL):
    """Label a [B,]H,W image array (uint8 or uint32 pixels, or a trailing
    byte axis for wider pixels).

    Returns ``(labels int32 same leading shape, n_regions int32[B])``; for a
    2-D input the batch axis is dropped from both.
    """
    a = np.ascontiguousarray(img)
    squeeze = False
    if a.dtype == np.uint8 and a.ndim == 4:      # [B,H,W,pixel_bytes]
        B, H, W, pb = a.shape
    elif a.ndim == 3:
        B, H, W = a.shape
        pb = a.dtype.itemsize
    elif a.ndim == 2:
        H, W = a.shape
        B, pb = 1, a.dtype.itemsize
        squeeze = True
    else:
        raise ValueError("expected a [B,]H,W array")
    labels = np.empty((B, H, W), dtype=np.int32)
    n = np.empty((B,), dtype=np.int32)
    rc = _load().oracle_label(a.ctypes.data, B, H, W, pb, connectivity, mode,
                              labels.ctypes.data, n.ctypes.data)
    if rc != 0:
        raise RuntimeError("oracle_label failed with status %d" % rc)
    if squeeze:
        return labels[0], n[0]
    return labels, n


def region_stats(labels: np.ndarray, n_regions):
    """Statistics of every labelled region (see ``oracle_region_stats`` in
    ``ccl_oracle.c`` for the definitions and citations): a structured array
    of ``STAT_DTYPE`` with one entry per region, image by image, label 1 first.
    ``labels`` is [B,]H,W int32, ``n_regions`` the region count per image."""
    lab = np.ascontiguousarray(labels, dtype=np.int32)
    if lab.ndim == 2:
        lab = lab[None]
    B, H, W = lab.shape
    n = np.ascontiguousarray(np.asarray(n_regions, dtype=np.int32).reshape(-1))
    if n.shape[0] != B:
        raise ValueError("one region count per image")
    total = int(n.astype(np.int64).sum())
    out = np.empty(max(total, 1), dtype=STAT_DTYPE)
    rc = _load().oracle_region_stats(lab.ctypes.data, B, H, W, n.ctypes.data, out.ctypes.data, total)
    if rc != 0:
        raise RuntimeError("oracle_region_stats failed with status %d" % rc)
    return out[:total]
