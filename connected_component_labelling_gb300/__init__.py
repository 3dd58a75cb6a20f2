"""GB300 connected-component labelling: thin Python binding over libccl.so.

Every step of the labelling runs in the CUDA kernels of ``csrc/ccl.cu``; this
module only marshals arguments to the C ABI declared in ``include/ccl.h``.
PyTorch is used for device memory and the current stream.  There is no CPU
path: if the compiled library is missing, every call raises.

Names follow the C ABI (``ccl_label``, ``ccl_label_ws``, ``ccl_label_host``,
``ccl_workspace_bytes``, ``ccl_last_status``, ``ccl_status_string``,
``ccl_set_option``); ``label`` is the tensor-level convenience wrapper.
"""
from __future__ import annotations

import ctypes
import os
import threading

from ._build import COUNTERS_LIB_PATH, LIB_PATH, build  # noqa: F401

CCL_OK = 0
CCL_ERR_INVALID_ARG = 1
CCL_ERR_TOO_LARGE = 2
CCL_ERR_CUDA = 3
CCL_ERR_NO_MEMORY = 4
CCL_ERR_DEVICE_LIMIT = 5
CCL_MODE_ALL = 0
CCL_MODE_BINARY = 1
CCL_OPT_WALK_CAP = 1
CCL_OPT_STAGE_EVENTS = 2

# every symbol include/ccl.h declares
EXPORTED = ("ccl_label", "ccl_workspace_bytes", "ccl_label_ws", "ccl_label_host",
            "ccl_last_status", "ccl_status_string", "ccl_set_option", "ccl_stage_times",
            "ccl_stage_name", "ccl_kernel_launches", "ccl_label_noalloc", "ccl_label_ignore",
            "ccl_region_stats_workspace_bytes", "ccl_region_stats", "ccl_debug_counters",
            "ccl_version")

# event counters of the counters build (include/ccl.h, CCL_CNT_*)
COUNTER_NAMES = ("tile_walks", "tile_steps", "tile_links", "global_walks", "global_steps",
                 "global_links", "seam_pairs", "resolve_steps")

# one region's statistics (struct ccl_region_stat, 40 bytes): six int32 then two int64
STAT_BYTES = 40
STAT_FIELDS_I32 = ("area", "y_min", "x_min", "y_max", "x_max", "first")
STAT_FIELDS_I64 = ("sum_y", "sum_x")

_lock = threading.Lock()
_lib = None


class CCLError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__("%s%s" % (what + ": " if what else "", ccl_status_string(status)))


def _declare(L):
    """Argument and result types of every entry point of a loaded library."""
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.ccl_label.argtypes = [vp, i32, i32, i32, i32, i32, i32, vp, vp, vp]
    L.ccl_label.restype = i32
    L.ccl_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    L.ccl_workspace_bytes.restype = sz
    L.ccl_label_ws.argtypes = [vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, sz, vp]
    L.ccl_label_ws.restype = i32
    L.ccl_label_host.argtypes = [vp, i32, i32, i32, i32, i32, i32, vp, vp, vp]
    L.ccl_label_host.restype = i32
    L.ccl_last_status.argtypes = [vp]
    L.ccl_last_status.restype = i32
    L.ccl_status_string.argtypes = [i32]
    L.ccl_status_string.restype = ctypes.c_char_p
    L.ccl_set_option.argtypes = [i32, ctypes.c_longlong]
    L.ccl_set_option.restype = i32
    L.ccl_stage_times.argtypes = [vp, i32, vp]
    L.ccl_stage_times.restype = i32
    L.ccl_stage_name.argtypes = [i32]
    L.ccl_stage_name.restype = ctypes.c_char_p
    L.ccl_kernel_launches.argtypes = []
    L.ccl_kernel_launches.restype = ctypes.c_longlong
    L.ccl_label_noalloc.argtypes = [vp, i32, i32, i32, i32, i32, i32, vp, vp, vp]
    L.ccl_label_noalloc.restype = i32
    L.ccl_label_ignore.argtypes = [vp, i32, i32, i32, i32, i32, ctypes.c_uint32, vp, vp,
                                   vp, sz, vp]
    L.ccl_label_ignore.restype = i32
    L.ccl_region_stats_workspace_bytes.argtypes = [i32]
    L.ccl_region_stats_workspace_bytes.restype = sz
    L.ccl_region_stats.argtypes = [vp, i32, i32, i32, vp, vp, ctypes.c_int64, vp, sz, vp]
    L.ccl_region_stats.restype = i32
    L.ccl_version.argtypes = []
    L.ccl_version.restype = i32
    L.ccl_debug_counters.argtypes = [vp, i32, i32]
    L.ccl_debug_counters.restype = i32
    return L


def lib():
    """The loaded libccl.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libccl.so is not built (%s); run "
                                   "connected_component_labelling_gb300.build()" % LIB_PATH)
            L = _declare(ctypes.CDLL(LIB_PATH))
            _lib = L
    return _lib


# ------------------------------------------------------------ raw C-ABI calls

def ccl_label(img, batch, H, W, pixel_bytes, connectivity, mode, labels, n_regions, stream):
    return lib().ccl_label(img, batch, H, W, pixel_bytes, connectivity, mode, labels,
                           n_regions, stream)


def ccl_workspace_bytes(batch, H, W, pixel_bytes, connectivity, mode):
    return lib().ccl_workspace_bytes(batch, H, W, pixel_bytes, connectivity, mode)


def ccl_label_ws(img, batch, H, W, pixel_bytes, connectivity, mode, labels, n_regions,
                 workspace, workspace_bytes, stream):
    return lib().ccl_label_ws(img, batch, H, W, pixel_bytes, connectivity, mode, labels,
                              n_regions, workspace, workspace_bytes, stream)


def ccl_label_host(img, batch, H, W, pixel_bytes, connectivity, mode, labels, n_regions,
                   stream):
    return lib().ccl_label_host(img, batch, H, W, pixel_bytes, connectivity, mode, labels,
                                n_regions, stream)


def ccl_last_status(stream=None):
    return lib().ccl_last_status(stream)


def ccl_status_string(status):
    return lib().ccl_status_string(int(status)).decode()


def ccl_set_option(option, value):
    return lib().ccl_set_option(option, value)


def ccl_stage_times(max_stages=8):
    """Returns (list of summed ms per stage, number of calls recorded)."""
    arr = (ctypes.c_double * max_stages)()
    n = ctypes.c_int(0)
    k = lib().ccl_stage_times(arr, max_stages, ctypes.byref(n))
    if k < 0:
        raise CCLError(-k, "ccl_stage_times")
    return [arr[i] for i in range(min(k, max_stages))], n.value


def ccl_stage_name(stage):
    return lib().ccl_stage_name(stage).decode()


def ccl_kernel_launches():
    return lib().ccl_kernel_launches()


def ccl_label_noalloc(img, batch, H, W, pixel_bytes, connectivity, mode, labels, n_regions,
                      stream):
    """ccl_label without any device allocation (scratch in a fixed array of
    CCL_NOALLOC_SCRATCH_BYTES inside the library); for callers that may not
    allocate device memory.  Calls on one device must not overlap."""
    return lib().ccl_label_noalloc(img, batch, H, W, pixel_bytes, connectivity, mode, labels,
                                   n_regions, stream)


CCL_NOALLOC_SCRATCH_BYTES = 32 << 20


def ccl_label_ignore(img, batch, H, W, pixel_bytes, connectivity, ignore_value, labels,
                     n_regions, workspace, workspace_bytes, stream):
    return lib().ccl_label_ignore(img, batch, H, W, pixel_bytes, connectivity, ignore_value,
                                  labels, n_regions, workspace, workspace_bytes, stream)


def label_ignore(img, ignore_value, connectivity=8, out=None, n_out=None, workspace=None,
                 stream=None):
    """Label a CUDA tensor of images with pixels equal to ``ignore_value``
    (the pixel's bytes as a little-endian integer) as background: label 0,
    joining nothing.  Returns (labels, n_regions) like ``label``."""
    import torch
    if not img.is_cuda:
        raise ValueError("label_ignore() needs a CUDA tensor; the library has no CPU path")
    img = img.contiguous()
    B, H, W, pb, squeeze = image_geometry(img)
    if out is None:
        out = torch.empty((B, H, W), dtype=torch.int32, device=img.device)
    _check_tensor(out, "out", torch.int32, B * H * W, img.device)
    if n_out is None:
        n_out = torch.empty((B,), dtype=torch.int32, device=img.device)
    _check_tensor(n_out, "n_out", torch.int32, B, img.device)
    wp, wb = _workspace_arg(workspace, img.device)
    st = stream if stream is not None else torch.cuda.current_stream(img.device)
    with torch.cuda.device(img.device):
        rc = ccl_label_ignore(img.data_ptr(), B, H, W, pb, connectivity,
                              int(ignore_value) & 0xFFFFFFFF, out.data_ptr(), n_out.data_ptr(),
                              wp, wb, st.cuda_stream)
    if rc != CCL_OK:
        raise CCLError(rc, "ccl_label_ignore")
    if squeeze:
        return out.view(H, W), n_out.view(())
    return out, n_out


def ccl_region_stats_workspace_bytes(batch):
    return lib().ccl_region_stats_workspace_bytes(batch)


def ccl_region_stats(labels, batch, H, W, n_regions, stats, capacity, workspace, workspace_bytes,
                     stream):
    return lib().ccl_region_stats(labels, batch, H, W, n_regions, stats, capacity, workspace,
                                  workspace_bytes, stream)


def region_stats(labels, n_regions, capacity=None, workspace=None, stream=None):
    """Statistics of every region of a label tensor from ``label`` /
    ``label_ignore`` (``n_regions``: their region counts, on the device).
    Returns ``(raw, fields)``: ``raw`` the uint8 tensor of ``capacity``
    40-byte entries (image by image, label 1 first), ``fields`` a dict of
    views into it -- int32 ``area``, ``y_min``, ``x_min``, ``y_max``,
    ``x_max``, ``first`` and int64 ``sum_y``, ``sum_x``.  ``capacity``
    defaults to the total number of regions (read from the device, which
    synchronises).  Device-side findings are reported by ``check_status``."""
    import torch
    if not labels.is_cuda:
        raise ValueError("region_stats() needs CUDA tensors; the library has no CPU path")
    if labels.dtype != torch.int32:
        raise ValueError("labels must be int32, not %s" % labels.dtype)
    labels = labels.contiguous()
    if labels.dim() == 2:
        B, (H, W) = 1, labels.shape
    elif labels.dim() == 3:
        B, H, W = labels.shape
    else:
        raise ValueError("expected [B,]H,W labels")
    if not isinstance(n_regions, torch.Tensor) or n_regions.device != labels.device:
        raise ValueError("n_regions must be a tensor on the labels' device")
    n = n_regions.reshape(-1).to(torch.int32).contiguous()
    if n.numel() != B:
        raise ValueError("n_regions holds %d counts for %d images" % (n.numel(), B))
    if capacity is None:
        capacity = int(n.to(torch.int64).sum().item())
    if capacity < 0:
        raise ValueError("capacity must be >= 0")
    raw = torch.empty((max(capacity, 1) * STAT_BYTES,), dtype=torch.uint8, device=labels.device)
    st = stream if stream is not None else torch.cuda.current_stream(labels.device)
    wp, wb = _workspace_arg(workspace, labels.device)
    with torch.cuda.device(labels.device):
        rc = ccl_region_stats(labels.data_ptr(), B, H, W, n.data_ptr(), raw.data_ptr(), capacity,
                              wp, wb, st.cuda_stream)
    if rc != CCL_OK:
        raise CCLError(rc, "ccl_region_stats")
    raw = raw[:capacity * STAT_BYTES]
    i32 = raw.view(torch.int32).view(capacity, STAT_BYTES // 4)
    i64 = raw.view(torch.int64).view(capacity, STAT_BYTES // 8)
    fields = {f: i32[:, k] for k, f in enumerate(STAT_FIELDS_I32)}
    fields.update({f: i64[:, 3 + k] for k, f in enumerate(STAT_FIELDS_I64)})
    return raw, fields


def ccl_debug_counters(out, n, reset):
    return lib().ccl_debug_counters(out, n, reset)


def counters_library():
    """The counters build of the library (built on first use): a separate
    libccl_counters.so with event counters compiled in, for measuring the
    method (bench.py --counters).  Same entry points as ``lib()``."""
    return _declare(ctypes.CDLL(build(counters=True)))


def read_counters(L, reset=True):
    """The event counters of library ``L`` as a dict (COUNTER_NAMES)."""
    buf = (ctypes.c_ulonglong * len(COUNTER_NAMES))()
    rc = L.ccl_debug_counters(buf, len(COUNTER_NAMES), 1 if reset else 0)
    if rc != CCL_OK:
        raise CCLError(rc, "ccl_debug_counters")
    return dict(zip(COUNTER_NAMES, (int(v) for v in buf)))


def ccl_version():
    return lib().ccl_version()


# ------------------------------------------------------------ tensor wrapper

_MODES = {"all": CCL_MODE_ALL, "binary": CCL_MODE_BINARY,
          CCL_MODE_ALL: CCL_MODE_ALL, CCL_MODE_BINARY: CCL_MODE_BINARY}


def _check_tensor(t, name, dtype, numel, device):
    """Caller-supplied buffers go to the kernels as raw pointers: each must be a
    contiguous tensor of the expected dtype and size on the image's device."""
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.device != device:
        raise ValueError("%s is on %s, the input on %s" % (name, t.device, device))
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, not %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if numel is not None and t.numel() != numel:
        raise ValueError("%s holds %d elements, %d expected" % (name, t.numel(), numel))


def _workspace_arg(workspace, device):
    """(pointer, bytes) of an optional caller workspace on ``device``."""
    if workspace is None:
        return None, 0
    _check_tensor(workspace, "workspace", None, None, device)
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def image_geometry(img):
    """(batch, H, W, pixel_bytes, squeeze) of a [B,]H,W tensor of 1/2/4-byte
    pixels, or a [B,]H,W,C uint8 tensor whose C (2, 3 or 4) bytes form one
    pixel (C = 3: packed 24-bit RGB)."""
    import torch
    if img.dtype == torch.uint8 and img.dim() == 4 and img.shape[-1] in (2, 3, 4):
        B, H, W, pb = img.shape
        return B, H, W, pb, False
    pb = img.element_size()
    if img.dim() == 3:
        B, H, W = img.shape
        return B, H, W, pb, False
    if img.dim() == 2:
        H, W = img.shape
        return 1, H, W, pb, True
    raise ValueError("expected a [B,]H,W tensor")


def label(img, connectivity=8, mode="all", out=None, n_out=None, workspace=None, stream=None):
    """Label a CUDA tensor of images.  Returns (labels int32 tensor shaped like
    the pixel grid, n_regions int32 tensor [B] (0-d for a 2-D input)).
    Asynchronous on ``stream`` (default: torch's current stream)."""
    import torch
    if not img.is_cuda:
        raise ValueError("label() needs a CUDA tensor; the library has no CPU path")
    img = img.contiguous()
    B, H, W, pb, squeeze = image_geometry(img)
    m = _MODES[mode]
    if out is None:
        out = torch.empty((B, H, W), dtype=torch.int32, device=img.device)
    _check_tensor(out, "out", torch.int32, B * H * W, img.device)
    if n_out is None:
        n_out = torch.empty((B,), dtype=torch.int32, device=img.device)
    _check_tensor(n_out, "n_out", torch.int32, B, img.device)
    wp, wb = _workspace_arg(workspace, img.device)
    st = stream if stream is not None else torch.cuda.current_stream(img.device)
    sp = st.cuda_stream
    with torch.cuda.device(img.device):
        if workspace is None:
            rc = ccl_label(img.data_ptr(), B, H, W, pb, connectivity, m, out.data_ptr(),
                           n_out.data_ptr(), sp)
        else:
            rc = ccl_label_ws(img.data_ptr(), B, H, W, pb, connectivity, m, out.data_ptr(),
                              n_out.data_ptr(), wp, wb, sp)
    if rc != CCL_OK:
        raise CCLError(rc, "ccl_label")
    if squeeze:
        return out.view(H, W), n_out.view(())
    return out, n_out


def check_status(stream=None):
    """Synchronise ``stream`` and raise if a device-side limit tripped."""
    import torch
    st = stream if stream is not None else torch.cuda.current_stream()
    rc = ccl_last_status(st.cuda_stream)
    if rc != CCL_OK:
        raise CCLError(rc, "device status")
