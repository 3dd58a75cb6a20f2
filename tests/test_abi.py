"""CPU-only checks of the C ABI: the library builds, loads, exports every
symbol include/ccl.h declares, and rejects bad arguments on the host before
touching any device."""
import ctypes
import os
import re

import pytest

import connected_component_labelling_gb300 as ccl

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "ccl.h")


@pytest.fixture(scope="module")
def lib():
    ccl.build()
    return ccl.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(ccl_\w+)\s*\(", text, re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("ccl_label", "ccl_label_ws", "ccl_workspace_bytes", "ccl_label_host",
              "ccl_last_status", "ccl_status_string", "ccl_set_option", "ccl_stage_times",
              "ccl_stage_name", "ccl_kernel_launches", "ccl_label_noalloc", "ccl_label_ignore",
              "ccl_version"):
        assert n in names
    assert sorted(ccl.EXPORTED) == names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # dynamic symbol table, checked through dlsym
    handle = ctypes.CDLL(ccl.LIB_PATH)
    for name in declared_functions():
        assert ctypes.cast(getattr(handle, name), ctypes.c_void_p).value


def test_status_strings_and_version(lib):
    assert ccl.ccl_status_string(ccl.CCL_OK) == "CCL_OK"
    assert ccl.ccl_status_string(ccl.CCL_ERR_DEVICE_LIMIT) == "CCL_ERR_DEVICE_LIMIT"
    assert ccl.ccl_status_string(99) == "CCL_ERR_UNKNOWN"
    assert ccl.ccl_version() >= 100


def test_workspace_bytes(lib):
    assert ccl.ccl_workspace_bytes(0, 10, 10, 1, 8, 0) == 0
    assert ccl.ccl_workspace_bytes(1, 10, 10, 5, 8, 0) == 0       # bad pixel_bytes
    assert ccl.ccl_workspace_bytes(1, 10, 10, 3, 8, 0) > 0        # 24-bit RGB
    assert ccl.ccl_workspace_bytes(1, 10, 10, 1, 6, 0) == 0       # bad connectivity
    assert ccl.ccl_workspace_bytes(1, 1 << 16, 1 << 15, 1, 8, 0) > 0    # H*W = 2^31 is accepted
    assert ccl.ccl_workspace_bytes(1, 1 << 16, 1 << 16, 1, 8, 0) == 0   # H*W = 2^32 is not
    a = ccl.ccl_workspace_bytes(1, 1024, 1024, 4, 8, 0)
    b = ccl.ccl_workspace_bytes(2, 1024, 1024, 4, 8, 0)
    assert 0 < a < b
    # run start bits (1 bit/px) + per 256 x 16 tile: run bases, a leader per run
    # (4096 x 2 B), leader bits, border records, slot parents (540 x 8 B) ...
    px = 1024 * 1024
    assert 3.5 * px <= a < 4.5 * px
    # the ignoring modes add foreground bits (1 bit/px)
    assert ccl.ccl_workspace_bytes(1, 1024, 1024, 4, 8, 1) == a + px // 8
    assert a % 256 == 0


FAKE = 1 << 20   # a host address never dereferenced: validation fails first


@pytest.mark.parametrize("args,expect", [
    ((FAKE, 1, 8, 8, 5, 8, 0), ccl.CCL_ERR_INVALID_ARG),     # pixel_bytes
    ((FAKE, 1, 8, 8, 0, 8, 0), ccl.CCL_ERR_INVALID_ARG),     # pixel_bytes
    ((FAKE, 1, 8, 8, 1, 6, 0), ccl.CCL_ERR_INVALID_ARG),     # connectivity
    ((FAKE, 1, 8, 8, 1, 8, 2), ccl.CCL_ERR_INVALID_ARG),     # mode
    ((FAKE, -1, 8, 8, 1, 8, 0), ccl.CCL_ERR_INVALID_ARG),    # batch
    ((FAKE, 1, -8, 8, 1, 8, 0), ccl.CCL_ERR_INVALID_ARG),    # H
    ((None, 1, 8, 8, 1, 8, 0), ccl.CCL_ERR_INVALID_ARG),     # null image
    ((FAKE + 1, 1, 8, 8, 4, 8, 0), ccl.CCL_ERR_INVALID_ARG), # misaligned RGBA
    ((FAKE, 1, 1 << 16, 1 << 16, 1, 8, 0), ccl.CCL_ERR_TOO_LARGE),   # H*W = 2^32
])
def test_invalid_arguments_rejected_on_host(lib, args, expect):
    img, B, H, W, pb, conn, mode = args
    labels = FAKE * 64
    assert ccl.ccl_label(img, B, H, W, pb, conn, mode, labels, None, None) == expect
    assert ccl.ccl_label_ws(img, B, H, W, pb, conn, mode, labels, None, FAKE * 128, 1 << 20,
                            None) == expect


def test_ignore_value_must_fit_the_pixel(lib):
    labels = FAKE * 64
    assert ccl.ccl_label_ignore(FAKE, 1, 8, 8, 1, 8, 0x100, labels, None, None, 0, None) == \
        ccl.CCL_ERR_INVALID_ARG
    assert ccl.ccl_label_ignore(FAKE, 1, 8, 8, 2, 8, 0x10000, labels, None, None, 0, None) == \
        ccl.CCL_ERR_INVALID_ARG
    assert ccl.ccl_label_ignore(FAKE, 1, 8, 8, 3, 8, 0x1000000, labels, None, None, 0, None) == \
        ccl.CCL_ERR_INVALID_ARG
    assert ccl.ccl_label_ignore(FAKE, 1, 8, 8, 1, 6, 0, labels, None, None, 0, None) == \
        ccl.CCL_ERR_INVALID_ARG
    assert ccl.ccl_label_ignore(FAKE, 1, 8, 8, 1, 8, 0, labels, None, FAKE * 128 + 8, 1 << 20,
                                None) == ccl.CCL_ERR_INVALID_ARG


def test_null_labels_and_overlap_rejected(lib):
    assert ccl.ccl_label(FAKE, 1, 8, 8, 1, 8, 0, None, None, None) == ccl.CCL_ERR_INVALID_ARG
    # labels overlapping the image
    assert ccl.ccl_label(FAKE, 1, 8, 8, 4, 8, 0, FAKE + 64, None, None) == ccl.CCL_ERR_INVALID_ARG
    # counts overlapping the labels (the counts are written before the labels)
    labels = FAKE * 64
    assert ccl.ccl_label(FAKE, 2, 8, 8, 1, 8, 0, labels, labels + 4 * 127, None) == \
        ccl.CCL_ERR_INVALID_ARG
    assert ccl.ccl_label_noalloc(FAKE, 2, 8, 8, 1, 8, 0, labels, labels, None) == \
        ccl.CCL_ERR_INVALID_ARG


def test_workspace_checks_on_host(lib):
    need = ccl.ccl_workspace_bytes(1, 64, 64, 1, 8, 0)
    need_ign = ccl.ccl_workspace_bytes(1, 64, 64, 1, 8, 1)   # ignoring: the binary mode's size
    args = (FAKE, 1, 64, 64, 1, 8, 0, FAKE * 64, None)
    assert ccl.ccl_label_ws(*args, FAKE * 128, need - 1, None) == ccl.CCL_ERR_NO_MEMORY
    assert ccl.ccl_label_ws(*args, FAKE * 128 + 16, need, None) == ccl.CCL_ERR_INVALID_ARG
    assert ccl.ccl_label_ws(*args, None, need, None) == ccl.CCL_ERR_INVALID_ARG
    # a workspace sharing bytes with the image, the labels or the counts
    img, labels, counts = FAKE * 64, FAKE * 128, FAKE * 192
    base = (img, 1, 64, 64, 1, 8, 0, labels)
    for ws in (img - (need // 256) * 256 + 256,    # its end reaches the image
               img + 1024,                          # inside the image
               labels + 4096 * 4 - 256):            # from the labels' last bytes on
        ws -= ws % 256
        assert ccl.ccl_label_ws(*base, None, ws, need, None) == ccl.CCL_ERR_INVALID_ARG, hex(ws)
        assert ccl.ccl_label_ignore(*base[:6], 5, labels, None, ws, need_ign, None) == \
            ccl.CCL_ERR_INVALID_ARG, hex(ws)
    assert need % 256 == 0
    ws = counts + 256 - need                        # its last 256 bytes hold the counts
    assert ccl.ccl_label_ws(*base, counts, ws, need, None) == ccl.CCL_ERR_INVALID_ARG


def test_stage_names_and_counter(lib):
    assert [ccl.ccl_stage_name(k) for k in range(5)] == [
        "tile_local", "seams", "scan", "resolve", "number"]
    assert ccl.ccl_stage_name(5) == ""
    assert ccl.ccl_kernel_launches() >= 0
    ms, n = ccl.ccl_stage_times()      # nothing recorded: no device work
    assert n == 0 and ms == [0.0] * 5


def test_set_option(lib):
    assert ccl.ccl_set_option(ccl.CCL_OPT_STAGE_EVENTS, 0) == ccl.CCL_OK
    assert ccl.ccl_set_option(ccl.CCL_OPT_WALK_CAP, 5) == ccl.CCL_OK
    assert ccl.ccl_set_option(ccl.CCL_OPT_WALK_CAP, 0) == ccl.CCL_OK
    assert ccl.ccl_set_option(12345, 1) == ccl.CCL_ERR_INVALID_ARG


def test_no_cpu_path():
    import torch
    with pytest.raises(ValueError):
        ccl.label(torch.zeros((4, 4), dtype=torch.uint8))


def test_region_stats_host_checks(lib):
    assert ccl.ccl_region_stats_workspace_bytes(-1) == 0
    assert ccl.ccl_region_stats_workspace_bytes(0) == 256
    assert ccl.ccl_region_stats_workspace_bytes(31) == 256
    assert ccl.ccl_region_stats_workspace_bytes(100) == 1024      # 101 int64 offsets
    lab, n, st, ws = FAKE * 64, FAKE * 96, FAKE * 128, FAKE * 160
    # empty calls touch nothing
    assert ccl.ccl_region_stats(lab, 0, 8, 8, n, st, 10, None, 0, None) == ccl.CCL_OK
    assert ccl.ccl_region_stats(lab, 2, 0, 8, n, st, 10, None, 0, None) == ccl.CCL_OK
    # bad sizes, pointers and alignment are refused on the host
    assert ccl.ccl_region_stats(lab, -1, 8, 8, n, st, 10, None, 0, None) == ccl.CCL_ERR_INVALID_ARG
    assert ccl.ccl_region_stats(lab, 1, 8, 8, n, st, -1, None, 0, None) == ccl.CCL_ERR_INVALID_ARG
    assert ccl.ccl_region_stats(None, 1, 8, 8, n, st, 10, None, 0, None) == ccl.CCL_ERR_INVALID_ARG
    assert ccl.ccl_region_stats(lab, 1, 8, 8, None, st, 10, None, 0, None) == ccl.CCL_ERR_INVALID_ARG
    assert ccl.ccl_region_stats(lab + 2, 1, 8, 8, n, st, 10, None, 0, None) == ccl.CCL_ERR_INVALID_ARG
    assert ccl.ccl_region_stats(lab, 1, 8, 8, n, st + 4, 10, None, 0, None) == ccl.CCL_ERR_INVALID_ARG
    assert ccl.ccl_region_stats(lab, 1, 8, 8, n, None, 10, None, 0, None) == ccl.CCL_ERR_INVALID_ARG
    assert ccl.ccl_region_stats(lab, 1, 1 << 16, 1 << 15, n, st, 10, None, 0, None) == \
        ccl.CCL_ERR_TOO_LARGE
    assert ccl.ccl_region_stats(lab, 1, 8, 8, n, st, 10, ws + 16, 256, None) == ccl.CCL_ERR_INVALID_ARG
    assert ccl.ccl_region_stats(lab, 100, 8, 8, n, st, 10, ws, 512, None) == ccl.CCL_ERR_NO_MEMORY


def test_counters_only_in_the_counters_build(lib):
    import ctypes
    buf = (ctypes.c_ulonglong * 8)()
    # the product library has no counters compiled in
    assert ccl.ccl_debug_counters(buf, 8, 0) == ccl.CCL_ERR_INVALID_ARG
    assert len(ccl.COUNTER_NAMES) == 8


def test_plain_c_consumer_links_and_runs(lib, tmp_path):
    """The header is C: a C99 program (tests/c/abi_consumer.c) compiles against
    it with -pedantic, links against libccl.so and checks the entry points
    that answer on the host, the statistics struct layout included."""
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    so = ccl.build()
    exe = str(tmp_path / "abi_consumer")
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                           "-I", os.path.join(root, "include"),
                           os.path.join(root, "tests", "c", "abi_consumer.c"),
                           "-o", exe, so, "-Wl,-rpath," + os.path.dirname(so)])
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, (out.returncode, out.stdout, out.stderr)
    assert "C consumer ok" in out.stdout


def test_workspace_bytes_of_the_largest_shapes(lib):
    """Geometry is computed in 64 bits and every per-tile record is sized by
    the image's full tile: images of up to 2^32 - 1 pixels are accepted.  A
    square of many whole tiles needs about 3.9 B/px; the one-row image of
    2^31 - 1 pixels about 15 B/px (every pixel of its one-row tiles is a
    border pixel with a possible slot); 2^32 pixels are refused, and so is an
    image whose tiles' slots would outnumber 32-bit ids (2 rows of 2^31 - 1)."""
    w1 = (1 << 31) - 1
    row = ccl.ccl_workspace_bytes(1, 1, w1, 1, 8, 0)
    assert 0 < row < 16 * w1
    sq = ccl.ccl_workspace_bytes(1, 46340, 46340, 1, 8, 0)
    assert 3.5 * 46340 ** 2 < sq < 4.5 * 46340 ** 2
    big = ccl.ccl_workspace_bytes(1, 65535, 65535, 1, 8, 0)   # 2^32 - 2^17 + 1 pixels
    assert 3.5 * 65535 ** 2 < big < 4.5 * 65535 ** 2
    col = ccl.ccl_workspace_bytes(1, w1, 1, 1, 8, 0)
    assert col > 0
    assert ccl.ccl_workspace_bytes(1, 1 << 16, 1 << 16, 1, 8, 0) == 0
    assert ccl.ccl_workspace_bytes(1, 2, w1, 1, 8, 0) == 0
