"""GPU parity of the region statistics (ccl_region_stats) against the
oracle's, field by field, bit-exact (all fields are integers).  The labels
given to each side are each side's own: the GPU's statistics are computed
from the GPU's labels, the oracle's from the oracle's labels (the two label
images are equal, checked here too)."""
import numpy as np
import pytest
import torch

import connected_component_labelling_gb300 as ccl
import oracle
import workloads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
NP_OF = {torch.uint8: np.uint8, torch.int16: np.uint16, torch.int32: np.uint32}


@pytest.fixture(scope="module", autouse=True)
def built():
    ccl.build()
    oracle.build()


def gpu_stats(img, conn, mode, capacity=None):
    lab, n = ccl.label(img, conn, mode)
    raw, f = ccl.region_stats(lab, n, capacity=capacity)
    torch.cuda.synchronize()
    return lab, n, {k: v.cpu().numpy() for k, v in f.items()}


def oracle_stats(img_np, conn, mode):
    lab, n = oracle.label(img_np, conn, mode)
    return lab, n, oracle.region_stats(lab, np.atleast_1d(n))


def compare(img, conn, mode):
    lab, n, got = gpu_stats(img, conn, mode)
    host = img.cpu().numpy().view(NP_OF[img.dtype])
    olab, on, want = oracle_stats(host, conn, mode)
    np.testing.assert_array_equal(lab.cpu().numpy().reshape(olab.shape), olab)
    np.testing.assert_array_equal(np.atleast_1d(n.cpu().numpy()), np.atleast_1d(on))
    assert len(want) == sum(int(v) for v in np.atleast_1d(on))
    for fld in oracle.STAT_DTYPE.names:
        np.testing.assert_array_equal(got[fld], want[fld], err_msg=fld)
    return want


@pytest.mark.parametrize("shape", [(1, 1), (3, 5), (16, 256), (17, 257), (40, 600), (129, 1000)])
@pytest.mark.parametrize("dtype", [torch.uint8, torch.int32])
@pytest.mark.parametrize("conn", [4, 8])
@pytest.mark.parametrize("mode", [ccl.CCL_MODE_ALL, ccl.CCL_MODE_BINARY])
def test_random_levels(shape, dtype, conn, mode):
    g = torch.Generator().manual_seed(hash((shape, conn, mode)) & 0xFFFF)
    img = torch.randint(0, 3, shape, generator=g).to(dtype).to(DEV)
    compare(img, conn, mode)


@pytest.mark.parametrize("B", [1, 5])
def test_batch_of_masks(B):
    img = workloads.bernoulli_masks(B, 96, 333, [0.3, 0.5, 0.7, 0.4, 0.6][:B], seed=3, device=DEV)
    compare(img, 8, ccl.CCL_MODE_BINARY)


def test_drawing_rgba():
    img = workloads.c0_drawing(device=DEV)
    compare(img, 8, ccl.CCL_MODE_ALL)


def test_long_regions_many_tiles():
    # one region through every tile (serpentine) and a constant image: the
    # same entry gets every tile's totals
    compare(workloads.serpentine(300, 1100, device=DEV), 8, ccl.CCL_MODE_BINARY)
    want = compare(torch.full((200, 700), 7, dtype=torch.uint8, device=DEV), 4, ccl.CCL_MODE_ALL)
    assert want["area"][0] == 200 * 700


def test_many_regions_per_tile_overflow_the_table():
    # 4-connectivity checkerboard: every pixel its own region, more than the
    # per-tile table holds, so runs go straight to the global entries
    r = torch.arange(64, device=DEV)[:, None]
    c = torch.arange(512, device=DEV)[None, :]
    compare(((r + c) & 1).to(torch.uint8), 4, ccl.CCL_MODE_ALL)


def test_ignore_labels():
    img = workloads.c0_drawing(device=DEV)
    white = 0xFFFFFFFF
    lab, n = ccl.label_ignore(img, white, connectivity=8)
    raw, f = ccl.region_stats(lab, n)
    olab, on = oracle.label_ignore(img.cpu().numpy().view(np.uint32), white, 8)
    want = oracle.region_stats(olab, [on])
    for fld in oracle.STAT_DTYPE.names:
        np.testing.assert_array_equal(f[fld].cpu().numpy(), want[fld], err_msg=fld)


def test_no_regions_and_empty():
    lab, n, got = gpu_stats(torch.zeros((40, 300), dtype=torch.uint8, device=DEV), 8, ccl.CCL_MODE_BINARY)
    assert int(n) == 0 and all(len(v) == 0 for v in got.values())
    ccl.check_status()


def test_capacity_too_small_is_reported():
    img = torch.randint(0, 2, (64, 256), generator=torch.Generator().manual_seed(1),
                        dtype=torch.uint8).to(DEV)
    lab, n = ccl.label(img, 4, ccl.CCL_MODE_ALL)
    total = int(n)
    raw, f = ccl.region_stats(lab, n, capacity=total - 5)
    assert ccl.ccl_last_status(torch.cuda.current_stream().cuda_stream) == ccl.CCL_ERR_NO_MEMORY
    olab, on = oracle.label(img.cpu().numpy(), 4, oracle.MODE_ALL)
    want = oracle.region_stats(olab, [on])[:total - 5]
    for fld in oracle.STAT_DTYPE.names:      # the entries that fit are complete
        np.testing.assert_array_equal(f[fld].cpu().numpy(), want[fld], err_msg=fld)


def test_label_out_of_range_is_reported():
    lab = torch.ones((16, 300), dtype=torch.int32, device=DEV)
    lab[3, 7] = 5                            # but the image has one region
    n = torch.ones((1,), dtype=torch.int32, device=DEV)
    ccl.region_stats(lab, n, capacity=1)
    assert ccl.ccl_last_status(torch.cuda.current_stream().cuda_stream) == ccl.CCL_ERR_INVALID_ARG


def test_caller_workspace_and_stream():
    img = workloads.bernoulli_masks(3, 64, 640, [0.4, 0.5, 0.6], seed=5, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        lab, n = ccl.label(img, 8, ccl.CCL_MODE_BINARY, stream=s)
        ws = torch.empty(ccl.ccl_region_stats_workspace_bytes(3), dtype=torch.uint8, device=DEV)
        raw, f = ccl.region_stats(lab, n, workspace=ws, stream=s)
    s.synchronize()
    olab, on = oracle.label(img.cpu().numpy(), 8, oracle.MODE_BINARY)
    want = oracle.region_stats(olab, on)
    for fld in oracle.STAT_DTYPE.names:
        np.testing.assert_array_equal(f[fld].cpu().numpy(), want[fld], err_msg=fld)


def test_sheet_full_size():
    img = workloads.c4_sheet(device=DEV)
    lab, n = ccl.label(img, 8, ccl.CCL_MODE_ALL)
    raw, f = ccl.region_stats(lab, n)
    ccl.check_status()
    host = img.cpu().numpy().view(np.uint32)
    del img
    olab, on = oracle.label(host, 8, oracle.MODE_ALL)
    assert int(n) == int(on)
    want = oracle.region_stats(olab, [on])
    for fld in oracle.STAT_DTYPE.names:
        np.testing.assert_array_equal(f[fld].cpu().numpy(), want[fld], err_msg=fld)
