"""ccl_label_noalloc: labelling for callers that may not allocate device memory
(their GPU memory belongs to a framework arena or a fixed budget, or they
cannot pay for the synchronisation cudaMalloc/cudaFree may cause).  Its
scratch is a fixed array inside the library, shared by every call on a
device.

Checked through the C ABI against ccl_label, bit for bit (labels are
integers: the tolerance is exact equality), on consecutive calls with
different images so that contents left in the shared array by one call
cannot leak into the next.  Collected last on purpose.
"""
import pytest
import torch

import connected_component_labelling_gb300 as ccl
import workloads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _noalloc(img, conn, mode):
    B, H, W, pb, squeeze = ccl.image_geometry(img)
    lab = torch.full((B, H, W), -7, dtype=torch.int32, device=DEV)
    n = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    with torch.cuda.device(DEV):
        rc = ccl.ccl_label_noalloc(img.data_ptr(), B, H, W, pb, conn, mode, lab.data_ptr(),
                                   n.data_ptr(), torch.cuda.current_stream(DEV).cuda_stream)
    assert rc == ccl.CCL_OK, ccl.ccl_status_string(rc)
    torch.cuda.synchronize(DEV)
    return (lab.view(H, W), n.view(())) if squeeze else (lab, n)


def test_noalloc_matches_ccl_label_on_consecutive_calls():
    ccl.build()
    sheet = workloads.c4_sheet(H=1500, W=2100).to(DEV)          # RGBA, 8-conn, all
    masks = workloads.bernoulli_masks(4, 517, 1031, (0.4, 0.6), seed=21).to(DEV)
    cases = [(sheet, 8, ccl.CCL_MODE_ALL), (masks, 4, ccl.CCL_MODE_BINARY),
             (sheet, 8, ccl.CCL_MODE_ALL)]
    for img, conn, mode in cases:
        ref_lab, ref_n = ccl.label(img, connectivity=conn, mode=mode)
        ccl.check_status()
        lab, n = _noalloc(img, conn, mode)
        assert torch.equal(n, ref_n)
        assert torch.equal(lab, ref_lab)
        assert int(n.min()) > 0


def test_noalloc_rejects_images_beyond_its_scratch():
    # 4000 x 4000 needs about 64 MB of scratch, more than the fixed 32 MiB
    img = torch.zeros((4000, 4000), dtype=torch.uint8, device=DEV)
    lab = torch.empty((4000, 4000), dtype=torch.int32, device=DEV)
    assert ccl.ccl_workspace_bytes(1, 4000, 4000, 1, 8, 0) > ccl.CCL_NOALLOC_SCRATCH_BYTES - 256
    with torch.cuda.device(DEV):
        rc = ccl.ccl_label_noalloc(img.data_ptr(), 1, 4000, 4000, 1, 8, 0, lab.data_ptr(), None,
                                   torch.cuda.current_stream(DEV).cuda_stream)
    assert rc == ccl.CCL_ERR_TOO_LARGE


def test_noalloc_reports_a_tripped_limit_in_its_counts():
    """A device limit tripped during a no-alloc call (here a walk cap of one
    step on a serpentine) comes back as -1 in every count, not through the
    device's sticky word; the call after it, with the cap restored, starts
    from a clean status and matches ccl_label again."""
    ccl.build()
    img = workloads.serpentine(256, 256).to(DEV)
    try:
        assert ccl.ccl_set_option(ccl.CCL_OPT_WALK_CAP, 1) == ccl.CCL_OK
        _, n = _noalloc(img, 8, ccl.CCL_MODE_BINARY)
        assert int(n) == -1
    finally:
        ccl.ccl_set_option(ccl.CCL_OPT_WALK_CAP, 0)
    lab, n = _noalloc(img, 8, ccl.CCL_MODE_BINARY)
    ref_lab, ref_n = ccl.label(img, connectivity=8, mode="binary")
    ccl.check_status()
    assert int(n) == int(ref_n) == 1
    assert torch.equal(lab, ref_lab)
