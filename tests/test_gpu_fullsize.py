"""GPU parity at the full sizes of the five workloads, through ccl_label_ws --
the call bench.py times -- against the oracle, element by element, bit-exact
(labels are integers).  The adversarial structures are also checked against
their closed forms."""
import numpy as np
import pytest
import torch

import connected_component_labelling_gb300 as ccl
import oracle
import workloads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
NP_OF = {torch.uint8: np.uint8, torch.int32: np.uint32}


@pytest.fixture(scope="module", autouse=True)
def built():
    ccl.build()
    oracle.build()


def label_ws(img, conn, mode):
    """The benchmark's call: caller-provided workspace, current stream."""
    B, H, W, pb, squeeze = ccl.image_geometry(img)
    need = ccl.ccl_workspace_bytes(B, H, W, pb, conn, mode)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    lab, n = ccl.label(img, conn, mode, workspace=ws)
    ccl.check_status()
    del ws
    return lab, n


def compare(img_dev, conn, mode):
    lab, n = label_ws(img_dev, conn, mode)
    host = img_dev.cpu().numpy()
    host = host.view(NP_OF[img_dev.dtype])
    olab, on = oracle.label(host, conn, mode)
    np.testing.assert_array_equal(np.asarray(n.cpu().numpy()).reshape(-1), np.asarray(on).reshape(-1))
    gl = lab.cpu().numpy()
    assert np.array_equal(gl, olab), "labels differ from the oracle"
    return gl, int(np.asarray(on).reshape(-1)[0])


def test_c0_drawing_1024():
    compare(workloads.c0_drawing(device=DEV), 8, ccl.CCL_MODE_ALL)


def test_c1_masks_64x1024():
    compare(workloads.c1_masks(device=DEV), 8, ccl.CCL_MODE_BINARY)


def test_c2_slide_20000():
    img = workloads.c2_slide(device=DEV)
    frac = img.float().mean().item()
    assert 0.40 < frac < 0.50          # the 55th-percentile threshold leaves ~45 % foreground
    compare(img, 4, ccl.CCL_MODE_BINARY)


@pytest.mark.parametrize("structure", ["serpentine", "checkerboard", "random4"])
@pytest.mark.parametrize("conn", [4, 8])
@pytest.mark.parametrize("mode", [ccl.CCL_MODE_ALL, ccl.CCL_MODE_BINARY])
def test_c3_structures_8192(structure, conn, mode):
    H = W = 8192
    img = workloads.c3_structures(device=DEV)[structure]
    _, n = compare(img, conn, mode)
    if structure == "serpentine":
        assert n == (1 if mode == ccl.CCL_MODE_BINARY else 1 + H // 2)
    if structure == "checkerboard":
        expect = {(8, 0): 2, (4, 0): H * W, (8, 1): 1, (4, 1): H * W // 2}[(conn, mode)]
        assert n == expect


def test_c4_sheet_24000x33600():
    img = workloads.c4_sheet(device=DEV)
    assert img.shape == (24000, 33600)
    _, n = compare(img, 8, ccl.CCL_MODE_ALL)
    assert n > 1_000_000


def test_c4_sheet_paper_ignored():
    # "every-colour", ch. 08 switch 4: the sheet with its white paper ignored
    img = workloads.c4_sheet(device=DEV)
    white = 0xFFFFFFFF
    # (ignoring a value runs the binary mode's pipeline: its workspace size)
    need = ccl.ccl_workspace_bytes(1, 24000, 33600, 4, 8, ccl.CCL_MODE_BINARY)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    lab, n = ccl.label_ignore(img, white, connectivity=8, workspace=ws)
    ccl.check_status()
    del ws
    olab, on = oracle.label_ignore(img.cpu().numpy().view(np.uint32), white, 8)
    assert int(n) == int(on)
    assert np.array_equal(lab.cpu().numpy(), olab)
