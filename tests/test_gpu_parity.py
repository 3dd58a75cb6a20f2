"""GPU parity: the CUDA library (through its C ABI) against the oracle,
element by element, bit-exact.  Sizes span several 256 x 16 tiles and ragged
tails; edge cases cover empty, 1-pixel, 1-row and 1-column images, batches
beyond the 65535 grid-z limit, every pixel width and both modes and
connectivities."""
import itertools

import numpy as np
import pytest
import torch

import connected_component_labelling_gb300 as ccl
import oracle
import workloads
from tests.helpers import read_golden

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
MODES = {"all": oracle.MODE_ALL, "binary": oracle.MODE_BINARY}
NP_OF = {torch.uint8: np.uint8, torch.int16: np.uint16, torch.int32: np.uint32}


@pytest.fixture(scope="module", autouse=True)
def built():
    ccl.build()
    oracle.build()
    yield
    ccl.check_status()


def to_np(img):
    a = img.cpu().numpy()
    return a.view(NP_OF[img.dtype])


def gpu_label(img, conn, mode):
    lab, n = ccl.label(img.to(DEV), connectivity=conn, mode=mode)
    ccl.check_status()
    return lab.cpu().numpy(), n.cpu().numpy()


def assert_parity(img, conn, mode):
    lab, n = gpu_label(img, conn, mode)
    olab, on = oracle.label(to_np(img), conn, MODES[mode])
    np.testing.assert_array_equal(n, on)
    np.testing.assert_array_equal(lab, olab)
    return lab, n


@pytest.mark.parametrize("name", ["p2_4x4_binary_8conn.txt", "p2_4x4_binary_4conn.txt",
                                  "p2_6x6_buf_8conn.txt", "p2_6x6_buf_4conn.txt",
                                  "p1_3x3_stepped_8conn.txt", "p1_3x3_stepped_4conn.txt"])
def test_worked_examples(name):
    g = read_golden(name)
    img = torch.as_tensor(g["image"].astype(np.uint8))
    lab, n = gpu_label(img, g["connectivity"], g["mode"])
    np.testing.assert_array_equal(lab, g["labels"])
    assert int(n) == g["n"]


@pytest.mark.parametrize("conn", [4, 8])
@pytest.mark.parametrize("mode", ["all", "binary"])
def test_every_binary_4x4_as_one_batch(conn, mode):
    # 65536 images in one call: more than the 65535 limit of a grid's z axis
    k = torch.arange(1 << 16)
    imgs = ((k[:, None] >> torch.arange(16)[None, :]) & 1).to(torch.uint8).view(-1, 4, 4)
    assert_parity(imgs, conn, mode)


@pytest.mark.parametrize("conn", [4, 8])
@pytest.mark.parametrize("mode", ["all", "binary"])
def test_every_3colour_3x3(conn, mode):
    imgs = torch.tensor(list(itertools.product(range(3), repeat=9)), dtype=torch.uint8).view(-1, 3, 3)
    assert_parity(imgs, conn, mode)


SHAPES = [(1, 1), (1, 700), (700, 1), (3, 5), (16, 256), (17, 257), (33, 513), (100, 1000),
          (255, 31), (300, 777)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("dtype", [torch.uint8, torch.int16, torch.int32])
@pytest.mark.parametrize("conn", [4, 8])
@pytest.mark.parametrize("mode", ["all", "binary"])
def test_random_shapes(shape, dtype, conn, mode):
    H, W = shape
    g = torch.Generator().manual_seed(H * 1009 + W * 7 + conn + (mode == "binary"))
    img = torch.randint(0, 3, (2, H, W), generator=g).to(dtype)
    assert_parity(img, conn, mode)


@pytest.mark.parametrize("p", [0.2, 0.4, 0.41, 0.6, 0.8])
@pytest.mark.parametrize("conn", [4, 8])
def test_bernoulli_near_percolation(p, conn):
    img = workloads.bernoulli_masks(3, 517, 1031, (p,), seed=int(p * 100))
    assert_parity(img, conn, "binary")


@pytest.mark.parametrize("structure", ["serpentine", "checkerboard", "random4"])
@pytest.mark.parametrize("conn", [4, 8])
@pytest.mark.parametrize("mode", ["all", "binary"])
def test_adversarial_structures(structure, conn, mode):
    H = W = 1024
    img = {"serpentine": workloads.serpentine(H, W), "checkerboard": workloads.checkerboard(H, W),
           "random4": workloads.random_levels(H, W, 4, seed=11)}[structure]
    lab, n = assert_parity(img, conn, mode)
    if structure == "serpentine":
        assert int(n) == (1 if mode == "binary" else 1 + H // 2)
    if structure == "checkerboard" and mode == "all":
        assert int(n) == (2 if conn == 8 else H * W)


def test_rgba_drawing():
    img = workloads.drawing(777, 1111, seed=5, n_segments=300, n_rects=12, levels=16,
                            hatched=False)
    assert_parity(img, 8, "all")
    assert_parity(img, 4, "all")
    sheet = workloads.c4_sheet(H=1200, W=1680)
    assert_parity(sheet, 8, "all")


def test_empty_inputs():
    for shape in [(0, 5), (5, 0)]:
        img = torch.zeros(shape, dtype=torch.uint8, device=DEV)
        lab, n = ccl.label(img)
        assert lab.shape == shape and int(n) == 0
    img = torch.zeros((0, 4, 4), dtype=torch.uint8, device=DEV)
    lab, n = ccl.label(img)
    assert n.shape == (0,)
    n = torch.full((3,), 7, dtype=torch.int32, device=DEV)
    img = torch.zeros((3, 0, 4), dtype=torch.uint8, device=DEV)
    ccl.label(img, n_out=n)
    assert n.tolist() == [0, 0, 0]


def test_all_background_and_all_one_value():
    z = torch.zeros((2, 70, 300), dtype=torch.uint8)
    lab, n = gpu_label(z, 8, "binary")
    assert (lab == 0).all() and n.tolist() == [0, 0]
    lab, n = gpu_label(z, 8, "all")
    assert (lab == 1).all() and n.tolist() == [1, 1]


def test_determinism():
    img = workloads.bernoulli_masks(2, 700, 900, (0.41,), seed=9).to(DEV)
    ref, rn = ccl.label(img, 8, "binary")
    for _ in range(10):
        lab, n = ccl.label(img, 8, "binary")
        assert torch.equal(lab, ref) and torch.equal(n, rn)
    ccl.check_status()


def test_workspace_and_host_entry_points():
    img = workloads.random_levels(333, 555, 3, seed=2)
    olab, on = oracle.label(img.numpy(), 8, oracle.MODE_BINARY)
    d = img.to(DEV)
    need = ccl.ccl_workspace_bytes(1, 333, 555, 1, 8, 1)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    lab, n = ccl.label(d, 8, "binary", workspace=ws)
    ccl.check_status()
    np.testing.assert_array_equal(lab.cpu().numpy(), olab)
    # host buffers in, host buffers out
    himg = img.pin_memory()
    hlab = torch.empty((333, 555), dtype=torch.int32).pin_memory()
    hn = torch.empty((1,), dtype=torch.int32)
    with torch.cuda.device(DEV):
        rc = ccl.ccl_label_host(himg.data_ptr(), 1, 333, 555, 1, 8, 1, hlab.data_ptr(),
                                hn.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == ccl.CCL_OK
    np.testing.assert_array_equal(hlab.numpy(), olab)
    assert int(hn[0]) == on


@pytest.mark.parametrize("B,H,W,pb,conn,mode", [
    (1, 20, 300, 1, 8, 1),      # 2 tile rows: fewer rows than copy bands
    (5, 37, 257, 1, 4, 0),      # 15 tile rows in 8 bands that cross image boundaries
    (3, 64, 520, 4, 8, 0),      # RGBA, whole tiles
    (2, 45, 264, 3, 8, 1),      # 24-bit RGB
])
def test_host_entry_point_in_bands(B, H, W, pb, conn, mode):
    """ccl_label_host copies the image up and the labels down in bands of
    tile rows while the kernels run; results are those of the oracle."""
    rng = np.random.default_rng(B * 1000 + H)
    host = rng.integers(0, 3, size=(B, H, W, pb) if pb != 1 else (B, H, W)).astype(np.uint8)
    olab, on = oracle.label(host, conn, mode)
    himg = torch.from_numpy(host).contiguous().pin_memory()
    hlab = torch.empty((B, H, W), dtype=torch.int32).pin_memory()
    hn = torch.empty((B,), dtype=torch.int32)
    with torch.cuda.device(DEV):
        rc = ccl.ccl_label_host(himg.data_ptr(), B, H, W, pb, conn, mode, hlab.data_ptr(),
                                hn.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == ccl.CCL_OK
    np.testing.assert_array_equal(hlab.numpy(), olab)
    np.testing.assert_array_equal(hn.numpy(), on)
    # pageable host memory and no region counts
    plab = np.zeros((B, H, W), dtype=np.int32)
    pimg = np.ascontiguousarray(host)
    with torch.cuda.device(DEV):
        rc = ccl.ccl_label_host(pimg.ctypes.data, B, H, W, pb, conn, mode, plab.ctypes.data, None,
                                torch.cuda.current_stream().cuda_stream)
    assert rc == ccl.CCL_OK
    np.testing.assert_array_equal(plab, olab)


def test_walk_cap_reports_device_limit_without_hanging():
    # a serpentine forces long union-find walks; a cap of 1 step must trip,
    # be reported, and leave the context usable
    img = workloads.serpentine(256, 256).to(DEV)
    try:
        assert ccl.ccl_set_option(ccl.CCL_OPT_WALK_CAP, 1) == ccl.CCL_OK
        ccl.label(img, 8, "binary")
        assert ccl.ccl_last_status(torch.cuda.current_stream().cuda_stream) == \
            ccl.CCL_ERR_DEVICE_LIMIT
    finally:
        ccl.ccl_set_option(ccl.CCL_OPT_WALK_CAP, 0)
    lab, n = ccl.label(img, 8, "binary")
    ccl.check_status()
    assert int(n) == 1


def test_walk_cap_through_the_host_entry_point():
    """ccl_label_host returns a limit tripped in its own call directly, and
    keeps to its own status word: a limit another call tripped stays in the
    device's sticky word for ccl_last_status, and a clean host call after it
    still reports CCL_OK."""
    img = workloads.serpentine(256, 256)
    himg = img.contiguous().pin_memory()
    hlab = torch.empty((256, 256), dtype=torch.int32).pin_memory()
    hn = torch.empty((1,), dtype=torch.int32).pin_memory()
    st = torch.cuda.current_stream(DEV).cuda_stream

    def host_call():
        return ccl.ccl_label_host(himg.data_ptr(), 1, 256, 256, 1, 8, ccl.CCL_MODE_BINARY,
                                  hlab.data_ptr(), hn.data_ptr(), st)
    try:
        assert ccl.ccl_set_option(ccl.CCL_OPT_WALK_CAP, 1) == ccl.CCL_OK
        assert host_call() == ccl.CCL_ERR_DEVICE_LIMIT
        assert ccl.ccl_last_status(st) == ccl.CCL_OK          # not in the sticky word
        ccl.label(img.to(DEV), 8, "binary")                   # trips the sticky word
    finally:
        ccl.ccl_set_option(ccl.CCL_OPT_WALK_CAP, 0)
    assert host_call() == ccl.CCL_OK                          # its own word is clean
    assert int(hn[0]) == 1
    np.testing.assert_array_equal(hlab.numpy(), img.numpy().astype(np.int32))
    assert ccl.ccl_last_status(st) == ccl.CCL_ERR_DEVICE_LIMIT   # the other call's finding
    assert ccl.ccl_last_status(st) == ccl.CCL_OK


def test_other_stream_and_batch_offsets():
    imgs = workloads.bernoulli_masks(5, 211, 389, (0.3, 0.5, 0.7), seed=4)
    olab, on = oracle.label(imgs.numpy(), 4, oracle.MODE_BINARY)
    s = torch.cuda.Stream(device=DEV)
    d = imgs.to(DEV)
    torch.cuda.current_stream(DEV).synchronize()
    with torch.cuda.stream(s):
        lab, n = ccl.label(d, 4, "binary")
    s.synchronize()
    ccl.check_status(s)
    np.testing.assert_array_equal(lab.cpu().numpy(), olab)
    np.testing.assert_array_equal(n.cpu().numpy(), on)


# ------------------------------------------------------ ignoring one value

@pytest.mark.parametrize("shape", [(1, 1), (17, 257), (100, 1000), (255, 31)])
@pytest.mark.parametrize("dtype", [torch.uint8, torch.int16, torch.int32])
@pytest.mark.parametrize("conn", [4, 8])
@pytest.mark.parametrize("ignore", [0, 2])
def test_ignore_random_shapes(shape, dtype, conn, ignore):
    H, W = shape
    g = torch.Generator().manual_seed(H * 31 + W + conn + 7 * ignore)
    img = torch.randint(0, 3, (2, H, W), generator=g).to(dtype)
    lab, n = ccl.label_ignore(img.to(DEV), ignore, connectivity=conn)
    ccl.check_status()
    olab, on = oracle.label_ignore(to_np(img), ignore, conn)
    np.testing.assert_array_equal(n.cpu().numpy(), on)
    np.testing.assert_array_equal(lab.cpu().numpy(), olab)


@pytest.mark.parametrize("conn", [4, 8])
def test_ignore_paper_of_a_drawing(conn):
    img = workloads.drawing(777, 1111, seed=5, n_segments=300, n_rects=12, levels=16,
                            hatched=False)
    white = 0xFFFFFFFF
    lab, n = ccl.label_ignore(img.to(DEV), white, connectivity=conn)
    ccl.check_status()
    olab, on = oracle.label_ignore(to_np(img), white, conn)
    assert int(n) == int(on)
    np.testing.assert_array_equal(lab.cpu().numpy(), olab)
    assert (lab.cpu().numpy()[to_np(img) == white] == 0).all()


def test_ignore_zero_equals_binary_mode():
    img = workloads.random_levels(333, 555, 3, seed=12).to(DEV)
    a, na = ccl.label_ignore(img, 0, connectivity=8)
    b, nb = ccl.label(img, 8, "binary")
    ccl.check_status()
    assert torch.equal(a, b) and torch.equal(na, nb)


def test_tensor_wrappers_reject_bad_buffers():
    """Caller buffers reach the kernels as raw pointers, so the tensor
    wrappers refuse a wrong dtype, size, layout or device before any call
    into the library; the right buffers then label as usual."""
    img = workloads.random_levels(40, 300, 3, seed=5).to(DEV)
    n = img.numel()
    bad_outs = [torch.empty(n, dtype=torch.int64, device=DEV),            # dtype
                torch.empty(n - 1, dtype=torch.int32, device=DEV),        # size
                torch.empty((300, 40), dtype=torch.int32, device=DEV).t(),  # layout
                torch.empty(n, dtype=torch.int32)]                       # host memory
    for out in bad_outs:
        with pytest.raises(ValueError):
            ccl.label(img, 8, "all", out=out)
        with pytest.raises(ValueError):
            ccl.label_ignore(img, 0, 8, out=out)
    for n_out in (torch.empty(2, dtype=torch.int32, device=DEV), torch.empty(1, dtype=torch.int32)):
        with pytest.raises(ValueError):
            ccl.label(img, 8, "all", n_out=n_out)
    with pytest.raises(ValueError):
        ccl.label(img, 8, "all", workspace=torch.empty(1 << 20, dtype=torch.uint8))
    lab, cnt = ccl.label(img, 8, "all", out=torch.empty(n, dtype=torch.int32, device=DEV),
                         n_out=torch.empty(1, dtype=torch.int32, device=DEV))
    ccl.check_status()
    olab, on = oracle.label(to_np(img.cpu()), 8, oracle.MODE_ALL)
    np.testing.assert_array_equal(lab.cpu().numpy().reshape(olab.shape), olab)
    with pytest.raises(ValueError):
        ccl.region_stats(lab.view(40, 300).to(torch.int64), cnt)
    with pytest.raises(ValueError):
        ccl.region_stats(lab.view(40, 300), cnt.cpu())
    with pytest.raises(ValueError):
        ccl.region_stats(lab.view(40, 300), cnt.reshape(1).repeat(2))
    ccl.check_status()
