"""GPU parity of the TMA tile-copy path against the oracle: bit-exact box images.

"2 . Le Tensor Memory Accelerator" 2.2-2.5 and "H100 . cuTensorMap (TMA descriptor)"
11 (swizzle), 14 (OOB fill in shared memory, source untouched)."""
import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_gb300 import inputs as gen
from tma_pipelined_tensor_gb300 import tg

from gpu_util import to_device, to_device_bf16

pytestmark = pytest.mark.gpu

# (swizzle, inner box width in bf16 elements) of the tile-copy workload: the inner
# width is cut to the swizzle span (128 bytes for none and 128B).
MODES = [(tg.TG_SWZ_NONE, 64), (tg.TG_SWZ_32B, 16), (tg.TG_SWZ_64B, 32), (tg.TG_SWZ_128B, 64)]


def run_copy(T_dev, H, W, es, box_w, box_h, swz, oob=tg.TG_OOB_ZERO, ld=None):
    import torch
    nbytes = tg.image_bytes(H, W, es, box_w, box_h)
    out = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")
    st = tg.tile_copy(T_dev, box_w, box_h, swz, out, oob=oob)
    assert st == tg.TG_OK
    assert tg.tg_status_sync(None) == tg.TG_OK
    return out.cpu().numpy()


@pytest.fixture(scope="module")
def copy_tensor_4100x8200():
    T = gen.copy_tensor(4100, 8200)
    return T, to_device_bf16(T)


@pytest.mark.parametrize("swz,box_w", MODES)
def test_full_workload_bit_exact(copy_tensor_4100x8200, swz, box_w):
    T, T_dev = copy_tensor_4100x8200
    got = run_copy(T_dev, 4100, 8200, 2, box_w, 128, swz)
    want = oracle.tma_box_images(T, 4100, 8200, 8200 * 2, 2, box_w, 128, swz)
    assert got.size == want.size
    mism = np.flatnonzero(got != want)
    assert mism.size == 0, "first mismatching bytes: %s" % mism[:8].tolist()


@pytest.mark.parametrize("stages,blocks,order,l2p", [
    (2, 1, 0, 0), (8, 1, 2, 1), (3, 2, 0, 2), (12, 0, 2, 3), (6, 2, 1, 4), (4, 3, 2, 0)])
def test_copy_knobs_keep_the_image(copy_tensor_4100x8200, stages, blocks, order, l2p):
    import torch
    T, T_dev = copy_tensor_4100x8200
    nbytes = tg.image_bytes(4100, 8200, 2, 64, 128)
    out = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")
    assert tg.tile_copy(T_dev, 64, 128, tg.TG_SWZ_128B, out, stages=stages,
                        blocks_per_sm=blocks, order=order, l2_promotion=l2p) == tg.TG_OK
    assert tg.tg_status_sync(None) == tg.TG_OK
    want = oracle.tma_box_images(T, 4100, 8200, 8200 * 2, 2, 64, 128, tg.TG_SWZ_128B)
    assert np.array_equal(out.cpu().numpy(), want)


def test_source_unchanged(copy_tensor_4100x8200):
    import torch
    T, T_dev = copy_tensor_4100x8200
    run_copy(T_dev, 4100, 8200, 2, 64, 128, tg.TG_SWZ_128B)
    assert np.array_equal(T_dev.view(torch.int16).cpu().numpy().view(np.uint16), T)


@pytest.mark.parametrize("swz,box_w", MODES)
@pytest.mark.parametrize("H,W,box_h", [(300, 200, 128), (1, 8, 128), (129, 72, 64), (37, 1000, 8)])
def test_unique_patterns_ragged(swz, box_w, H, W, box_h):
    T = gen.unique_bits_tensor(H, W, seed=H * 131 + W)
    got = run_copy(to_device_bf16(T), H, W, 2, box_w, box_h, swz)
    want = oracle.tma_box_images(T, H, W, W * 2, 2, box_w, box_h, swz)
    assert np.array_equal(got, want)


def test_row_stride_with_padding():
    H, W, ld = 257, 200, 264
    T = np.full((H, ld), 0xBEEF, dtype=np.uint16)
    T[:, :W] = gen.unique_bits_tensor(H, W, seed=21)
    Td = to_device_bf16(T)[:, :W]
    got = run_copy(Td, H, W, 2, 64, 128, tg.TG_SWZ_128B)
    want = oracle.tma_box_images(T, H, W, ld * 2, 2, 64, 128, tg.TG_SWZ_128B)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("dtype,es,box_w,swz", [
    ("f32", 4, 32, tg.TG_SWZ_128B), ("f32", 4, 8, tg.TG_SWZ_32B), ("u8", 1, 128, tg.TG_SWZ_128B),
    ("u8", 1, 64, tg.TG_SWZ_64B), ("u8", 1, 48, tg.TG_SWZ_NONE)])
def test_other_element_sizes(dtype, es, box_w, swz):
    H, W = 100, (333 if es == 1 else 150)
    ld_bytes = -(-W * es // 16) * 16  # row stride rounded up to 16 bytes
    raw = np.zeros((H, ld_bytes), dtype=np.uint8)
    raw[:, :W * es] = gen.unique_bits_tensor(H, ld_bytes // 2, seed=es).view(np.uint8)[:, :W * es]
    arr = raw.view(np.float32) if dtype == "f32" else raw
    got = run_copy(to_device(arr)[:, :W], H, W, es, box_w, 64, swz)
    want = oracle.tma_box_images(raw, H, W, ld_bytes, es, box_w, 64, swz)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("swz,box_w", MODES)
def test_nan_fill_out_of_bounds(swz, box_w):
    H, W = 130, 104  # 208-byte rows: a multiple of 16
    T = gen.copy_tensor(H, W)
    got = run_copy(to_device_bf16(T), H, W, 2, box_w, 128, swz, oob=tg.TG_OOB_NAN)
    want = oracle.tma_box_images(T, H, W, W * 2, 2, box_w, 128, swz, oob_nan=True)
    g16, w16 = got.view(np.uint16), want.view(np.uint16)
    oob = w16 == 0xFFFF  # the oracle marks fill positions with all-ones (a NaN)
    assert np.array_equal(g16[~oob], w16[~oob])
    assert np.isnan(gen.bf16_bits_to_f32(g16[oob])).all()


# ------------------------------------------------------------------------------------
# Rank 1..5 tensors with element strides
# ------------------------------------------------------------------------------------
ND_CASES = [
    # torch shape (outermost first), extent and element strides (innermost first), swizzle
    ((5, 12, 200), [64, 8, 2], [1, 2, 1], tg.TG_SWZ_128B),
    ((7, 9, 100), [32, 4, 3], [1, 1, 2], tg.TG_SWZ_64B),
    ((3, 4, 6, 70), [16, 4, 2, 2], [1, 2, 1, 2], tg.TG_SWZ_32B),
    ((2, 3, 3, 5, 64), [64, 4, 2, 2, 1], [1, 1, 2, 1, 1], tg.TG_SWZ_NONE),
    ((2, 2, 3, 4, 128), [64, 2, 3, 1, 2], [1, 2, 1, 1, 1], tg.TG_SWZ_128B),
    ((1000,), [64], [1], tg.TG_SWZ_128B),
    ((300, 200), [64, 128], [1, 3], tg.TG_SWZ_128B),
]


def _padded_nd(shape, seed, pad=8):
    """bf16 unique-pattern tensor with the innermost rows padded (non-packed strides)."""
    import torch
    inner = -(-(shape[-1] + pad) // 8) * 8   # padded rows stay 16-byte multiples
    n = int(np.prod(shape[:-1])) * inner
    flat = gen.unique_bits_tensor(1, n, seed=seed)[0]
    full = flat.reshape(tuple(shape[:-1]) + (inner,))
    dev = torch.from_numpy(full.view(np.int16).copy()).view(torch.bfloat16).cuda()
    view = dev[..., :shape[-1]]
    return full, view


@pytest.mark.parametrize("shape,extent,estr,swz", ND_CASES)
def test_nd_copy_bit_exact(shape, extent, estr, swz):
    import torch
    full, view = _padded_nd(shape, seed=sum(shape))
    dims = list(reversed(shape))
    strides = [view.stride(view.dim() - 1 - i) * 2 for i in range(1, view.dim())]
    t = tg.make_tensor_nd(view.data_ptr(), tg.TG_DTYPE_BF16, dims, strides)
    b = tg.make_box_nd(extent, estr)
    nbytes = tg.tma_tile_copy_nd_image_bytes(t, b)
    out = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")
    assert tg.tile_copy_nd(view, extent, estr, swz, out) == tg.TG_OK
    assert tg.tg_status_sync(None) == tg.TG_OK
    want = oracle.tma_box_images_nd(full.view(np.uint8).reshape(-1), dims, strides, 2, extent,
                                    estr, swz)
    got = out.cpu().numpy()
    assert got.size == want.size
    assert np.array_equal(got, want), np.flatnonzero(got != want)[:8].tolist()


def test_nd_rank2_equals_2d_entry_point(copy_tensor_4100x8200):
    import torch
    T, T_dev = copy_tensor_4100x8200
    nbytes = tg.image_bytes(4100, 8200, 2, 64, 128)
    a = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    b = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    tg.tile_copy(T_dev, 64, 128, tg.TG_SWZ_128B, a)
    tg.tile_copy_nd(T_dev, [64, 128], [1, 1], tg.TG_SWZ_128B, b)
    assert tg.tg_status_sync(None) == tg.TG_OK
    assert torch.equal(a, b)


def test_nd_nan_fill():
    import torch
    shape, extent, estr = (3, 5, 72), [64, 4, 2], [1, 1, 1]
    vals = gen.copy_tensor(15, 72).reshape(shape)
    view = torch.from_numpy(vals.view(np.int16).copy()).view(torch.bfloat16).cuda()
    dims = list(reversed(shape))
    strides = [view.stride(2 - i) * 2 for i in range(1, 3)]
    t = tg.make_tensor_nd(view.data_ptr(), tg.TG_DTYPE_BF16, dims, strides)
    nbytes = tg.tma_tile_copy_nd_image_bytes(t, tg.make_box_nd(extent, estr))
    out = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    assert tg.tile_copy_nd(view, extent, estr, tg.TG_SWZ_128B, out, oob=tg.TG_OOB_NAN) == tg.TG_OK
    assert tg.tg_status_sync(None) == tg.TG_OK
    want = oracle.tma_box_images_nd(vals, dims, strides, 2, extent, estr, tg.TG_SWZ_128B,
                                    oob_nan=True).view(np.uint16)
    got = out.cpu().numpy().view(np.uint16)
    fill = want == 0xFFFF
    assert np.array_equal(got[~fill], want[~fill])
    assert np.isnan(gen.bf16_bits_to_f32(got[fill])).all()


# ------------------------------------------------------------------------------------
# Region copies: the box grid starts at any index (negative included) and may run past
# the tensor's end; every out-of-bounds element reads the fill value
# ------------------------------------------------------------------------------------
REGION_CASES = [
    # shape (outermost first), extent, estr, swizzle, origin, nboxes (innermost first)
    ((300, 200), [64, 128], [1, 1], tg.TG_SWZ_128B, [-8, -8], [4, 4]),
    ((300, 200), [64, 128], [1, 1], tg.TG_SWZ_NONE, [-64, -128], [6, 5]),   # a ring of empty boxes
    ((40, 48), [16, 16], [1, 1], tg.TG_SWZ_32B, [-8, -8], [1, 1]),          # the corner box
    ((129, 72), [32, 64], [1, 1], tg.TG_SWZ_64B, [40, 100], [3, 2]),        # starts inside, runs past
    ((6, 9, 40), [64, 4, 3], [1, 2, 1], tg.TG_SWZ_128B, [-16, -3, -1], [2, 4, 4]),
    ((2, 3, 4, 5, 64), [64, 2, 2, 3, 2], [1, 1, 2, 1, 1], tg.TG_SWZ_128B, [0, -1, 1, -2, 1],
     [1, 4, 2, 2, 2]),
]


@pytest.mark.parametrize("shape,extent,estr,swz,origin,nboxes", REGION_CASES)
def test_region_copy_bit_exact(shape, extent, estr, swz, origin, nboxes):
    import torch
    full, view = _padded_nd(shape, seed=sum(shape) + 7)
    dims = list(reversed(shape))
    strides = [view.stride(view.dim() - 1 - i) * 2 for i in range(1, view.dim())]
    t = tg.make_tensor_nd(view.data_ptr(), tg.TG_DTYPE_BF16, dims, strides)
    b = tg.make_box_nd(extent, estr)
    nbytes = tg.tma_tile_copy_region_nd_image_bytes(t, b, nboxes)
    out = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")
    assert tg.tile_copy_region(view, extent, origin, nboxes, swz, out, estr) == tg.TG_OK
    assert tg.tg_status_sync(None) == tg.TG_OK
    want = oracle.tma_box_images_region(full.view(np.uint8).reshape(-1), dims, strides, 2,
                                        extent, estr, origin, nboxes, swz)
    got = out.cpu().numpy()
    assert got.size == want.size
    assert np.array_equal(got, want), np.flatnonzero(got != want)[:8].tolist()


def test_region_at_origin_zero_equals_whole_copy(copy_tensor_4100x8200):
    import torch
    T, T_dev = copy_tensor_4100x8200
    nbytes = tg.image_bytes(4100, 8200, 2, 64, 128)
    a = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    b = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    tg.tile_copy_nd(T_dev, [64, 128], [1, 1], tg.TG_SWZ_128B, a)
    tg.tile_copy_region(T_dev, [64, 128], [0, 0], [129, 33], tg.TG_SWZ_128B, b)
    assert tg.tg_status_sync(None) == tg.TG_OK
    assert torch.equal(a, b)


def test_region_nan_fill_on_both_sides():
    import torch
    H, W = 37, 72
    vals = gen.copy_tensor(H, W)
    view = torch.from_numpy(vals.view(np.int16).copy()).view(torch.bfloat16).cuda()
    extent, origin, nboxes = [64, 16], [-64, -8], [3, 4]
    t = tg.make_tensor_nd(view.data_ptr(), tg.TG_DTYPE_BF16, [W, H], [W * 2])
    nbytes = tg.tma_tile_copy_region_nd_image_bytes(t, tg.make_box_nd(extent), nboxes)
    out = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    assert tg.tile_copy_region(view, extent, origin, nboxes, tg.TG_SWZ_128B, out,
                               oob=tg.TG_OOB_NAN) == tg.TG_OK
    assert tg.tg_status_sync(None) == tg.TG_OK
    want = oracle.tma_box_images_region(vals, [W, H], [W * 2], 2, extent, [1, 1], origin, nboxes,
                                        tg.TG_SWZ_128B, oob_nan=True).view(np.uint16)
    got = out.cpu().numpy().view(np.uint16)
    fill = want == 0xFFFF
    assert fill.any() and (~fill).any()
    assert np.array_equal(got[~fill], want[~fill])
    assert np.isnan(gen.bf16_bits_to_f32(got[fill])).all()


# ------------------------------------------------------------------------------------
# Copy back (tensor store through the same descriptor): the hardware's inverse of the
# swizzled image, which checks the oracle's image model against the copy engine
# ------------------------------------------------------------------------------------
BACK_CASES = [
    ((300, 200), [64, 128], tg.TG_SWZ_128B),
    ((300, 200), [64, 128], tg.TG_SWZ_NONE),
    ((129, 72), [32, 64], tg.TG_SWZ_64B),
    ((37, 1000), [16, 8], tg.TG_SWZ_32B),
    ((6, 9, 40), [64, 4, 3], tg.TG_SWZ_128B),
    ((2, 3, 4, 5, 64), [64, 2, 2, 3, 2], tg.TG_SWZ_128B),
]


@pytest.mark.parametrize("shape,extent,swz", BACK_CASES)
def test_oracle_image_copied_back_restores_the_tensor(shape, extent, swz):
    import torch
    full, view = _padded_nd(shape, seed=sum(shape) + 11)
    dims = list(reversed(shape))
    strides = [view.stride(view.dim() - 1 - i) * 2 for i in range(1, view.dim())]
    # the oracle's image of the tensor, written back by the hardware into a blank tensor
    img = oracle.tma_box_images_nd(full.view(np.uint8).reshape(-1), dims, strides, 2, extent,
                                   [1] * len(extent), swz)
    blank_full = torch.full(full.shape, 0x7FC1, dtype=torch.int16, device="cuda")
    blank = blank_full.view(torch.bfloat16)[..., :shape[-1]]
    img_dev = torch.from_numpy(img).cuda()
    assert tg.tile_copy_back(blank, extent, swz, img_dev) == tg.TG_OK
    assert tg.tg_status_sync(None) == tg.TG_OK
    got = blank_full.cpu().numpy().view(np.uint16)
    assert np.array_equal(got[..., :shape[-1]], full[..., :shape[-1]])
    assert (got[..., shape[-1]:] == 0x7FC1).all()        # row padding untouched


def test_copy_round_trip_full_workload(copy_tensor_4100x8200):
    import torch
    T, T_dev = copy_tensor_4100x8200
    # 4100 x 8200: rows of 16400 bytes; the last box row and column run past the edge
    nbytes = tg.image_bytes(4100, 8200, 2, 64, 128)
    img = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    tg.tile_copy(T_dev, 64, 128, tg.TG_SWZ_128B, img)
    back = torch.zeros_like(T_dev)
    assert tg.tile_copy_back(back, [64, 128], tg.TG_SWZ_128B, img) == tg.TG_OK
    assert tg.tg_status_sync(None) == tg.TG_OK
    assert torch.equal(back.view(torch.int16), T_dev.view(torch.int16))


def test_copy_back_rules():
    import torch
    T = torch.zeros((8, 16), dtype=torch.bfloat16, device="cuda")[:, :12]   # 24-byte rows
    img = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    assert tg.tile_copy_back(T, [8, 8], tg.TG_SWZ_NONE, img, check=False) == tg.TG_ERR_UNSUPPORTED
    T = torch.zeros((8, 16), dtype=torch.bfloat16, device="cuda")
    t = tg.make_tensor_nd(T.data_ptr(), tg.TG_DTYPE_BF16, [16, 8], [32])
    assert tg.tma_tile_copy_back_nd(t, tg.make_box_nd([8, 8], [1, 2]), tg.TG_SWZ_NONE,
                                    img.data_ptr(), img.numel()) == tg.TG_ERR_UNSUPPORTED
    assert tg.tma_tile_copy_back_nd(t, tg.make_box_nd([8, 8]), tg.TG_SWZ_NONE, None,
                                    1 << 16) == tg.TG_ERR_INVALID_VALUE
    assert tg.tma_tile_copy_back_nd(t, tg.make_box_nd([8, 8]), tg.TG_SWZ_NONE, img.data_ptr(),
                                    64) == tg.TG_ERR_BUFFER_TOO_SMALL
