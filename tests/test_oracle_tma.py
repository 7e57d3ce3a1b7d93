"""Pins of the oracle's TMA box/swizzle/zero-fill model.

Sources: "H100 . cuTensorMap (TMA 描述符)", section 11.3 (swizzle formula and bit maps),
section 11.4 (the permutation moves 16-byte units inside 128-byte rows), section 14
(out-of-bounds fill happens in shared memory, the source is unchanged); "2 . Le Tensor
Memory Accelerator", section 2.5 (out-of-bounds parts of a tile become zeros).
"""
import os

import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_gb300 import inputs as gen

HERE = os.path.dirname(os.path.abspath(__file__))
SPAN = {0: None, 1: 32, 2: 64, 3: 128}


def golden_bitmaps():
    maps = {}
    with open(os.path.join(HERE, "golden", "swizzle_bitmaps.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            pairs = [tuple(int(x) for x in p.split("^")) for p in parts[2:]]
            maps[int(parts[1])] = pairs
    return maps


def swizzle_from_bitmap(a, pairs):
    """Applies the page's printed bit maps: bit dst ^= bit src (sources read first)."""
    out = a
    for dst, src in pairs:
        out ^= ((a >> src) & 1) << dst
    return out


def test_golden_bitmaps_cover_all_modes():
    assert sorted(golden_bitmaps()) == [0, 1, 2, 3]


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_formula_reproduces_printed_bitmaps(mode):
    pairs = golden_bitmaps()[mode]
    for a in range(0, 1 << 13):
        assert oracle.swizzle(a, mode) == swizzle_from_bitmap(a, pairs), (mode, a)


@pytest.mark.parametrize("mode", [1, 2, 3])
def test_low_four_bits_fixed_and_atom_bijection(mode):
    for a in range(0, 1 << 14, 7):
        assert oracle.swizzle(a, mode) & 15 == a & 15
    for base in range(0, 8192, 1024):
        atom = set(range(base, base + 1024))
        assert {oracle.swizzle(a, mode) for a in atom} == atom
    for a in range(4096):  # an involution: bits 7..9 are never changed
        assert oracle.swizzle(oracle.swizzle(a, mode), mode) == a


def test_128b_chunk_j_of_row_r_lands_at_j_xor_r():
    for r in range(32):
        for j in range(8):
            a = r * 128 + j * 16
            assert oracle.swizzle(a, 3) == r * 128 + ((j ^ (r % 8)) * 16)


@pytest.mark.parametrize("mode", [1, 2, 3])
def test_one_logical_column_over_eight_rows_hits_eight_bank_groups(mode):
    span = SPAN[mode]
    for j in range(span // 16):
        slots = {(oracle.swizzle(r * span + j * 16, mode) % 128) // 16 for r in range(8)}
        assert len(slots) == 8


def _unswizzle_box(img, box_h, box_w, es, mode):
    n = box_h * box_w * es
    idx = np.array([oracle.swizzle(a, mode) for a in range(n)], dtype=np.int64)
    return img[idx].reshape(box_h, box_w * es)


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_boxes_unswizzle_to_tensor_blocks_with_zero_fill(mode):
    H, W, es = 300, 200, 2
    box_w = 64 if mode in (0, 3) else SPAN[mode] // es
    box_h = 128
    T = gen.unique_bits_tensor(H, W)
    img = oracle.tma_box_images(T, H, W, W * es, es, box_w, box_h, mode)
    nbi, nbj = oracle.box_grid(H, W, box_w, box_h)
    box_bytes = box_h * box_w * es
    assert img.size == nbi * nbj * box_bytes
    Tb = T.view(np.uint8).reshape(H, W * es)
    for bi in range(nbi):
        for bj in range(nbj):
            b = bi * nbj + bj
            dense = _unswizzle_box(img[b * box_bytes:(b + 1) * box_bytes], box_h, box_w, es, mode)
            r1 = min(box_h, H - bi * box_h)
            c1 = min(box_w, W - bj * box_w) * es
            want = Tb[bi * box_h:bi * box_h + r1, bj * box_w * es:bj * box_w * es + c1]
            assert np.array_equal(dense[:r1, :c1], want)
            assert not dense[r1:, :].any() and not dense[:, c1:].any()


def test_image_multiset_equals_tensor_plus_fill():
    H, W, es, box_w, box_h = 100, 72, 2, 64, 64
    T = gen.unique_bits_tensor(H, W, seed=3)
    img = oracle.tma_box_images(T, H, W, W * es, es, box_w, box_h, 3).view(np.uint16)
    nbi, nbj = oracle.box_grid(H, W, box_w, box_h)
    n_fill = nbi * nbj * box_w * box_h - H * W
    vals, counts = np.unique(img, return_counts=True)
    tv, tc = np.unique(np.concatenate([T.ravel(), np.zeros(n_fill, np.uint16)]),
                       return_counts=True)
    assert np.array_equal(vals, tv) and np.array_equal(counts, tc)


def test_row_stride_padding_is_skipped():
    H, W, es = 40, 24, 2
    ld = 40
    T = np.full((H, ld), 0xDEAD, dtype=np.uint16)
    T[:, :W] = gen.unique_bits_tensor(H, W, seed=5)
    a = oracle.tma_box_images(T, H, W, ld * es, es, 16, 32, 1)
    b = oracle.tma_box_images(T[:, :W].copy(), H, W, W * es, es, 16, 32, 1)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("es", [1, 4])
def test_other_element_sizes_move_whole_elements(es):
    H, W = 9, 32 // es * 3 + 1
    box_w, box_h = 32 // es, 4
    raw = gen.unique_bits_tensor(H, W * es // 2 + 1, seed=9).view(np.uint8)[:, :W * es].copy()
    img = oracle.tma_box_images(raw, H, W, W * es, es, box_w, box_h, 1)
    nbi, nbj = oracle.box_grid(H, W, box_w, box_h)
    box_bytes = box_h * box_w * es
    for b in range(nbi * nbj):
        bi, bj = divmod(b, nbj)
        dense = _unswizzle_box(img[b * box_bytes:(b + 1) * box_bytes], box_h, box_w, es, 1)
        r1 = min(box_h, H - bi * box_h)
        c1 = min(box_w, W - bj * box_w) * es
        assert np.array_equal(dense[:r1, :c1],
                              raw[bi * box_h:bi * box_h + r1, bj * box_w * es:bj * box_w * es + c1])


def test_brute_force_python_model_tiny():
    """A second, loop-by-loop model built on the printed bit maps, on a tiny tensor."""
    maps = golden_bitmaps()
    H, W, es = 10, 40, 2
    T = gen.unique_bits_tensor(H, W, seed=11)
    Tb = T.view(np.uint8).reshape(H, W * es)
    for mode, box_w in [(0, 24), (1, 16), (2, 32), (3, 64)]:
        box_h = 4
        nbi, nbj = -(-H // box_h), -(-W // box_w)
        box_bytes = box_h * box_w * es
        want = np.zeros(nbi * nbj * box_bytes, dtype=np.uint8)
        for bi in range(nbi):
            for bj in range(nbj):
                for r in range(box_h):
                    for c in range(box_w):
                        for byte in range(es):
                            row, col = bi * box_h + r, bj * box_w + c
                            v = Tb[row, col * es + byte] if (row < H and col < W) else 0
                            a = r * box_w * es + c * es + byte
                            want[(bi * nbj + bj) * box_bytes + swizzle_from_bitmap(a, maps[mode])] = v
        got = oracle.tma_box_images(T, H, W, W * es, es, box_w, box_h, mode)
        assert np.array_equal(got, want), mode


def test_nan_fill_marks_only_out_of_bounds():
    H, W = 5, 10
    T = gen.copy_tensor(H, W)
    img = oracle.tma_box_images(T, H, W, W * 2, 2, 16, 8, 1, oob_nan=True)
    dense = gen.bf16_bits_to_f32(_unswizzle_box(img, 8, 16, 2, 1).view(np.uint16))
    assert np.isnan(dense[H:, :]).all() and np.isnan(dense[:, W:]).all()
    assert np.array_equal(dense[:H, :W], gen.bf16_bits_to_f32(T))


def test_copy_config_grid_and_image_sizes():
    # 4100 x 8200 bf16, box 128 rows; inner width = swizzle span (64 elements for
    # none/128B, 32 for 64B, 16 for 32B)
    H, W = 4100, 8200
    got = {}
    for box_w in (64, 32, 16):
        nbi, nbj = oracle.box_grid(H, W, box_w, 128)
        got[box_w] = (nbi, nbj, nbi * nbj * 128 * box_w * 2)
    assert got[64] == (33, 129, 69_746_688)
    assert got[32] == (33, 257, 69_476_352)
    assert got[16] == (33, 513, 69_341_184)


def test_copy_tensor_values():
    T = gen.copy_tensor(4100, 8200)
    f = gen.bf16_bits_to_f32(T)
    assert f[0, 0] == 0 and f[0, 1] == 1 and f[0, 255] == 255
    # (7*8200 + 2) mod 65521 = 57402 -> bf16 keeps 8 significant bits
    assert f[7, 2] == 57344.0
    # (4099*8200 + 8199) mod 65521 = 7726 = 0b1111000101110 -> RNE to 8 bits: 7712
    assert f[4099, 8199] == 7712.0


# ------------------------------------------------------------------------------------
# Rank 1..5 boxes with element strides ("H100 . cuTensorMap", sections 8-9)
# ------------------------------------------------------------------------------------
@pytest.mark.parametrize("mode,box_w", [(0, 64), (1, 16), (2, 32), (3, 64)])
def test_nd_rank2_unit_strides_equals_2d_model(mode, box_w):
    H, W, es = 300, 200, 2
    T = gen.unique_bits_tensor(H, W, seed=31)
    want = oracle.tma_box_images(T, H, W, W * es, es, box_w, 128, mode)
    got = oracle.tma_box_images_nd(T, [W, H], [W * es], es, [box_w, 128], [1, 1], mode)
    assert np.array_equal(got, want)


def _loop_model_nd(T_bytes, dims, strides, es, ext, estr, mode_pairs):
    """Independent element-by-element model using the printed bit maps for the swizzle."""
    import itertools
    rank = len(dims)
    stride_all = [es] + list(strides)
    nb = [-(-d // e) for d, e in zip(dims, ext)]
    L = [-(-e // s) for e, s in zip(ext, estr)]
    box_bytes = int(np.prod(L)) * es
    out = np.zeros(int(np.prod(nb)) * box_bytes, dtype=np.uint8)
    for bidx, b in enumerate(itertools.product(*[range(n) for n in reversed(nb)])):
        b = list(reversed(b))          # dimension 0 fastest
        for eidx, j in enumerate(itertools.product(*[range(l) for l in reversed(L)])):
            j = list(reversed(j))
            idx = [b[i] * ext[i] + j[i] * estr[i] for i in range(rank)]
            inside = all(idx[i] < dims[i] for i in range(rank))
            off = sum(idx[i] * stride_all[i] for i in range(rank))
            for byte in range(es):
                a = eidx * es + byte
                v = T_bytes[off + byte] if inside else 0
                out[bidx * box_bytes + swizzle_from_bitmap(a, mode_pairs)] = v
    return out


@pytest.mark.parametrize("dims,ext,estr,es,mode", [
    ([24, 5, 3], [8, 2, 2], [1, 1, 2], 2, 0),            # rank 3, stride 2 on the outer dim
    ([16, 7, 4], [16, 4, 3], [1, 2, 1], 2, 1),           # 32 B rows, 32B swizzle, stride 2
    ([8, 3, 2, 5], [8, 2, 2, 3], [1, 1, 1, 2], 4, 1),    # rank 4, fp32, stride 2
    ([64, 2, 2, 2, 3], [64, 1, 2, 1, 2], [1, 1, 2, 1, 1], 2, 3),   # rank 5, 128B swizzle
    ([40], [16], [1], 2, 1),                             # rank 1
])
def test_nd_matches_loop_model(dims, ext, estr, es, mode):
    maps = golden_bitmaps()
    # pad every row so that strides are larger than the packed extents
    strides, acc = [], dims[0] * es + 16
    for d in dims[1:]:
        strides.append(acc)
        acc = acc * d + 32
    nbytes = (strides[-1] * dims[-1] if strides else dims[0] * es) + 64
    T = gen.unique_bits_tensor(1, nbytes // 2 + 1, seed=sum(dims)).view(np.uint8)[0, :nbytes].copy()
    got = oracle.tma_box_images_nd(T, dims, strides, es, ext, estr, mode)
    want = _loop_model_nd(T, dims, strides, es, ext, estr, maps[mode])
    assert np.array_equal(got, want)


def test_nd_element_stride_picks_every_sth_index():
    # rank 2, outer stride 3: the box of 9 outer indices holds rows 0, 3, 6 only
    H, W = 9, 16
    T = gen.unique_bits_tensor(H, W, seed=41)
    img = oracle.tma_box_images_nd(T, [W, H], [W * 2], 2, [16, 9], [1, 3], 0).view(np.uint16)
    assert img.size == 3 * 16
    assert np.array_equal(img.reshape(3, 16), T[[0, 3, 6], :])


# ------------------------------------------------------------------------------------
# Box grids that start anywhere: negative origins and boxes past the tensor's end are
# out of bounds on every side (the edge fill of the TMA page and cuTensorMap section 14)
# ------------------------------------------------------------------------------------
def _loop_model_region(T_bytes, dims, strides, es, ext, estr, origin, nb, mode_pairs):
    import itertools
    rank = len(dims)
    stride_all = [es] + list(strides)
    L = [-(-e // s) for e, s in zip(ext, estr)]
    box_bytes = int(np.prod(L)) * es
    out = np.zeros(int(np.prod(nb)) * box_bytes, dtype=np.uint8)
    for bidx, b in enumerate(itertools.product(*[range(n) for n in reversed(nb)])):
        b = list(reversed(b))
        for eidx, j in enumerate(itertools.product(*[range(l) for l in reversed(L)])):
            j = list(reversed(j))
            idx = [origin[i] + b[i] * ext[i] + j[i] * estr[i] for i in range(rank)]
            inside = all(0 <= idx[i] < dims[i] for i in range(rank))
            for byte in range(es):
                a = eidx * es + byte
                v = T_bytes[sum(idx[i] * stride_all[i] for i in range(rank)) + byte] if inside else 0
                out[bidx * box_bytes + swizzle_from_bitmap(a, mode_pairs)] = v
    return out


def test_region_at_origin_zero_is_the_whole_tensor_copy():
    H, W, es = 300, 200, 2
    T = gen.unique_bits_tensor(H, W, seed=43)
    for mode, bw in [(0, 64), (3, 64), (2, 32)]:
        want = oracle.tma_box_images_nd(T, [W, H], [W * es], es, [bw, 128], [1, 1], mode)
        got = oracle.tma_box_images_region(T, [W, H], [W * es], es, [bw, 128], [1, 1], [0, 0],
                                           [-(-W // bw), -(-H // 128)], mode)
        assert np.array_equal(got, want)


def test_region_box_at_minus_eight_holds_the_corner():
    # a 16 x 16 box at (-8, -8): its lower-right quarter is T[0:8, 0:8], the rest zero
    H, W = 40, 48
    T = gen.unique_bits_tensor(H, W, seed=44)
    img = oracle.tma_box_images_region(T, [W, H], [W * 2], 2, [16, 16], [1, 1], [-8, -8],
                                       [1, 1], 0).view(np.uint16).reshape(16, 16)
    assert np.array_equal(img[8:, 8:], T[:8, :8])
    assert not img[:8, :].any() and not img[:, :8].any()


def test_region_box_wholly_outside_is_all_fill():
    T = gen.unique_bits_tensor(8, 16, seed=45)
    img = oracle.tma_box_images_region(T, [16, 8], [32], 2, [8, 4], [1, 1], [-16, -4], [1, 1], 0)
    assert not img.any()
    img = oracle.tma_box_images_region(T, [16, 8], [32], 2, [8, 4], [1, 1], [16, 0], [1, 2], 0,
                                       oob_nan=True)
    assert (img == 0xFF).all()


@pytest.mark.parametrize("dims,ext,estr,es,mode,origin,nb", [
    ([24, 5], [8, 2], [1, 1], 2, 0, [-8, -1], [5, 4]),                 # both sides past
    ([16, 7, 4], [16, 4, 3], [1, 2, 1], 2, 1, [-16, -3, 2], [3, 3, 1]),
    ([8, 3, 2, 5], [8, 2, 2, 3], [1, 1, 1, 2], 4, 1, [4, -2, -1, 3], [2, 3, 2, 2]),
    ([64, 2, 2, 2, 3], [64, 1, 2, 1, 2], [1, 1, 2, 1, 1], 2, 3, [-64, 1, -1, -1, 0], [3, 2, 2, 3, 2]),
    ([40], [16], [1], 2, 1, [-24], [5]),
])
def test_region_matches_loop_model(dims, ext, estr, es, mode, origin, nb):
    maps = golden_bitmaps()
    strides, acc = [], dims[0] * es + 16
    for d in dims[1:]:
        strides.append(acc)
        acc = acc * d + 32
    nbytes = (strides[-1] * dims[-1] if strides else dims[0] * es) + 64
    T = gen.unique_bits_tensor(1, nbytes // 2 + 1, seed=sum(dims) + 3).view(np.uint8)[0, :nbytes].copy()
    got = oracle.tma_box_images_region(T, dims, strides, es, ext, estr, origin, nb, mode)
    want = _loop_model_region(T, dims, strides, es, ext, estr, origin, nb, maps[mode])
    assert np.array_equal(got, want)
