"""Pins of the MX (microscaling) oracle.

Definition followed (OCP Microscaling Formats (MX) specification v1.0): a block of 32
elements along K shares one E8M0 scale X (value 2^(X - 127), X = 255 is NaN); an
element's value is its FP8 value times its block's scale; the GEMM is the ordinary matrix
product of those values.  The pins below check the oracle against things that do not
come from the oracle: the scale code's values, offsets of the storage layout worked out
by hand, closed forms on matrices of ones, and the reduction to the unscaled FP8 oracle
(itself pinned on every bit pattern) when every scale is 1.
"""
import math

import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_gb300 import inputs as gen

ONE_E4M3 = 0x38   # 1.0 in E4M3: exponent 7 (bias 7), mantissa 0


def test_e8m0_values():
    assert oracle.e8m0_to_double(127) == 1.0
    assert oracle.e8m0_to_double(128) == 2.0
    assert oracle.e8m0_to_double(126) == 0.5
    assert oracle.e8m0_to_double(0) == 2.0 ** -127
    assert oracle.e8m0_to_double(254) == 2.0 ** 127
    assert math.isnan(oracle.e8m0_to_double(255))


@pytest.mark.parametrize("rows,r,j,want", [
    (300, 37, 5, 1621),     # atom (k-slice 1, row group 0) = 3 * 512; line 5 * 16; quarter 1 * 4; block 1
    (128, 0, 0, 0),
    (128, 127, 3, 511),     # last line (31 * 16), last quarter (3 * 4), last block of the atom (3)
    (256, 128, 4, 1536),    # k-slice 1 of a 2-row-group operand, row group 1: (1 * 2 + 1) * 512
    (129, 128, 0, 512),     # second row group of the first k-slice
])
def test_scale_offsets_worked_by_hand(rows, r, j, want):
    assert oracle.mx_scale_offset(rows, r, j) == want


def test_generator_packs_at_the_same_offsets():
    lg, pk = gen.mx_scales(300, 200, 1, 4)
    assert lg.shape == (300, 7) and pk.size == gen.mx_scale_bytes(300, 200) == 3 * 2 * 512
    for r, j in [(0, 0), (37, 5), (299, 6), (128, 3), (255, 4)]:
        assert pk[oracle.mx_scale_offset(300, r, j)] == lg[r, j]


def ones(rows, K):
    return np.full((rows, K), ONE_E4M3, dtype=np.uint8)


def test_unit_scales_reduce_to_the_fp8_oracle():
    M, N, K = 37, 29, 200
    A = gen.f8_matrix(M, K, 3, 0, "normal")
    B = gen.f8_matrix(N, K, 3, 1, "normal")
    SA = gen.mx_pack_scales(np.full((M, 7), 127, np.uint8), K)
    SB = gen.mx_pack_scales(np.full((N, 7), 127, np.uint8), K)
    got, mag = oracle.gemm_mx(A, SA, B, SB, M, N, K)
    ref, refmag = oracle.gemm(A, B, M, N, K, in_kind="e4m3")
    assert np.array_equal(got, ref) and np.array_equal(mag, refmag)
    A5 = gen.f8_matrix(M, K, 4, 0, "normal", e5m2=True)
    B5 = gen.f8_matrix(N, K, 4, 1, "normal", e5m2=True)
    got, _ = oracle.gemm_mx(A5, SA, B5, SB, M, N, K, kind="e5m2")
    ref, _ = oracle.gemm(A5, B5, M, N, K, in_kind="e5m2")
    assert np.array_equal(got, ref)


def test_ones_closed_form():
    # K = 96: three blocks.  Row i's scales 2^(i % 3) in every block; column j's scales
    # 1, 1/2, 1 in blocks 0, 1, 2.  C_ij = 32 * 2^(i % 3) * (1 + 1/2 + 1) = 80 * 2^(i % 3).
    M, N, K = 6, 5, 96
    la = np.array([[127 + i % 3] * 3 for i in range(M)], np.uint8)
    lb = np.array([[127, 126, 127]] * N, np.uint8)
    got, _ = oracle.gemm_mx(ones(M, K), gen.mx_pack_scales(la, K), ones(N, K),
                            gen.mx_pack_scales(lb, K), M, N, K)
    want = np.array([[80.0 * 2 ** (i % 3)] * N for i in range(M)])
    assert np.array_equal(got, want)


def test_one_scale_byte_moves_one_row_and_one_block():
    # every scale 1 except byte 1621 of A's scales (row 37, block 5, worked out above),
    # which is 2: row 37 gains the 32 elements of block 5 once more, nothing else moves
    M, N, K = 300, 4, 256
    SA = np.full(gen.mx_scale_bytes(M, K), 127, np.uint8)
    SA[1621] = 128
    SB = np.full(gen.mx_scale_bytes(N, K), 127, np.uint8)
    got, _ = oracle.gemm_mx(ones(M, K), SA, ones(N, K), SB, M, N, K)
    want = np.full((M, N), float(K))
    want[37, :] = K + 32
    assert np.array_equal(got, want)


def test_partial_last_block():
    # K = 70: blocks of 32, 32 and 6 elements; the last block's scale (8) applies to its 6
    M, N, K = 3, 2, 70
    la = np.full((M, 3), 127, np.uint8)
    lb = np.array([[127, 127, 130]] * N, np.uint8)
    got, _ = oracle.gemm_mx(ones(M, K), gen.mx_pack_scales(la, K), ones(N, K),
                            gen.mx_pack_scales(lb, K), M, N, K)
    assert np.array_equal(got, np.full((M, N), 32 + 32 + 6 * 8.0))


def test_nan_scale_and_alpha_beta():
    M, N, K = 4, 3, 64
    la = np.full((M, 2), 127, np.uint8)
    la[2, 1] = 255                                   # NaN scale: row 2 becomes NaN
    lb = np.full((N, 2), 127, np.uint8)
    C0 = np.arange(M * N, dtype=np.float32).reshape(M, N)
    got, _ = oracle.gemm_mx(ones(M, K), gen.mx_pack_scales(la, K), ones(N, K),
                            gen.mx_pack_scales(lb, K), M, N, K, C0=C0, ldc=N, alpha=0.5,
                            beta=-2.0)
    assert np.isnan(got[2]).all()
    keep = [0, 1, 3]
    assert np.array_equal(got[keep], 0.5 * K - 2.0 * C0[keep].astype(np.float64))
