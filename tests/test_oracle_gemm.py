"""Pins of the oracle's GEMM against facts fixed by mathematics, not by the oracle.

GEMM definition: "GEMM: la moltiplicazione di matrici sull'hardware", section "Il
conto, e il problema della versione ingenua" (C_ij = sum_k A_ik B_kj) and section "I
tensor core" (C <- alpha*A*B + beta*C, 16-bit inputs, 32-bit accumulation).  Storage
convention: A is M x K row-major, B is stored N x K row-major (its transpose is the
mathematical operand), C is M x N row-major.
"""
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_gb300 import inputs as gen

BF16_ONE = 0x3F80


def bf16_value(bits: int) -> Fraction:
    """Exact rational value of a bf16 pattern (decoded via struct, not the oracle)."""
    f = struct.unpack(">f", struct.pack(">I", (int(bits) & 0xFFFF) << 16))[0]
    return Fraction(f)


def to_f64(bits):
    return gen.bf16_bits_to_f32(bits).astype(np.float64)


def test_hand_worked_example_checks_operand_orientation():
    # A = [[1,2,3],[4,5,6]], B stored = [[1,0,-1],[2,1,0]]  ->  C = A * B_stored^T
    # C00 = 1*1 + 2*0 + 3*(-1) = -2, C01 = 1*2 + 2*1 + 3*0 = 4,
    # C10 = 4*1 + 5*0 + 6*(-1) = -2, C11 = 4*2 + 5*1 + 6*0 = 13.
    A = gen.f32_to_bf16_bits(np.array([[1, 2, 3], [4, 5, 6]], dtype=np.float32))
    B = gen.f32_to_bf16_bits(np.array([[1, 0, -1], [2, 1, 0]], dtype=np.float32))
    C, mag = oracle.gemm(A, B, 2, 2, 3)
    assert C.tolist() == [[-2.0, 4.0], [-2.0, 13.0]]
    assert mag.tolist() == [[4.0, 4.0], [10.0, 13.0]]


@pytest.mark.parametrize("M,N,K", [(5, 7, 300), (130, 257, 65), (1, 1, 1), (3, 2, 4096)])
def test_ones_times_ones_is_k(M, N, K):
    A = np.full((M, K), BF16_ONE, dtype=np.uint16)
    B = np.full((N, K), BF16_ONE, dtype=np.uint16)
    C, mag = oracle.gemm(A, B, M, N, K)
    assert np.all(C == K) and np.all(mag == K)


def test_identity_b_returns_alpha_a():
    M, K = 33, 40
    A = gen.bf16_matrix(M, K, 11, 0, "normal")
    B = np.zeros((K, K), dtype=np.uint16)
    B[np.arange(K), np.arange(K)] = BF16_ONE
    C, _ = oracle.gemm(A, B, M, K, K, alpha=0.5)
    assert np.array_equal(C, 0.5 * to_f64(A))


def test_rank_one_with_beta():
    M, N, K = 9, 11, 6
    u = gen.bf16_matrix(M, 1, 12, 0, "uniform")[:, 0]
    v = gen.bf16_matrix(N, 1, 12, 1, "uniform")[:, 0]
    A = np.zeros((M, K), dtype=np.uint16)
    B = np.zeros((N, K), dtype=np.uint16)
    A[:, 0], B[:, 0] = u, v
    C0 = gen.bf16_matrix(M, N, 12, 2, "uniform")
    C, _ = oracle.gemm(A, B, M, N, K, C0=C0, alpha=2.0, beta=0.25)
    for i in range(M):
        for j in range(N):
            want = 2 * bf16_value(u[i]) * bf16_value(v[j]) + Fraction(1, 4) * bf16_value(C0[i, j])
            assert C[i, j] == float(want)


@pytest.mark.parametrize("cdt", ["f32", "bf16"])
def test_alpha_zero_beta_one_returns_c0(cdt):
    M, N, K = 17, 19, 23
    A = gen.bf16_matrix(M, K, 13, 0, "normal")
    B = gen.bf16_matrix(N, K, 13, 1, "normal")
    if cdt == "bf16":
        C0 = gen.bf16_matrix(M, N, 13, 2, "uniform")
        want = to_f64(C0)
    else:
        C0 = gen.uniform(13, 2, M * N).astype(np.float32).reshape(M, N)
        want = C0.astype(np.float64)
    C, _ = oracle.gemm(A, B, M, N, K, C0=C0, alpha=0.0, beta=1.0)
    assert np.array_equal(C, want)


def test_beta_zero_never_reads_c():
    M, N, K = 8, 8, 8
    A = gen.bf16_matrix(M, K, 14, 0, "normal")
    B = gen.bf16_matrix(N, K, 14, 1, "normal")
    C0 = np.full((M, N), np.nan, dtype=np.float32)
    C, _ = oracle.gemm(A, B, M, N, K, C0=C0, beta=0.0)
    assert np.isfinite(C).all()


def test_brute_force_8x8x8_exact_rationals():
    M = N = K = 8
    A = gen.bf16_matrix(M, K, 15, 0, "uniform")
    B = gen.bf16_matrix(N, K, 15, 1, "uniform")
    C0 = gen.bf16_matrix(M, N, 15, 2, "uniform")
    C, mag = oracle.gemm(A, B, M, N, K, C0=C0, alpha=1.5, beta=-0.75)
    for i in range(M):
        for j in range(N):
            s = sum(bf16_value(A[i, k]) * bf16_value(B[j, k]) for k in range(K))
            m = sum(abs(bf16_value(A[i, k]) * bf16_value(B[j, k])) for k in range(K))
            want = Fraction(3, 2) * s - Fraction(3, 4) * bf16_value(C0[i, j])
            assert abs(C[i, j] - float(want)) <= 1e-15 * float(m + 1)
            assert abs(mag[i, j] - float(m)) <= 1e-15 * float(m)


def test_matches_library_matmul_in_fp64():
    M, N, K = 64, 48, 40
    A = gen.bf16_matrix(M, K, 16, 0, "normal")
    B = gen.bf16_matrix(N, K, 16, 1, "normal")
    C, mag = oracle.gemm(A, B, M, N, K)
    ref = to_f64(A) @ to_f64(B).T
    assert np.all(np.abs(C - ref) <= 1e-13 * mag)
    assert np.allclose(mag, np.abs(to_f64(A)) @ np.abs(to_f64(B)).T, rtol=1e-14, atol=0)


def _blocked(A, B, T):
    """Tile loop over T x T blocks of C with K blocks (the page's blocked scheme)."""
    M, K = A.shape
    N = B.shape[0]
    C = np.zeros((M, N))
    for i in range(0, M, T):
        for j in range(0, N, T):
            acc = np.zeros((min(T, M - i), min(T, N - j)))
            for k in range(0, K, T):
                acc += A[i:i + T, k:k + T] @ B[j:j + T, k:k + T].T
            C[i:i + T, j:j + T] = acc
    return C


@pytest.mark.parametrize("T", [1, 8, 32])
def test_blocked_equals_direct(T):
    M, N, K = 96, 64, 80
    A = gen.bf16_matrix(M, K, 17, 0, "normal")
    B = gen.bf16_matrix(N, K, 17, 1, "normal")
    C, mag = oracle.gemm(A, B, M, N, K)
    assert np.all(np.abs(_blocked(to_f64(A), to_f64(B), T) - C) <= 1e-13 * mag)


def test_leading_dimensions_skip_padding():
    M, N, K = 21, 13, 37
    A = gen.bf16_matrix(M, K, 18, 0, "normal", ld=K + 11)
    B = gen.bf16_matrix(N, K, 18, 1, "normal", ld=K + 3)
    C0 = gen.bf16_matrix(M, N, 18, 2, "uniform", ld=N + 8)
    C, _ = oracle.gemm(A, B, M, N, K, lda=K + 11, ldb=K + 3, C0=C0, ldc=N + 8, beta=0.5)
    Cc, _ = oracle.gemm(A[:, :K].copy(), B[:, :K].copy(), M, N, K,
                        C0=C0[:, :N].copy(), beta=0.5)
    assert np.isfinite(C).all() and np.array_equal(C, Cc)


def test_entries_and_row_bands_agree_with_full():
    M, N, K = 50, 70, 33
    A = gen.bf16_matrix(M, K, 19, 0, "normal")
    B = gen.bf16_matrix(N, K, 19, 1, "normal")
    C0 = gen.uniform(19, 2, M * N).astype(np.float32).reshape(M, N)
    full, mag = oracle.gemm(A, B, M, N, K, C0=C0, beta=-1.0)
    band, _ = oracle.gemm(A, B, M, N, K, C0=C0, beta=-1.0, rows=(10, 23))
    assert np.array_equal(band, full[10:23])
    rng = np.random.default_rng(0)
    ii, jj = rng.integers(0, M, 200), rng.integers(0, N, 200)
    e, em = oracle.gemm_entries(A, B, K, ii, jj, C0=C0, ldc=N, beta=-1.0)
    assert np.array_equal(e, full[ii, jj]) and np.array_equal(em, mag[ii, jj])


def test_absprod_is_gemm_of_absolute_values():
    M, N, K = 12, 14, 31
    A = gen.bf16_matrix(M, K, 20, 0, "normal")
    B = gen.bf16_matrix(N, K, 20, 1, "normal")
    _, mag = oracle.gemm(A, B, M, N, K)
    absA, absB = A & np.uint16(0x7FFF), B & np.uint16(0x7FFF)
    C_abs, _ = oracle.gemm(absA, absB, M, N, K)
    assert np.array_equal(mag, C_abs)


def test_k_zero_gives_beta_c():
    M, N = 4, 5
    A = np.zeros((M, 1), dtype=np.uint16)
    B = np.zeros((N, 1), dtype=np.uint16)
    C0 = gen.uniform(21, 2, M * N).astype(np.float32).reshape(M, N)
    C, _ = oracle.gemm(A, B, M, N, 0, lda=1, ldb=1, C0=C0, beta=2.0)
    assert np.array_equal(C, 2.0 * C0.astype(np.float64))


def test_hand_worked_example_in_every_storage():
    # the same product as the hand-worked example, with A and/or B stored MN-major:
    # A (2x3) M-major is stored as its 3 x 2 transpose; the K x N operand (3 x 2) N-major is
    # stored as written, [[1,2],[0,1],[-1,0]]
    A_k = gen.f32_to_bf16_bits(np.array([[1, 2, 3], [4, 5, 6]], dtype=np.float32))
    A_m = gen.f32_to_bf16_bits(np.array([[1, 4], [2, 5], [3, 6]], dtype=np.float32))
    B_k = gen.f32_to_bf16_bits(np.array([[1, 0, -1], [2, 1, 0]], dtype=np.float32))
    B_n = gen.f32_to_bf16_bits(np.array([[1, 2], [0, 1], [-1, 0]], dtype=np.float32))
    for A, a_mn in [(A_k, False), (A_m, True)]:
        for B, b_mn in [(B_k, False), (B_n, True)]:
            C, _ = oracle.gemm(A, B, 2, 2, 3, a_mn=a_mn, b_mn=b_mn)
            assert C.tolist() == [[-2.0, 4.0], [-2.0, 13.0]], (a_mn, b_mn)


@pytest.mark.parametrize("a_mn,b_mn", [(True, False), (False, True), (True, True)])
def test_mn_major_storage_matches_numpy(a_mn, b_mn):
    M, N, K = 37, 29, 45
    ld_a = (M + 3) if a_mn else (K + 5)
    ld_b = (N + 7) if b_mn else (K + 2)
    A = gen.bf16_matrix(K if a_mn else M, M if a_mn else K, 23, 0, "normal", ld=ld_a)
    B = gen.bf16_matrix(K if b_mn else N, N if b_mn else K, 23, 1, "normal", ld=ld_b)
    Af = to_f64(A)[:, :(M if a_mn else K)]
    Bf = to_f64(B)[:, :(N if b_mn else K)]
    A_math = Af.T if a_mn else Af            # M x K
    B_math = Bf if b_mn else Bf.T            # K x N
    C, mag = oracle.gemm(A, B, M, N, K, lda=ld_a, ldb=ld_b, a_mn=a_mn, b_mn=b_mn)
    assert np.all(np.abs(C - A_math @ B_math) <= 1e-13 * mag)
    e, _ = oracle.gemm_entries(A, B, K, [0, M - 1, 5], [N - 1, 0, 7], lda=ld_a, ldb=ld_b,
                               a_mn=a_mn, b_mn=b_mn)
    assert np.array_equal(e, C[[0, M - 1, 5], [N - 1, 0, 7]])


def test_f16_decoder_matches_library_on_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_value(int(b)) for b in bits])
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all(), np.flatnonzero(~same)[:5]


def test_f16_operands_match_numpy():
    M, N, K = 40, 36, 52
    A = gen.f16_matrix(M, K, 24, 0, "normal")
    B = gen.f16_matrix(N, K, 24, 1, "normal")
    Af = A.view(np.float16).astype(np.float64)
    Bf = B.view(np.float16).astype(np.float64)
    C, mag = oracle.gemm(A, B, M, N, K, in_f16=True)
    assert np.all(np.abs(C - Af @ Bf.T) <= 1e-13 * mag)
    # the same bits read as bf16 give a different product: the flag is honoured
    Cb, _ = oracle.gemm(A, B, M, N, K)
    assert not np.allclose(Cb, C)


def test_f16_c0():
    M, N, K = 6, 10, 4
    A = np.zeros((M, K), dtype=np.uint16)
    B = np.zeros((N, K), dtype=np.uint16)
    C0 = gen.f16_matrix(M, N, 25, 2, "uniform")
    C, _ = oracle.gemm(A, B, M, N, K, C0=C0, beta=1.0, in_f16=True, c_f16=True)
    assert np.array_equal(C, C0.view(np.float16).astype(np.float64))


@pytest.mark.parametrize("e5m2", [False, True])
def test_f8_decoders_match_library_on_every_pattern(e5m2):
    import torch
    dt = torch.float8_e5m2 if e5m2 else torch.float8_e4m3fn
    want = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(dt).to(torch.float64).numpy()
    got = np.array([oracle.f8_value(b, e5m2) for b in range(256)])
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all(), np.flatnonzero(~same)[:5]


@pytest.mark.parametrize("kind", ["e4m3", "e5m2"])
def test_f8_operands_match_torch(kind):
    import torch
    M, N, K = 33, 40, 96
    A = gen.f8_matrix(M, K, 26, 0, "normal", e5m2=(kind == "e5m2"))
    B = gen.f8_matrix(N, K, 26, 1, "normal", e5m2=(kind == "e5m2"))
    dt = torch.float8_e5m2 if kind == "e5m2" else torch.float8_e4m3fn
    Af = torch.from_numpy(A).view(dt).to(torch.float64).numpy()
    Bf = torch.from_numpy(B).view(dt).to(torch.float64).numpy()
    C, mag = oracle.gemm(A, B, M, N, K, in_kind=kind)
    assert np.all(np.abs(C - Af @ Bf.T) <= 1e-13 * mag)


def _f32_bits(x):
    return int(np.array([x], dtype=np.float32).view(np.uint32)[0])


def test_tf32_truncation_pins():
    # The GEMM page's tensor-core section: tf32 keeps 10 of float32's 23 mantissa bits by
    # truncation.  1 + 2^-12 and 1 + 2^-11 + 2^-12 (which rounding would take up to
    # 1 + 2^-10) both become 1; 1 + 2^-10 is already tf32.
    assert oracle.tf32_value(_f32_bits(1 + 2.0 ** -12)) == 1.0
    assert oracle.tf32_value(_f32_bits(1 + 2.0 ** -11 + 2.0 ** -12)) == 1.0
    assert oracle.tf32_value(_f32_bits(1 + 2.0 ** -10)) == 1 + 2.0 ** -10
    assert oracle.tf32_value(_f32_bits(-(1 + 2.0 ** -12))) == -1.0     # toward zero
    assert oracle.tf32_value(0x7F7FFFFF) == (2 - 2.0 ** -10) * 2.0 ** 127
    assert oracle.tf32_value(0x00001FFF) == 0.0                         # subnormal low bits
    assert oracle.tf32_value(0x00002001) == 2.0 ** -136
    assert oracle.tf32_value(0x7F800000) == float("inf")


def test_tf32_truncates_both_operands():
    x = np.array([[1 + 2.0 ** -12]], dtype=np.float32)
    three = np.array([[3.0]], dtype=np.float32)
    C, _ = oracle.gemm(x, x, 1, 1, 1, in_kind="tf32")
    assert C[0, 0] == 1.0
    C, _ = oracle.gemm(three, x, 1, 1, 1, in_kind="tf32")
    assert C[0, 0] == 3.0


@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (True, True)])
def test_tf32_exact_inputs_match_integer_matmul(a_mn, b_mn):
    # integers of at most 11 significant bits are exact in tf32, so the product is the
    # plain integer matrix product
    M, N, K = 19, 23, 37
    rng = np.random.default_rng(5)
    A = rng.integers(-2048, 2049, size=(M, K))
    B = rng.integers(-2048, 2049, size=(N, K))
    As = np.ascontiguousarray(A.T if a_mn else A).astype(np.float32)
    Bs = np.ascontiguousarray(B.T if b_mn else B).astype(np.float32)
    C, mag = oracle.gemm(As, Bs, M, N, K, a_mn=a_mn, b_mn=b_mn, in_kind="tf32")
    assert np.array_equal(C, (A @ B.T).astype(np.float64))
    assert np.array_equal(mag, (np.abs(A) @ np.abs(B).T).astype(np.float64))
