"""GPU parity of gemm_mx (MX operands: FP8 elements with E8M0 scales per 32 elements of K,
tcgen05.mma kind::mxf8f6f4 with block scales) against the fp64 MX oracle.

Definition: OCP Microscaling Formats (MX) v1.0 (a block of 32 elements along K shares a
scale 2^(X - 127)); the TMA page, 2.8, names block-scaled formats among Blackwell's
additions.  Bound (elementwise): |C - C_ref| <= 2*K*2^-24*|alpha|*sum_k |a_ik||b_jk| (the
scaled values) + 2^-8*|C_ref| (bf16 C) + 2^-23*|beta*C0|; bit-exact where every partial sum
is exact in fp32 (ones with power-of-two scales, small integers with unit scales)."""
import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_gb300 import inputs as gen
from tma_pipelined_tensor_gb300 import tg

from gpu_util import assert_within, c_to_f64, gemm_bound, stratified_positions

pytestmark = pytest.mark.gpu

ONE_E4M3, ONE_E5M2 = 0x38, 0x3C

# the two kernels: the CTA pair with 256 x 256 tiles (default) and one CTA per 128 x 128 tile
KERNELS = {"pair": dict(), "cta": dict(mma=1)}


def kernel_cfg(kernel, **kw):
    return tg.make_config(**KERNELS[kernel], **kw) if (KERNELS[kernel] or kw) else None


def to_dev_u8(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def run_mx(A, SA, B, SB, M, N, K, kind="e4m3", out="f32", alpha=1.0, beta=0.0, C0=None, cfg=None):
    """A and B may carry padding columns (row strides above K, 16-byte multiples)."""
    import torch
    dt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[out]
    per16 = 4 if out == "f32" else 8
    ldc = -(-N // per16) * per16             # C rows padded to 16 bytes
    Cbuf = torch.full((M, ldc), float("nan"), dtype=dt, device="cuda")
    Cd = Cbuf[:, :N]
    if C0 is not None:
        Cd.copy_(torch.from_numpy(C0.view(np.int16)).view(torch.bfloat16) if out == "bf16"
                 else torch.from_numpy(C0))
    Ad, Bd, SAd, SBd = to_dev_u8(A)[:, :K], to_dev_u8(B)[:, :K], to_dev_u8(SA), to_dev_u8(SB)
    st = tg.gemm_mx(Ad, SAd, Bd, SBd, Cd, alpha=alpha, beta=beta, kind=kind, config=cfg,
                    check=False)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    assert tg.tg_status_sync(None) == tg.TG_OK
    return c_to_f64(Cd)


def describe_mismatch(got, want):
    bad = np.argwhere(got != want)
    rows = sorted({int(i) for i, _ in bad})
    cols = sorted({int(j) for _, j in bad})
    return "%d mismatches; rows %s...; cols %s...; first got %s want %s" % (
        len(bad), rows[:12], cols[:12], got[tuple(bad[0])], want[tuple(bad[0])])


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 256, 512), (300, 520, 200),
                                   (512, 768, 640)])
def test_scale_layout_exact_on_ones(M, N, K, kernel):
    """Ones times power-of-two scales: every partial sum is exact, so C must equal the
    oracle bit for bit; a scale read from the wrong row, block or byte shows up here."""
    ld = -(-K // 16) * 16
    la, SA = gen.mx_scales(M, K, 11, 4, 124, 130)
    lb, SB = gen.mx_scales(N, K, 11, 5, 124, 130)
    A = np.full((M, ld), 0x7F, np.uint8)     # padding columns hold NaN: never read
    B = np.full((N, ld), 0x7F, np.uint8)
    A[:, :K] = ONE_E4M3
    B[:, :K] = ONE_E4M3
    got = run_mx(A, SA, B, SB, M, N, K, cfg=kernel_cfg(kernel))
    want, _ = oracle.gemm_mx(A, SA, B, SB, M, N, K, lda=ld, ldb=ld)
    assert np.array_equal(got, want), describe_mismatch(got, want)


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("kind", ["e4m3", "e5m2"])
def test_unit_scales_small_integers_bit_exact(kind, kernel):
    M, N, K = 256, 384, 1024
    one = ONE_E4M3 if kind == "e4m3" else ONE_E5M2
    v = gen.bf16_bits_to_f32(gen.small_int_matrix(M, K, 21, 0))    # integers in [-2, 2]
    w = gen.bf16_bits_to_f32(gen.small_int_matrix(N, K, 21, 1))
    A = gen.f32_to_f8_bits(v, kind == "e5m2")
    B = gen.f32_to_f8_bits(w, kind == "e5m2")
    assert np.abs(v).max() == 2.0
    SA = np.full(gen.mx_scale_bytes(M, K), 127, np.uint8)
    SB = np.full(gen.mx_scale_bytes(N, K), 127, np.uint8)
    got = run_mx(A, SA, B, SB, M, N, K, kind=kind, cfg=kernel_cfg(kernel))
    want, _ = oracle.gemm_mx(A, SA, B, SB, M, N, K, kind=kind)
    assert np.array_equal(got, want), describe_mismatch(got, want)
    assert np.array_equal(want, oracle.gemm(A, B, M, N, K, in_kind=kind)[0])


@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (129, 257, 96), (1000, 640, 1100),
                                   (1, 1, 1), (64, 1000, 33)])
@pytest.mark.parametrize("kind", ["e4m3", "e5m2"])
@pytest.mark.parametrize("kernel", sorted(KERNELS))
def test_random_within_bound(M, N, K, kind, kernel):
    ld = -(-K // 16) * 16                    # 16-byte rows; padding columns hold NaN
    A = gen.f8_matrix(M, K, M + K, 0, "normal", ld=ld, e5m2=(kind == "e5m2"))
    B = gen.f8_matrix(N, K, M + K, 1, "normal", ld=ld, e5m2=(kind == "e5m2"))
    _, SA = gen.mx_scales(M, K, M + K, 4)
    _, SB = gen.mx_scales(N, K, M + K, 5)
    got = run_mx(A, SA, B, SB, M, N, K, kind=kind, cfg=kernel_cfg(kernel))
    ref, mag = oracle.gemm_mx(A, SA, B, SB, M, N, K, kind=kind, lda=ld, ldb=ld)
    assert_within(got, ref, gemm_bound(ref, mag, K, 1.0, 0.0, None, False),
                  "mx %s %dx%dx%d" % (kind, M, N, K))


@pytest.mark.parametrize("kernel", sorted(KERNELS))
def test_alpha_beta_bf16_out(kernel):
    M, N, K = 333, 500, 288
    A = gen.f8_matrix(M, K, 7, 0, "normal")
    B = gen.f8_matrix(N, K, 7, 1, "normal")
    _, SA = gen.mx_scales(M, K, 7, 4)
    _, SB = gen.mx_scales(N, K, 7, 5)
    C0 = gen.bf16_matrix(M, N, 7, 2, "uniform")
    got = run_mx(A, SA, B, SB, M, N, K, out="bf16", alpha=-0.75, beta=0.5, C0=C0,
                 cfg=kernel_cfg(kernel))
    ref, mag = oracle.gemm_mx(A, SA, B, SB, M, N, K, C0=C0, ldc=N, alpha=-0.75, beta=0.5)
    c0v = gen.bf16_bits_to_f32(C0).astype(np.float64)
    assert_within(got, ref, gemm_bound(ref, mag, K, -0.75, 0.5, c0v, True), "mx alpha/beta")


@pytest.mark.parametrize("kernel", sorted(KERNELS))
@pytest.mark.parametrize("stages", [2, 3, 4, 5])
def test_ring_depths(stages, kernel):
    M, N, K = 640, 384, 1536
    A = gen.f8_matrix(M, K, 9, 0, "normal")
    B = gen.f8_matrix(N, K, 9, 1, "normal")
    _, SA = gen.mx_scales(M, K, 9, 4)
    _, SB = gen.mx_scales(N, K, 9, 5)
    got = run_mx(A, SA, B, SB, M, N, K, cfg=kernel_cfg(kernel, stages=stages))
    ref, mag = oracle.gemm_mx(A, SA, B, SB, M, N, K)
    assert_within(got, ref, gemm_bound(ref, mag, K, 1.0, 0.0, None, False), "stages %d" % stages)
    st, last = tg.tg_gemm_last_plan()
    if kernel == "pair":
        assert (last.stages, last.mma, last.tile_n, last.cluster) == (stages, 2, 256, 2)
    else:
        assert (last.stages, last.mma, last.tile_n, last.cluster) == (stages, 1, 128, 1)


@pytest.mark.parametrize("kernel", sorted(KERNELS))
def test_many_tiles_per_cluster(kernel):
    """Four CTAs take all the tiles (10 per CTA pair, 20 per lone CTA): the pair kernel's
    single accumulator is handed back and forth between the MMA issuer and the epilogue
    many times, and the ring's phases wrap inside and across tiles."""
    M, N, K = 1024, 1280, 640
    A = gen.f8_matrix(M, K, 13, 0, "normal")
    B = gen.f8_matrix(N, K, 13, 1, "normal")
    _, SA = gen.mx_scales(M, K, 13, 4)
    _, SB = gen.mx_scales(N, K, 13, 5)
    got = run_mx(A, SA, B, SB, M, N, K, out="bf16", cfg=kernel_cfg(kernel, max_ctas=4, stages=3))
    ref, mag = oracle.gemm_mx(A, SA, B, SB, M, N, K)
    assert_within(got, ref, gemm_bound(ref, mag, K, 1.0, 0.0, None, True), "many tiles")
    st, last = tg.tg_gemm_last_plan()
    assert last.grid == 4


def test_full_size_stratified_default_launch():
    """8192^3 MXE4M3 with the benchmark's inputs and scales, default launch (CTA pairs,
    256 x 256 tiles, single accumulator): two outputs in every (128-row tile, 32-row
    epilogue quarter, 64-column chunk) cell of the tiling against the oracle's entries."""
    import torch
    name = "gemm_8192_mxe4m3"
    M, N, K = gen.GEMM_WORKLOADS[name][:3]
    A, B, _ = gen.gemm_inputs(name)
    _, SA, _, SB = gen.gemm_mx_scale_inputs(name)
    got = run_mx(A, SA, B, SB, M, N, K, out="bf16")
    st, last = tg.tg_gemm_last_plan()
    assert (last.mma, last.tile_n, last.cluster) == (2, 256, 2)
    torch.cuda.empty_cache()
    ii, jj = stratified_positions(M, N, 256, seed=3)
    assert len(ii) == 2 * (M // 32) * (N // 64)
    ref, mag = oracle.gemm_mx_entries(A, SA, B, SB, M, N, K, ii, jj)
    assert_within(got[ii, jj], ref, gemm_bound(ref, mag, K, 1.0, 0.0, None, True),
                  "mx 8192^3 stratified")


def test_default_launch_is_the_pair():
    M, N, K = 512, 512, 256
    A = np.full((M, K), ONE_E4M3, np.uint8)
    B = np.full((N, K), ONE_E4M3, np.uint8)
    SA = np.full(gen.mx_scale_bytes(M, K), 127, np.uint8)
    SB = np.full(gen.mx_scale_bytes(N, K), 127, np.uint8)
    got = run_mx(A, SA, B, SB, M, N, K)
    assert np.all(got == K)
    st, last = tg.tg_gemm_last_plan()
    assert (last.mma, last.tile_n, last.cluster, last.stages) == (2, 256, 2, 4)


def test_refusals():
    import torch
    A = torch.zeros((256, 256), dtype=torch.uint8, device="cuda")
    S = torch.full((gen.mx_scale_bytes(256, 256),), 127, dtype=torch.uint8, device="cuda")
    C = torch.zeros((256, 256), dtype=torch.float32, device="cuda")
    L = tg.TG_C_F32 | tg.TG_IN_MXE4M3
    call = lambda sa=S.data_ptr(), layout=L, cfg=None: tg.gemm_mx_raw(
        256, 256, 256, A.data_ptr(), 256, sa, A.data_ptr(), 256, S.data_ptr(), C.data_ptr(), 256,
        1.0, 0.0, layout, cfg)
    assert call(sa=None) == tg.TG_ERR_INVALID_VALUE
    assert call(sa=S.data_ptr() + 8) == tg.TG_ERR_MISALIGNED
    host = torch.full((S.numel(),), 127, dtype=torch.uint8, pin_memory=True)
    assert call(sa=host.data_ptr()) == tg.TG_ERR_INVALID_VALUE
    assert call(layout=tg.TG_C_F32 | tg.TG_IN_E4M3) == tg.TG_ERR_INVALID_VALUE
    assert call(cfg=tg.make_config(mma=3)) == tg.TG_ERR_INVALID_VALUE
    assert call(cfg=tg.make_config(mma=2, tile_n=224)) == tg.TG_ERR_INVALID_VALUE
    assert call(cfg=tg.make_config(mma=1, cluster=2)) == tg.TG_ERR_INVALID_VALUE
    assert call(cfg=tg.make_config(schedule=2)) == tg.TG_ERR_INVALID_VALUE
    assert call(cfg=tg.make_config(stages=6)) == tg.TG_ERR_UNSUPPORTED   # does not fit
    assert call(cfg=tg.make_config(stages=6, mma=1)) == tg.TG_ERR_UNSUPPORTED
    assert tg.gemm_bf16(256, 256, 256, A.data_ptr(), 256, A.data_ptr(), 256, C.data_ptr(), 256,
                        1.0, 0.0, L, None) == tg.TG_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert tg.tg_status_sync(None) == tg.TG_OK
