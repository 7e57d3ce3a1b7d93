"""GPU parity of gemm_bf16 against the fp64 oracle.

Bound (elementwise): |C - C_ref| <= 2*K*2^-24*|alpha|*(|A||B|)_ij + 2^-8*|C_ref_ij| (bf16
out only) + 2^-23*|beta*C0_ij|.  Definition: "GEMM: la moltiplicazione di matrici
sull'hardware", sections "Il conto" and "I tensor core" (C <- alpha*A*B + beta*C, 16-bit
inputs, fp32 accumulation)."""
import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_gb300 import inputs as gen
from tma_pipelined_tensor_gb300 import tg

from gpu_util import (assert_within, c0_values, c_to_f64, gemm_bound, stratified_positions, to_device,
                      to_device_bf16)

pytestmark = pytest.mark.gpu


GUARD_ROWS = 8  # sentinel rows allocated below C: the kernel must never write them


def device_c(M, N, ldc, out_bf16, C0=None, fill=np.nan):
    """M x ldc device C (from C0 or filled), followed by GUARD_ROWS sentinel rows."""
    import torch
    dt = torch.bfloat16 if out_bf16 else torch.float32
    buf = torch.full((M + GUARD_ROWS, ldc), fill, dtype=dt, device="cuda")
    if C0 is not None:
        buf[:M] = to_device_bf16(C0) if out_bf16 else to_device(C0)
    return buf[:M]


def guard_rows_untouched(C):
    import torch
    M = C.shape[0]
    full = torch.as_strided(C, (M + GUARD_ROWS, C.shape[1]), C.stride())
    return bool(torch.isnan(full[M:].float()).all())


def run_gemm(A, B, M, N, K, lda, ldb, ldc, out_bf16, alpha=1.0, beta=0.0, C0=None, cfg=None):
    Ad = to_device_bf16(A)
    Bd = to_device_bf16(B)
    Cd = device_c(M, N, ldc, out_bf16, C0)
    layout = tg.TG_C_BF16 if out_bf16 else tg.TG_C_F32
    st = tg.gemm_bf16_ex(M, N, K, Ad.data_ptr(), lda, Bd.data_ptr(), ldb, Cd.data_ptr(), ldc,
                         alpha, beta, layout, cfg, None)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    assert tg.tg_status_sync(None) == tg.TG_OK
    assert guard_rows_untouched(Cd)
    return c_to_f64(Cd)


def full_check(M, N, K, out_bf16, alpha=1.0, beta=0.0, seed=0, pad=(0, 0, 0), cfg=None,
               dist="normal"):
    # leading dimensions: the smallest legal ones (16-byte rows) plus the requested padding
    rup = lambda x, m: -(-x // m) * m
    lda, ldb = rup(K, 8) + pad[0], rup(K, 8) + pad[1]
    ldc = rup(N, 8 if out_bf16 else 4) + pad[2]
    A = gen.bf16_matrix(M, K, seed, 0, dist, ld=lda)
    B = gen.bf16_matrix(N, K, seed, 1, dist, ld=ldb)
    C0 = None
    if beta != 0.0 or ldc > N:
        if out_bf16:
            C0 = gen.bf16_matrix(M, N, seed, 2, "uniform", ld=ldc)
        else:
            C0 = np.full((M, ldc), np.nan, dtype=np.float32)
            C0[:, :N] = gen.uniform(seed, 2, M * N).astype(np.float32).reshape(M, N)
    got = run_gemm(A, B, M, N, K, lda, ldb, ldc, out_bf16, alpha, beta, C0, cfg)
    ref, mag = oracle.gemm(A, B, M, N, K, lda, ldb, C0, ldc, alpha, beta)
    c0v = c0_values(C0)[:, :N] if (C0 is not None) else None
    bound = gemm_bound(ref, mag, K, alpha, beta, c0v, out_bf16)
    assert_within(got[:, :N], ref, bound, "M=%d N=%d K=%d" % (M, N, K))
    if ldc > N:  # columns beyond N are never written
        before = c0_values(C0)[:, N:]
        assert np.array_equal(np.isnan(got[:, N:]), np.isnan(before))
        assert np.array_equal(np.nan_to_num(got[:, N:]), np.nan_to_num(before))
    return got, ref


@pytest.mark.parametrize("out_bf16", [False, True])
def test_workload_256_full(out_bf16):
    # 256^3, U[-1,1], seed 0, alpha = 1, beta = 0 (fp32 out in the workload; bf16 too)
    full_check(256, 256, 256, out_bf16, seed=0, dist="uniform")


@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (128, 256, 64), (1, 1, 1), (129, 257, 65),
                                   (1000, 24, 8), (64, 1000, 1000)])
@pytest.mark.parametrize("out_bf16", [False, True])
def test_ragged_small(M, N, K, out_bf16):
    full_check(M, N, K, out_bf16, seed=M + N + K)


@pytest.mark.parametrize("out_bf16", [False, True])
def test_alpha_beta_and_padded_leading_dims(out_bf16):
    full_check(333, 500, 136, out_bf16, alpha=-0.75, beta=0.5, pad=(8, 24, 8 if out_bf16 else 4),
               seed=5)


@pytest.mark.parametrize("out_bf16", [False, True])
def test_k_zero_scales_c(out_bf16):
    import torch
    M, N, ldc = 200, 300, 304
    C0 = (gen.bf16_matrix(M, N, 9, 2, "uniform", ld=ldc) if out_bf16
          else np.pad(gen.uniform(9, 2, M * N).astype(np.float32).reshape(M, N),
                      ((0, 0), (0, ldc - N)), constant_values=np.nan))
    Cd = device_c(M, N, ldc, out_bf16, C0)
    st = tg.gemm_bf16(M, N, 0, None, 0, None, 0, Cd.data_ptr(), ldc, 1.0, 0.25,
                      tg.TG_C_BF16 if out_bf16 else tg.TG_C_F32, None)
    assert st == tg.TG_OK and tg.tg_status_sync(None) == tg.TG_OK
    got = c_to_f64(Cd)
    assert np.array_equal(got[:, :N], 0.25 * c0_values(C0)[:, :N])
    assert np.isnan(got[:, N:]).all()


def test_beta_zero_ignores_nan_in_c():
    got, _ = full_check(130, 140, 70, False, seed=3)   # C starts as NaN, beta = 0
    assert np.isfinite(got).all()


@pytest.mark.parametrize("out_bf16", [False, True])
def test_exact_integer_regime_bit_exact(out_bf16):
    # entries in {-2..2}, K = 4096: every partial sum is an integer below 2^24, so the fp32
    # accumulation is exact; |C| <= 256 is not guaranteed, so bf16 output is compared
    # against the oracle rounded the same way only where |C| <= 256.
    M, N, K = 256, 512, 4096
    A = gen.small_int_matrix(M, K, 31, 0)
    B = gen.small_int_matrix(N, K, 31, 1)
    got = run_gemm(A, B, M, N, K, K, K, N, out_bf16)
    ref, _ = oracle.gemm(A, B, M, N, K)
    if out_bf16:
        small = np.abs(ref) <= 256
        assert np.array_equal(got[small], ref[small])
    else:
        assert np.array_equal(got, ref)


# (tile_n, stages, cluster, mma): per-CTA MMAs with and without B multicast, and the
# CTA-pair MMA (256-row tiles, half of B per CTA) over the 2..6 stage range.
SWEEP = ([(256, s, c, 1) for s in (2, 3, 4) for c in (1, 2)]
         + [(128, s, c, 1) for s in (2, 4, 6) for c in (1, 2)]
         + [(256, s, 2, 2) for s in (2, 3, 4, 5, 6)] + [(128, s, 2, 2) for s in (2, 4, 6)])


@pytest.mark.parametrize("tile_n,stages,cluster,mma", SWEEP)
def test_config_sweep(tile_n, stages, cluster, mma):
    cfg = tg.make_config(tile_n=tile_n, stages=stages, cluster=cluster, mma=mma)
    full_check(520, 1000, 300, True, seed=tile_n + stages + cluster, cfg=cfg, beta=0.5)
    full_check(384, 512, 64, False, seed=7, cfg=cfg)


@pytest.mark.parametrize("group_m,max_ctas", [(1, 0), (3, 0), (16, 7), (64, 2)])
@pytest.mark.parametrize("mma", [1, 2])
def test_schedule_knobs(group_m, max_ctas, mma):
    cfg = tg.make_config(group_m=group_m, max_ctas=max_ctas, mma=mma)
    full_check(1100, 1300, 200, True, seed=11, cfg=cfg)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (129, 257, 65), (257, 129, 8), (600, 40, 1000)])
@pytest.mark.parametrize("out_bf16", [False, True])
def test_pair_ragged_small(M, N, K, out_bf16):
    full_check(M, N, K, out_bf16, seed=M * 3 + N + K, beta=0.25, cfg=tg.make_config(mma=2))


# Stream-K: shapes whose tiles split over one to several clusters (few tiles, long K),
# with ragged edges, beta != 0 and both MMA kinds.
SK_SHAPES = [(1100, 1300, 2000), (4096, 1024, 1024), (300, 520, 4096), (1, 8, 640),
             (2048, 2048, 256), (129, 264, 4100)]


@pytest.mark.parametrize("M,N,K", SK_SHAPES)
@pytest.mark.parametrize("mma", [1, 2])
@pytest.mark.parametrize("out_bf16", [False, True])
def test_stream_k(M, N, K, mma, out_bf16):
    cfg = tg.make_config(mma=mma, schedule=2)
    st, plan = tg.tg_gemm_plan_for(M, N, K, tg.TG_C_BF16 if out_bf16 else tg.TG_C_F32, cfg, 0)
    assert st == tg.TG_OK
    full_check(M, N, K, out_bf16, seed=M + 7 * N + K + mma, beta=0.5, alpha=1.25, cfg=cfg)


@pytest.mark.parametrize("mma", [1, 2])
def test_stream_k_on_a_capped_grid(mma):
    # max_ctas caps the persistent grid; the stream-K shares spread over the clusters left
    cfg = tg.make_config(mma=mma, schedule=2, max_ctas=14)
    st, plan = tg.tg_gemm_plan_for(1100, 1300, 2000, tg.TG_C_BF16, cfg, 0)
    assert st == tg.TG_OK and plan.sk_iters > 0 and plan.grid <= 14
    full_check(1100, 1300, 2000, True, seed=71 + mma, beta=0.5, cfg=cfg)


def test_stream_k_on_two_streams_at_once():
    """Concurrent stream-K GEMMs on two streams use separate workspaces."""
    import torch
    M, N, K = 1100, 1300, 2000
    cfg = tg.make_config(schedule=2)
    probs = []
    for seed in (51, 52):
        A = gen.bf16_matrix(M, K, seed, 0, "normal")
        B = gen.bf16_matrix(N, K, seed, 1, "normal")
        probs.append((A, B, to_device_bf16(A), to_device_bf16(B),
                      torch.empty((M, N), dtype=torch.float32, device="cuda")))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for _ in range(5):
        for (A, B, Ad, Bd, Cd), s in zip(probs, streams):
            st = tg.gemm_bf16_ex(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, Cd.data_ptr(), N,
                                 1.0, 0.0, tg.TG_C_F32, cfg, ctypes_stream(s))
            assert st == tg.TG_OK
    torch.cuda.synchronize()
    assert tg.tg_status_sync(None) == tg.TG_OK
    for A, B, Ad, Bd, Cd in probs:
        ref, mag = oracle.gemm(A, B, M, N, K)
        assert_within(Cd.cpu().numpy().astype(np.float64), ref,
                      gemm_bound(ref, mag, K, 1.0, 0.0, None, False), "two streams")


def ctypes_stream(s):
    import ctypes
    return ctypes.c_void_p(s.cuda_stream)


# Stream-K tiles finished in the fast epilogue (beta = 0, 16-bit C, whole tiles): the
# other clusters' partials are summed chunk by chunk.  (512, 512, 8192) splits each of its
# four tiles over about nineteen clusters; (2048, 2000, 4096) mixes whole tiles with a
# ragged last tile column that takes the general path.
@pytest.mark.parametrize("M,N,K", [(2048, 2048, 4096), (512, 512, 8192), (2048, 2000, 4096),
                                   (1024, 1024, 1000)])
@pytest.mark.parametrize("mma", [1, 2])
def test_stream_k_fast_epilogue(M, N, K, mma):
    cfg = tg.make_config(mma=mma, schedule=2)
    full_check(M, N, K, True, seed=M + N + K + mma, alpha=0.75, cfg=cfg)


@pytest.mark.parametrize("mma", [1, 2])
def test_stream_k_fast_epilogue_exact_integers(mma):
    # integer partials stay exact through the fp32 workspace and the sum of up to nineteen
    # of them (each tile spans about nineteen clusters' shares); the bf16 result is the
    # oracle's value wherever that is a bf16 number
    M, N, K = 512, 512, 4096
    A = gen.small_int_matrix(M, K, 35, 0)
    B = gen.small_int_matrix(N, K, 35, 1)
    cfg = tg.make_config(mma=mma, schedule=2)
    ref, _ = oracle.gemm(A, B, M, N, K)
    got = run_gemm(A, B, M, N, K, K, K, N, True, cfg=cfg)
    small = np.abs(ref) <= 256
    assert small.mean() > 0.9
    assert np.array_equal(got[small], ref[small])


@pytest.mark.parametrize("mma", [1, 2])
def test_stream_k_exact_integers_and_repeat(mma):
    # integer partial sums stay exact through the fp32 workspace; a second launch on the
    # same workspace (new launch number) must not pick up the first launch's partials
    M, N, K = 512, 768, 4096
    A = gen.small_int_matrix(M, K, 33, 0)
    B = gen.small_int_matrix(N, K, 33, 1)
    cfg = tg.make_config(mma=mma, schedule=2)
    ref, _ = oracle.gemm(A, B, M, N, K)
    for _ in range(2):
        got = run_gemm(A, B, M, N, K, K, K, N, False, cfg=cfg)
        assert np.array_equal(got, ref)


# Split tail: the units of a last wave that would keep at most half of the clusters busy
# are computed as two 256 x 128 half tiles each.  max_ctas shrinks the persistent grid so
# that small shapes have several waves: (1280, 512): 10 units on 4 clusters -> 2 split;
# (1300, 780): 24 units on 7 clusters -> 3 split, ragged edges; (512, 1024): 8 units, all
# split; (300, 520): 6 units, all split, one right half entirely past N.
SPLIT_CASES = [(1280, 512, 520, 8), (1300, 780, 136, 14), (512, 1024, 1000, 0), (300, 520, 200, 0)]


@pytest.mark.parametrize("M,N,K,max_ctas", SPLIT_CASES)
@pytest.mark.parametrize("out_bf16", [False, True])
def test_split_tail(M, N, K, max_ctas, out_bf16):
    # the CTA pair named explicitly: with these row strides (not 128-byte multiples) the
    # automatic choice would be the two-pair cluster, which has no split tail
    cfg = tg.make_config(tile_n=256, max_ctas=max_ctas, mma=2)
    layout = tg.TG_C_BF16 if out_bf16 else tg.TG_C_F32
    st, plan = tg.tg_gemm_plan_for(M, N, K, layout, cfg, 0)
    assert st == tg.TG_OK and plan.split_units > 0 and plan.sk_iters == 0
    full_check(M, N, K, out_bf16, seed=M + N + K, alpha=1.25, beta=0.5 if out_bf16 else 0.0,
               cfg=cfg)
    off = tg.make_config(tile_n=256, max_ctas=max_ctas, mma=2,
                         flags=tg.TG_GEMM_FLAG_NO_SPLIT_TAIL)
    st, plan = tg.tg_gemm_plan_for(M, N, K, layout, off, 0)
    assert st == tg.TG_OK and plan.split_units == 0
    full_check(M, N, K, out_bf16, seed=M + N + K, cfg=off)


def test_split_tail_exact_integers():
    # the half tiles' sums are exact (integers, K = 4096), so both schedules agree bit for bit
    M, N, K = 1280, 512, 4096
    A = gen.small_int_matrix(M, K, 37, 0)
    B = gen.small_int_matrix(N, K, 37, 1)
    ref, _ = oracle.gemm(A, B, M, N, K)
    for flags in (0, tg.TG_GEMM_FLAG_NO_SPLIT_TAIL):
        cfg = tg.make_config(tile_n=256, max_ctas=8, flags=flags)
        got = run_gemm(A, B, M, N, K, K, K, N, False, cfg=cfg)
        assert np.array_equal(got, ref)


def test_split_tail_other_operand_types():
    cfg = tg.make_config(tile_n=256, max_ctas=14, mma=2)
    mn_check(1300, 780, 136, True, False, True, cfg, seed=40, beta=0.5)   # A stored K x M
    f16_check(1300, 780, 136, "f16", False, False, cfg, seed=41, beta=0.5)
    f8_check(1300, 780, 256, "bf16", "e4m3", cfg, seed=42, beta=-1.0)
    tf32_check(1300, 780, 136, "bf16", cfg, seed=43)


# IEEE specials: a NaN in A poisons its row, an infinity in B gives +-inf down its column
# (the sign of the A entry it meets), exactly as the fp64 oracle computes; every other
# entry stays within the bound.  Through the default launch and both stream-K kernels.
@pytest.mark.parametrize("cfg", [None, {"schedule": 2, "mma": 2}, {"schedule": 2, "mma": 1}])
@pytest.mark.parametrize("out_bf16", [False, True])
def test_nan_and_inf_propagate(cfg, out_bf16):
    M, N, K = 300, 520, 200
    A = gen.bf16_matrix(M, K, 61, 0, "normal")
    B = gen.bf16_matrix(N, K, 61, 1, "normal")
    A[7, 13] = 0x7FC0                       # NaN
    A[:, 50] = np.where(A[:, 50] == 0, 0x3F80, A[:, 50])   # no zero meets the infinity
    A[:, 3] = np.where(A[:, 3] == 0, 0x3F80, A[:, 3])
    B[11, 50] = 0x7F80                      # +inf
    B[400, 3] = 0xFF80                      # -inf
    c = tg.make_config(**cfg) if cfg else None
    got = run_gemm(A, B, M, N, K, K, K, N, out_bf16, cfg=c)
    ref, mag = oracle.gemm(A, B, M, N, K)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.isnan(got[7]).all()
    inf = np.isinf(ref)
    assert inf[:, 11].sum() == M - 1 and inf[:, 400].sum() == M - 1
    assert np.array_equal(np.isinf(got), inf)
    assert np.array_equal(np.sign(got[inf]), np.sign(ref[inf]))
    fin = np.isfinite(ref)
    bound = gemm_bound(ref[fin], mag[fin], K, 1.0, 0.0, None, out_bf16)
    assert_within(got[fin], ref[fin], bound, "finite entries")


# Large extents: 2049 M tiles (1025 pair rows), or 1171 N tiles of 224, with a short K.
@pytest.mark.parametrize("M,N,K", [(262151, 24, 72), (24, 262151, 72)])
def test_large_extents(M, N, K):
    full_check(M, N, K, False, seed=M % 97 + N % 89)


# ------------------------------------------------------------------------------------
# MN-major operands (layout bit 0: A stored K x M, bit 1: B stored K x N)
# ------------------------------------------------------------------------------------
def mn_check(M, N, K, a_mn, b_mn, out_bf16, cfg, seed, alpha=1.0, beta=0.0):
    rup = lambda x, m: -(-x // m) * m
    lda = (rup(M, 8) if a_mn else rup(K, 8)) + 8
    ldb = (rup(N, 8) if b_mn else rup(K, 8)) + 16
    ldc = rup(N, 8)
    A = gen.bf16_matrix(K if a_mn else M, M if a_mn else K, seed, 0, "normal", ld=lda)
    B = gen.bf16_matrix(K if b_mn else N, N if b_mn else K, seed, 1, "normal", ld=ldb)
    C0 = None
    if beta != 0.0:
        C0 = (gen.bf16_matrix(M, N, seed, 2, "uniform", ld=ldc) if out_bf16 else
              np.pad(gen.uniform(seed, 2, M * N).astype(np.float32).reshape(M, N),
                     ((0, 0), (0, ldc - N))))
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    Cd = device_c(M, N, ldc, out_bf16, C0)
    layout = ((tg.TG_C_BF16 if out_bf16 else tg.TG_C_F32) | (tg.TG_LAYOUT_A_MN_MAJOR if a_mn else 0)
              | (tg.TG_LAYOUT_B_MN_MAJOR if b_mn else 0))
    st = tg.gemm_bf16_ex(M, N, K, Ad.data_ptr(), lda, Bd.data_ptr(), ldb, Cd.data_ptr(), ldc,
                         alpha, beta, layout, cfg, None)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    assert tg.tg_status_sync(None) == tg.TG_OK
    assert guard_rows_untouched(Cd)
    got = c_to_f64(Cd)[:, :N]
    ref, mag = oracle.gemm(A, B, M, N, K, lda=lda, ldb=ldb, C0=C0, ldc=ldc, alpha=alpha,
                           beta=beta, a_mn=a_mn, b_mn=b_mn)
    c0v = c0_values(C0)[:, :N] if C0 is not None else None
    assert_within(got, ref, gemm_bound(ref, mag, K, alpha, beta, c0v, out_bf16),
                  "mn M=%d N=%d K=%d a_mn=%s b_mn=%s" % (M, N, K, a_mn, b_mn))


MN_LAYOUTS = [(True, False), (False, True), (True, True)]


@pytest.mark.parametrize("a_mn,b_mn", MN_LAYOUTS)
@pytest.mark.parametrize("M,N,K", [(64, 64, 64), (300, 520, 200), (129, 257, 65), (1024, 768, 1000)])
@pytest.mark.parametrize("mma", [1, 2])
def test_mn_major(a_mn, b_mn, M, N, K, mma):
    mn_check(M, N, K, a_mn, b_mn, True, tg.make_config(mma=mma), seed=M + N + K)


@pytest.mark.parametrize("a_mn,b_mn", MN_LAYOUTS)
@pytest.mark.parametrize("cfg", [dict(mma=1, cluster=2), dict(mma=1, tile_n=128, stages=6),
                                 dict(mma=2, tile_n=128), dict(mma=2, schedule=2),
                                 dict(mma=1, schedule=2)])
def test_mn_major_configs(a_mn, b_mn, cfg):
    mn_check(1100, 1300, 2000, a_mn, b_mn, False, tg.make_config(**cfg), seed=5, alpha=0.5,
             beta=-0.25)
    mn_check(257, 520, 72, a_mn, b_mn, True, tg.make_config(**cfg), seed=6, beta=0.5)


@pytest.mark.parametrize("a_mn,b_mn", MN_LAYOUTS)
def test_mn_major_full_size_sampled(a_mn, b_mn):
    import torch
    M = N = K = 4096
    A = gen.bf16_matrix(K if a_mn else M, M if a_mn else K, 1, 0, "normal")
    B = gen.bf16_matrix(K if b_mn else N, N if b_mn else K, 1, 1, "normal")
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    Cd = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    layout = (tg.TG_C_BF16 | (tg.TG_LAYOUT_A_MN_MAJOR if a_mn else 0)
              | (tg.TG_LAYOUT_B_MN_MAJOR if b_mn else 0))
    assert tg.gemm_bf16(M, N, K, Ad.data_ptr(), A.shape[1], Bd.data_ptr(), B.shape[1],
                        Cd.data_ptr(), N, 1.0, 0.0, layout, None) == tg.TG_OK
    assert tg.tg_status_sync(None) == tg.TG_OK
    got = c_to_f64(Cd)
    ii, jj = sample_positions(M, N, seed=9)
    ref, mag = oracle.gemm_entries(A, B, K, ii, jj, lda=A.shape[1], ldb=B.shape[1], a_mn=a_mn,
                                   b_mn=b_mn)
    assert_within(got[ii, jj], ref, gemm_bound(ref, mag, K, 1.0, 0.0, None, True), "mn full")


def test_torch_views_select_the_storage():
    """tg.gemm takes transposed torch views (unit stride along M or N) as MN-major."""
    import torch
    M, N, K = 304, 264, 136   # M-major / N-major rows of 608 / 528 bytes: 16-byte multiples
    A = gen.bf16_matrix(M, K, 3, 0, "normal")
    B = gen.bf16_matrix(N, K, 3, 1, "normal")
    ref, mag = oracle.gemm(A, B, M, N, K)
    bound = gemm_bound(ref, mag, K, 1.0, 0.0, None, False)
    A_km, B_km = to_device_bf16(A), to_device_bf16(B)
    A_mn = A_km.t().contiguous().t()          # same values, M contiguous
    B_nm = B_km.t().contiguous().t()          # same values, N contiguous
    for Av, Bv in [(A_km, B_km), (A_mn, B_km), (A_km, B_nm), (A_mn, B_nm)]:
        C = torch.empty((M, N), dtype=torch.float32, device="cuda")
        tg.gemm(Av, Bv, C)
        assert tg.tg_status_sync(None) == tg.TG_OK
        assert_within(C.cpu().numpy().astype(np.float64), ref, bound, "views")


# ------------------------------------------------------------------------------------
# fp16 operands (layout bits 4-5) and fp16 C (layout bits 2-3 = 2)
# ------------------------------------------------------------------------------------
def f16_check(M, N, K, out, a_mn, b_mn, cfg, seed, alpha=1.0, beta=0.0):
    import torch
    from gpu_util import to_device_f16
    rup = lambda x, m: -(-x // m) * m
    lda = (rup(M, 8) if a_mn else rup(K, 8)) + 8
    ldb = (rup(N, 8) if b_mn else rup(K, 8)) + 8
    ldc = rup(N, 8)
    A = gen.f16_matrix(K if a_mn else M, M if a_mn else K, seed, 0, "normal", ld=lda)
    B = gen.f16_matrix(K if b_mn else N, N if b_mn else K, seed, 1, "normal", ld=ldb)
    C0 = None
    if out == "f32":
        C0 = np.pad(gen.uniform(seed, 2, M * N).astype(np.float32).reshape(M, N),
                    ((0, 0), (0, ldc - N)))
        Cd = to_device(C0)
    elif out == "bf16":
        C0 = gen.bf16_matrix(M, N, seed, 2, "uniform", ld=ldc)
        Cd = to_device_bf16(C0)
    else:
        C0 = gen.f16_matrix(M, N, seed, 2, "uniform", ld=ldc)
        Cd = to_device_f16(C0)
    Ad, Bd = to_device_f16(A), to_device_f16(B)
    layout = ({"f32": tg.TG_C_F32, "bf16": tg.TG_C_BF16, "f16": tg.TG_C_F16}[out] | tg.TG_IN_F16
              | (tg.TG_LAYOUT_A_MN_MAJOR if a_mn else 0) | (tg.TG_LAYOUT_B_MN_MAJOR if b_mn else 0))
    st = tg.gemm_bf16_ex(M, N, K, Ad.data_ptr(), lda, Bd.data_ptr(), ldb, Cd.data_ptr(), ldc,
                         alpha, beta, layout, cfg, None)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    assert tg.tg_status_sync(None) == tg.TG_OK
    got = c_to_f64(Cd)[:, :N]
    ref, mag = oracle.gemm(A, B, M, N, K, lda=lda, ldb=ldb, C0=C0, ldc=ldc, alpha=alpha,
                           beta=beta, a_mn=a_mn, b_mn=b_mn, in_f16=True, c_f16=(out == "f16"))
    c0v = c0_values(C0, f16=(out == "f16"))[:, :N]
    bound = gemm_bound(ref, mag, K, alpha, beta, c0v, out == "bf16", out == "f16")
    assert_within(got, ref, bound, "f16 in, %s out, M=%d N=%d K=%d" % (out, M, N, K))


@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (True, True), (True, False)])
@pytest.mark.parametrize("mma", [1, 2])
def test_f16_operands(out, a_mn, b_mn, mma):
    cfg = tg.make_config(mma=mma)
    f16_check(300, 520, 200, out, a_mn, b_mn, cfg, seed=3)
    f16_check(1100, 1304, 2000, out, a_mn, b_mn, cfg, seed=4, alpha=0.75, beta=0.5)


@pytest.mark.parametrize("out", ["bf16", "f16"])
def test_f16_stream_k_and_edges(out):
    f16_check(1100, 1300, 2000, out, False, False, tg.make_config(schedule=2), seed=8, beta=0.25)
    f16_check(129, 264, 65, out, False, True, tg.make_config(mma=2), seed=9, beta=-1.0)


def test_f16_full_size_sampled():
    import torch
    from gpu_util import to_device_f16
    M = N = K = 4096
    A = gen.f16_matrix(M, K, 1, 0, "normal")
    B = gen.f16_matrix(N, K, 1, 1, "normal")
    Ad, Bd = to_device_f16(A), to_device_f16(B)
    Cd = torch.empty((M, N), dtype=torch.float16, device="cuda")
    assert tg.gemm_bf16(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, Cd.data_ptr(), N, 1.0, 0.0,
                        tg.TG_IN_F16 | tg.TG_C_F16, None) == tg.TG_OK
    assert tg.tg_status_sync(None) == tg.TG_OK
    got = c_to_f64(Cd)
    ii, jj = sample_positions(M, N, seed=11)
    ref, mag = oracle.gemm_entries(A, B, K, ii, jj, in_f16=True)
    assert_within(got[ii, jj], ref, gemm_bound(ref, mag, K, 1.0, 0.0, None, False, True), "f16")


# ------------------------------------------------------------------------------------
# 8-bit operands (E4M3 / E5M2, layout bits 4-5 = 2 / 3): one byte per element, K-major
# ------------------------------------------------------------------------------------
F8_LAYOUT = {"e4m3": tg.TG_IN_E4M3, "e5m2": tg.TG_IN_E5M2}


def f8_check(M, N, K, out, kind, cfg, seed, alpha=1.0, beta=0.0, pad=16):
    import torch
    from gpu_util import to_device_f16
    rup = lambda x, m: -(-x // m) * m
    lda = rup(K, 16) + pad          # padding bytes hold a NaN pattern (0x7F)
    ldb = rup(K, 16) + pad
    ldc = rup(N, 8)
    e5m2 = kind == "e5m2"
    A = gen.f8_matrix(M, K, seed, 0, "normal", ld=lda, e5m2=e5m2)
    B = gen.f8_matrix(N, K, seed, 1, "normal", ld=ldb, e5m2=e5m2)
    if out == "f32":
        C0 = np.pad(gen.uniform(seed, 2, M * N).astype(np.float32).reshape(M, N),
                    ((0, 0), (0, ldc - N)))
        Cd = to_device(C0)
    elif out == "bf16":
        C0 = gen.bf16_matrix(M, N, seed, 2, "uniform", ld=ldc)
        Cd = to_device_bf16(C0)
    else:
        C0 = gen.f16_matrix(M, N, seed, 2, "uniform", ld=ldc)
        Cd = to_device_f16(C0)
    Ad, Bd = to_device(A), to_device(B)
    layout = {"f32": tg.TG_C_F32, "bf16": tg.TG_C_BF16, "f16": tg.TG_C_F16}[out] | F8_LAYOUT[kind]
    st = tg.gemm_bf16_ex(M, N, K, Ad.data_ptr(), lda, Bd.data_ptr(), ldb, Cd.data_ptr(), ldc,
                         alpha, beta, layout, cfg, None)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    assert tg.tg_status_sync(None) == tg.TG_OK
    got = c_to_f64(Cd)[:, :N]
    ref, mag = oracle.gemm(A, B, M, N, K, lda=lda, ldb=ldb, C0=C0, ldc=ldc, alpha=alpha,
                           beta=beta, in_kind=kind, c_f16=(out == "f16"))
    c0v = c0_values(C0, f16=(out == "f16"))[:, :N]
    bound = gemm_bound(ref, mag, K, alpha, beta, c0v, out == "bf16", out == "f16")
    assert_within(got, ref, bound, "%s in, %s out, M=%d N=%d K=%d" % (kind, out, M, N, K))


@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("kind", ["e4m3", "e5m2"])
@pytest.mark.parametrize("mma", [1, 2])
def test_f8_operands(out, kind, mma):
    cfg = tg.make_config(mma=mma)
    f8_check(300, 520, 200, out, kind, cfg, seed=13)
    f8_check(1100, 1304, 2000, out, kind, cfg, seed=14, alpha=0.75, beta=0.5)


@pytest.mark.parametrize("kind", ["e4m3", "e5m2"])
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (129, 257, 65), (257, 129, 16), (600, 40, 1000),
                                   (256, 256, 129)])
def test_f8_ragged(kind, M, N, K):
    f8_check(M, N, K, "bf16", kind, tg.make_config(mma=2), seed=M + N + K, beta=-1.0)
    f8_check(M, N, K, "f32", kind, tg.make_config(mma=1, cluster=1), seed=M + N + K)


@pytest.mark.parametrize("kind", ["e4m3", "e5m2"])
def test_f8_stream_k_and_configs(kind):
    f8_check(1100, 1300, 4000, "bf16", kind, tg.make_config(schedule=2), seed=15, beta=0.25)
    f8_check(1100, 1300, 4000, "f32", kind, tg.make_config(schedule=2, mma=1), seed=16)
    for cfg in [dict(mma=1, cluster=2), dict(mma=1, tile_n=128, stages=6), dict(mma=2, stages=4),
                dict(mma=2, tile_n=128)]:
        f8_check(700, 900, 777, "bf16", kind, tg.make_config(**cfg), seed=17)


def test_f8_exact_integers_bit_exact():
    # integers in [-2, 2] are exact in E4M3 and every partial sum (|.| <= 4 K) is exact in
    # fp32, so the result is exact whatever the summation order
    import torch
    M, N, K = 512, 640, 1000
    A = gen.f32_to_f8_bits(np.floor(gen.uniform(21, 0, M * K, -2.0, 3.0)).clip(-2, 2)).reshape(M, K)
    B = gen.f32_to_f8_bits(np.floor(gen.uniform(21, 1, N * K, -2.0, 3.0)).clip(-2, 2)).reshape(N, K)
    lda = ldb = 1008
    Ap = np.zeros((M, lda), np.uint8)
    Bp = np.zeros((N, ldb), np.uint8)
    Ap[:, :K], Bp[:, :K] = A, B
    Ad, Bd = to_device(Ap), to_device(Bp)
    for mma in (1, 2):
        Cd = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        st = tg.gemm_bf16_ex(M, N, K, Ad.data_ptr(), lda, Bd.data_ptr(), ldb,
                             Cd.data_ptr(), N, 1.0, 0.0, tg.TG_C_F32 | tg.TG_IN_E4M3,
                             tg.make_config(mma=mma), None)
        assert st == tg.TG_OK and tg.tg_status_sync(None) == tg.TG_OK
        ref, _ = oracle.gemm(Ap, Bp, M, N, K, lda=lda, ldb=ldb, in_kind="e4m3")
        assert np.array_equal(Cd.cpu().numpy().astype(np.float64), ref)


def test_f8_torch_tensors():
    import torch
    M, N, K = 264, 392, 320
    A = gen.f8_matrix(M, K, 18, 0, "normal")
    B = gen.f8_matrix(N, K, 18, 1, "normal", e5m2=False)
    At = to_device(A).view(torch.float8_e4m3fn)
    Bt = to_device(B).view(torch.float8_e4m3fn)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    tg.gemm(At, Bt, C)
    assert tg.tg_status_sync(None) == tg.TG_OK
    ref, mag = oracle.gemm(A, B, M, N, K, in_kind="e4m3")
    assert_within(c_to_f64(C), ref, gemm_bound(ref, mag, K, 1.0, 0.0, None, True), "torch f8")
    with pytest.raises(tg.TgError):
        # the same A stored M-major (unit stride along M): unsupported for 8-bit types
        tg.gemm(to_device(np.ascontiguousarray(A.T)).view(torch.float8_e4m3fn).t(), Bt, C)


@pytest.mark.parametrize("kind", ["e4m3", "e5m2"])
def test_f8_full_size_sampled(kind):
    import torch
    M = N = K = 8192
    if kind == "e4m3":     # the benchmark's E4M3 workload, in its launch configuration
        A, B, _ = gen.gemm_inputs("gemm_8192_e4m3")
    else:
        A = gen.f8_matrix(M, K, 3, 0, "uniform", e5m2=True)
        B = gen.f8_matrix(N, K, 3, 1, "uniform", e5m2=True)
    Ad, Bd = to_device(A), to_device(B)
    Cd = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert tg.gemm_bf16(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, Cd.data_ptr(), N, 1.0, 0.0,
                        F8_LAYOUT[kind] | tg.TG_C_BF16, None) == tg.TG_OK
    assert tg.tg_status_sync(None) == tg.TG_OK
    got = c_to_f64(Cd)
    ii, jj = sample_positions(M, N, seed=19)
    ref, mag = oracle.gemm_entries(A, B, K, ii, jj, in_kind=kind)
    assert_within(got[ii, jj], ref, gemm_bound(ref, mag, K, 1.0, 0.0, None, True), kind)


# ------------------------------------------------------------------------------------
# tf32 operands (layout bits 4-6 = 4): binary32 arrays, truncated to 10 mantissa bits
# ------------------------------------------------------------------------------------
def tf32_check(M, N, K, out, cfg, seed, alpha=1.0, beta=0.0, pad=4, dist="normal"):
    import torch
    from gpu_util import to_device_f16
    rup = lambda x, m: -(-x // m) * m
    lda = rup(K, 4) + pad           # padding holds NaN
    ldb = rup(K, 4) + pad
    ldc = rup(N, 8)
    draw = gen.normal if dist == "normal" else gen.uniform
    A = np.full((M, lda), np.nan, dtype=np.float32)
    B = np.full((N, ldb), np.nan, dtype=np.float32)
    A[:, :K] = draw(seed, 0, M * K).astype(np.float32).reshape(M, K)
    B[:, :K] = draw(seed, 1, N * K).astype(np.float32).reshape(N, K)
    if out == "f32":
        C0 = np.pad(gen.uniform(seed, 2, M * N).astype(np.float32).reshape(M, N),
                    ((0, 0), (0, ldc - N)))
        Cd = to_device(C0)
    elif out == "bf16":
        C0 = gen.bf16_matrix(M, N, seed, 2, "uniform", ld=ldc)
        Cd = to_device_bf16(C0)
    else:
        C0 = gen.f16_matrix(M, N, seed, 2, "uniform", ld=ldc)
        Cd = to_device_f16(C0)
    Ad, Bd = to_device(A), to_device(B)
    layout = {"f32": tg.TG_C_F32, "bf16": tg.TG_C_BF16, "f16": tg.TG_C_F16}[out] | tg.TG_IN_TF32
    st = tg.gemm_bf16_ex(M, N, K, Ad.data_ptr(), lda, Bd.data_ptr(), ldb, Cd.data_ptr(), ldc,
                         alpha, beta, layout, cfg, None)
    assert st == tg.TG_OK, tg.tg_status_string(st)
    assert tg.tg_status_sync(None) == tg.TG_OK
    got = c_to_f64(Cd)[:, :N]
    ref, mag = oracle.gemm(A, B, M, N, K, lda=lda, ldb=ldb, C0=C0, ldc=ldc, alpha=alpha,
                           beta=beta, in_kind="tf32", c_f16=(out == "f16"))
    c0v = c0_values(C0, f16=(out == "f16"))[:, :N]
    bound = gemm_bound(ref, mag, K, alpha, beta, c0v, out == "bf16", out == "f16")
    assert_within(got, ref, bound, "tf32 in, %s out, M=%d N=%d K=%d" % (out, M, N, K))


def test_tf32_inputs_are_truncated_not_rounded():
    # B = identity: C is A as the tensor core reads it.  Values in [1, 2) with random low
    # mantissa bits: the page's tf32 keeps 10 bits by truncation, so C must equal A with
    # its 13 low mantissa bits cleared, bit for bit (rounding would differ in about half).
    import torch
    M, K = 256, 64
    A = (1.0 + gen.uniform(31, 0, M * K, 0.0, 1.0)).astype(np.float32).reshape(M, K)
    A[:, 1::2] *= -1.0
    B = np.eye(K, dtype=np.float32)
    for mma in (1, 2):
        Cd = torch.full((M, K), float("nan"), dtype=torch.float32, device="cuda")
        Ad, Bd = to_device(A), to_device(B)
        st = tg.gemm_bf16_ex(M, K, K, Ad.data_ptr(), K, Bd.data_ptr(), K, Cd.data_ptr(), K, 1.0,
                             0.0, tg.TG_C_F32 | tg.TG_IN_TF32, tg.make_config(mma=mma), None)
        assert st == tg.TG_OK and tg.tg_status_sync(None) == tg.TG_OK
        got = Cd.cpu().numpy()
        ref, _ = oracle.gemm(A, B, M, K, K, in_kind="tf32")
        assert np.array_equal(got.astype(np.float64), ref)
        assert not np.array_equal(got, A)          # the low bits really were dropped


@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("mma", [1, 2])
def test_tf32_operands(out, mma):
    cfg = tg.make_config(mma=mma)
    tf32_check(300, 520, 200, out, cfg, seed=23)
    tf32_check(1100, 1304, 2000, out, cfg, seed=24, alpha=0.75, beta=0.5)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (129, 257, 33), (257, 129, 8), (600, 40, 1000),
                                   (256, 256, 129)])
def test_tf32_ragged(M, N, K):
    tf32_check(M, N, K, "bf16", tg.make_config(mma=2), seed=M + N + K, beta=-1.0)
    tf32_check(M, N, K, "f32", tg.make_config(mma=1, cluster=1), seed=M + N + K)


def test_tf32_stream_k_and_configs():
    tf32_check(1100, 1300, 4000, "bf16", tg.make_config(schedule=2), seed=25, beta=0.25)
    tf32_check(1100, 1300, 4000, "f32", tg.make_config(schedule=2, mma=1), seed=26)
    for cfg in [dict(mma=1, cluster=2), dict(mma=1, tile_n=128, stages=6), dict(mma=2, stages=4),
                dict(mma=2, tile_n=128)]:
        tf32_check(700, 900, 777, "bf16", tg.make_config(**cfg), seed=27)


def test_tf32_torch_tensors():
    import torch
    M, N, K = 264, 392, 320
    A = gen.normal(28, 0, M * K).astype(np.float32).reshape(M, K)
    B = gen.normal(28, 1, N * K).astype(np.float32).reshape(N, K)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    tg.gemm(to_device(A), to_device(B), C)
    assert tg.tg_status_sync(None) == tg.TG_OK
    ref, mag = oracle.gemm(A, B, M, N, K, in_kind="tf32")
    assert_within(c_to_f64(C), ref, gemm_bound(ref, mag, K, 1.0, 0.0, None, False), "torch tf32")


def test_tf32_full_size_sampled():
    import torch
    M = N = K = 8192
    A, B, _ = gen.gemm_inputs("gemm_8192_tf32")
    Ad, Bd = to_device(A), to_device(B)
    Cd = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert tg.gemm_bf16(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, Cd.data_ptr(), N, 1.0, 0.0,
                        tg.TG_IN_TF32 | tg.TG_C_BF16, None) == tg.TG_OK
    assert tg.tg_status_sync(None) == tg.TG_OK
    got = c_to_f64(Cd)
    ii, jj = sample_positions(M, N, seed=29)
    ref, mag = oracle.gemm_entries(A, B, K, ii, jj, in_kind="tf32")
    assert_within(got[ii, jj], ref, gemm_bound(ref, mag, K, 1.0, 0.0, None, True), "tf32")


# ------------------------------------------------------------------------------------
# Dynamic schedule (schedule = 3): one cluster per unit, cluster launch control
# ------------------------------------------------------------------------------------
DYN = [dict(schedule=3, mma=2), dict(schedule=3, mma=1, cluster=1),
       dict(schedule=3, mma=1, cluster=2), dict(schedule=3, mma=2, tile_n=128)]


@pytest.mark.parametrize("cfg", DYN)
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (300, 520, 200), (1100, 1304, 2000),
                                   (2048, 2048, 256)])
def test_dynamic_schedule(cfg, M, N, K):
    full_check(M, N, K, True, beta=0.5, seed=M + K, cfg=tg.make_config(**cfg))


@pytest.mark.parametrize("cfg", DYN[:2])
def test_dynamic_schedule_other_types(cfg):
    f8_check(1100, 1304, 2000, "bf16", "e4m3", tg.make_config(**cfg), seed=33)
    tf32_check(700, 900, 777, "f32", tg.make_config(**cfg), seed=34, beta=0.5)
    f16_check(300, 520, 200, "f16", False, False, tg.make_config(**cfg), seed=35)


def test_dynamic_schedule_full_size_sampled():
    import torch
    M, N, K, _, _, _, _, seed, out, alpha, beta = gen.GEMM_WORKLOADS["gemm_8192"]
    A, B, _ = gen.gemm_inputs("gemm_8192")
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    Cd = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    for _ in range(2):   # the second launch reuses the ring of barriers from a clean start
        st = tg.gemm_bf16_ex(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, Cd.data_ptr(), N, alpha,
                             beta, tg.TG_C_BF16, tg.make_config(schedule=3), None)
        assert st == tg.TG_OK and tg.tg_status_sync(None) == tg.TG_OK
    got = c_to_f64(Cd)
    ii, jj = sample_positions(M, N, seed=37)
    ref, mag = oracle.gemm_entries(A, B, K, ii, jj)
    assert_within(got[ii, jj], ref, gemm_bound(ref, mag, K, alpha, beta, None, True), "dynamic")


def test_dynamic_schedule_on_two_streams_at_once():
    # two launches share the GPU: each grid's clusters take over the units of their own
    # grid's pending clusters only
    import torch
    M, N, K = 2048, 3072, 1024
    A = gen.bf16_matrix(M, K, 38, 0, "normal")
    B = gen.bf16_matrix(N, K, 38, 1, "normal")
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    ref, mag = oracle.gemm(A, B, M, N, K)
    bound = gemm_bound(ref, mag, K, 1.0, 0.0, None, True)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    for rep in range(3):
        for s, C in zip(streams, outs):
            st = tg.gemm_bf16_ex(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, C.data_ptr(), N, 1.0,
                                 0.0, tg.TG_C_BF16, tg.make_config(schedule=3),
                                 ctypes_stream(s))
            assert st == tg.TG_OK
    torch.cuda.synchronize()
    assert tg.tg_status_sync(None) == tg.TG_OK
    for C in outs:
        assert_within(c_to_f64(C), ref, bound, "dynamic, two streams")


# ------------------------------------------------------------------------------------
# 256 x 224 pair tiles (tile_n = 224): a last 32-column chunk per tile for 16-bit C
# ------------------------------------------------------------------------------------
@pytest.mark.parametrize("M,N,K,out_bf16,beta", [(300, 520, 200, True, 0.5), (1100, 1304, 2000, True, 0.0),
                                                 (257, 224, 65, False, -1.0), (512, 4096, 1024, True, 0.0),
                                                 (600, 900, 777, False, 0.5)])
@pytest.mark.parametrize("schedule", [0, 2, 3])
def test_tile_224(M, N, K, out_bf16, beta, schedule):
    full_check(M, N, K, out_bf16, beta=beta, seed=M + N + schedule,
               cfg=tg.make_config(tile_n=224, schedule=schedule))


def test_tile_224_other_types_and_storage():
    cfg = tg.make_config(tile_n=224)
    for out in ("f16", "bf16", "f32"):
        f16_check(300, 520, 200, out, True, False, cfg, seed=71, beta=0.5)   # M-major A
    f8_check(1100, 1304, 2000, "bf16", "e4m3", cfg, seed=72, beta=0.5)
    tf32_check(700, 900, 777, "f16", cfg, seed=73)
    # an N-major B tile cannot be split into 64-element boxes per CTA at this width
    import torch
    A = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((256, 256), dtype=torch.bfloat16, device="cuda").t()
    C = torch.zeros((256, 256), dtype=torch.float32, device="cuda")
    assert tg.gemm(A, B, C, config=cfg, check=False) == tg.TG_ERR_UNSUPPORTED


def test_tile_224_dw_sampled():
    import torch
    M, N, K, _, _, _, _, seed, out, alpha, beta = gen.GEMM_WORKLOADS["dw"]
    A, B, C0 = gen.gemm_inputs("dw")
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    Cd = device_c(M, N, N, True, C0)
    st = tg.gemm_bf16_ex(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, Cd.data_ptr(), N, alpha, beta,
                         tg.TG_C_BF16, tg.make_config(tile_n=224), None)
    assert st == tg.TG_OK and tg.tg_status_sync(None) == tg.TG_OK
    got = c_to_f64(Cd)
    ii, jj = sample_positions(M, N, seed=74)
    ref, mag = oracle.gemm_entries(A, B, K, ii, jj)
    assert_within(got[ii, jj], ref, gemm_bound(ref, mag, K, alpha, beta, None, True), "224 dW")


def test_tensor_rate_probe_kinds_keep_their_ratios():
    # the same bytes of K per MMA: E4M3 does twice and tf32 half the bf16 FLOPs per cycle
    import torch
    rates = {}
    for name, layout in [("bf16", tg.TG_IN_BF16), ("e4m3", tg.TG_IN_E4M3), ("tf32", tg.TG_IN_TF32)]:
        tg.tensor_rate_probe(layout, 256)                      # warm-up
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        st, pairs, flops = tg.tensor_rate_probe(layout, 1 << 13)
        e1.record()
        torch.cuda.synchronize()
        assert st == tg.TG_OK and pairs > 0
        assert tg.tg_status_sync(None) == tg.TG_OK
        rates[name] = flops / (e0.elapsed_time(e1) * 1e-3)
    assert 1.6 < rates["e4m3"] / rates["bf16"] < 2.4
    assert 0.35 < rates["tf32"] / rates["bf16"] < 0.65


def test_tensor_rate_probe_timed_by_the_gpu():
    # the GPU's own count: cycles / ns is a plausible SM clock, and the per-SM FLOP per
    # cycle is at most the tensor cores' 8192 (bf16), twice that for E4M3, half for tf32
    import torch
    timing = torch.zeros(2, dtype=torch.int64, device="cuda")
    for layout, top in [(tg.TG_IN_BF16, 8192), (tg.TG_IN_E4M3, 16384), (tg.TG_IN_TF32, 4096)]:
        tg.tensor_rate_probe(layout, 256)                      # warm-up
        st, pairs, flops = tg.tensor_rate_probe_timed(timing.data_ptr(), layout, 1 << 12)
        torch.cuda.synchronize()
        assert st == tg.TG_OK and pairs > 0
        assert tg.tg_status_sync(None) == tg.TG_OK
        cycles, ns = timing.cpu().tolist()
        assert cycles > 0 and ns > 0
        assert 0.5 < cycles / ns < 2.5                         # GHz
        per_sm_clk = flops / pairs / 2 / cycles
        assert 0.7 * top < per_sm_clk <= 1.02 * top


@pytest.mark.parametrize("kernel", [
    {"mma": 1},                      # per CTA, cluster of one
    {"mma": 1, "cluster": 2},        # per CTA, B multicast across a cluster of two
    {"mma": 2},                      # CTA pair (the default kernel)
    {"mma": 3},                      # two CTA pairs sharing B by multicast (cluster of four)
])
def test_device_timeout_is_reported_and_context_survives(kernel):
    # The hook makes the first cluster's producers issue nothing, so the MMA issuer's first
    # wait runs out while no copy is in flight; max_ctas keeps the launch to that one
    # cluster.  Every wait is bounded (50 ms here), the error is latched with the role that
    # gave up, and a correct GEMM follows on the same context.
    import torch
    cluster = kernel.get("cluster", {1: 1, 2: 2, 3: 4}[kernel["mma"]])
    cfg = tg.make_config(flags=tg.TG_GEMM_FLAG_TEST_SKIP_FIRST_LOAD, timeout_ns=50_000_000,
                         max_ctas=cluster, **kernel)
    M = N = K = 256
    A = gen.bf16_matrix(M, K, 1, 0, "normal")
    B = gen.bf16_matrix(N, K, 1, 1, "normal")
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    Cd = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    st, plan = tg.tg_gemm_plan_for(M, N, K, tg.TG_C_F32, cfg, 0)
    assert st == tg.TG_OK and plan.grid == cluster
    st = tg.gemm_bf16_ex(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, Cd.data_ptr(), N, 1.0, 0.0,
                         tg.TG_C_F32, cfg, None)
    assert st == tg.TG_OK
    assert tg.tg_status_sync(None) == tg.TG_ERR_DEVICE_TIMEOUT
    detail = tg.tg_status_detail()
    assert (detail & 0xFF) == tg.TG_ERR_DEVICE_TIMEOUT
    # the MMA issuer's wait for the first stage, or the epilogue's for the accumulator,
    # ran out first (they start together)
    assert (detail >> 8) & 0xF in (2, 3)
    assert tg.tg_status_sync(None) == tg.TG_OK       # cleared once read
    # the same kernel, without the hook, on the same context
    ok_cfg = tg.make_config(**kernel)
    full_check(256, 256, 256, False, seed=0, dist="uniform", cfg=ok_cfg)
    full_check(300, 520, 200, True, beta=0.5, seed=4, cfg=ok_cfg)


# ------------------------------------------------------------------------------------
# Full-size workloads, in the launch configuration the benchmark times: sampled outputs
# checked one by one against the oracle, plus whole rows at tile edges.
# ------------------------------------------------------------------------------------
FULL = ["gemm_4096", "ffn_up", "ffn_down", "dw", "ragged", "gemm_8192"]


def sample_positions(M, N, n=3000, seed=0):
    rng = np.random.default_rng(seed)
    ii = list(rng.integers(0, M, n))
    jj = list(rng.integers(0, N, n))
    edges_m = sorted({0, 1, 127, 128, 255, 256, M // 2, M - 129, M - 128, M - 2, M - 1} & set(range(M)))
    edges_n = sorted({0, 1, 127, 128, 255, 256, N // 2, N - 257, N - 256, N - 2, N - 1} & set(range(N)))
    for i in edges_m:
        for j in edges_n:
            ii.append(i)
            jj.append(j)
    return np.array(ii, dtype=np.int64), np.array(jj, dtype=np.int64)


@pytest.mark.parametrize("name,schedule,expect", [
    ("gemm_8192", 0, "split"),      # 1024 pair tiles on 76 pairs: the last 36 as 72 half tiles
    ("ffn_down", 0, "split"),       # three waves, then 28 tiles as 56 half tiles
    ("ffn_down", 2, "stream_k"),    # the last waves' tiles finished from other clusters' partials
    ("dw", 0, "w224"),              # 76 pair tiles 256 x 224
])
def test_full_size_stratified(name, schedule, expect):
    """The default launch (the one the benchmark times; for FFN down also its stream-K
    schedule) checked in every cell of its tiling: two outputs per (tile, epilogue quarter,
    64-column chunk), including every split-tail half tile and every stream-K owner tile,
    against the oracle's entries."""
    import torch
    M, N, K, _, _, _, _, seed, out, alpha, beta = gen.GEMM_WORKLOADS[name]
    out_bf16 = out == "bf16"
    layout = tg.TG_C_BF16 if out_bf16 else tg.TG_C_F32
    cfg = tg.make_config(schedule=schedule) if schedule else None
    st, plan = tg.tg_gemm_plan_for(M, N, K, layout, cfg, 0)
    assert st == tg.TG_OK
    if expect == "split":
        assert plan.split_units > 0 and plan.tile_n == 256
    elif expect == "stream_k":
        assert plan.sk_iters > 0
    else:
        assert plan.tile_n == 224
    A, B, C0 = gen.gemm_inputs(name)
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    Cd = device_c(M, N, N, out_bf16, C0)
    st = tg.gemm_bf16_ex(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, Cd.data_ptr(), N, alpha,
                         beta, layout, cfg, None)
    assert st == tg.TG_OK
    assert tg.tg_status_sync(None) == tg.TG_OK
    st, last = tg.tg_gemm_last_plan()
    assert st == tg.TG_OK and last.sk_iters == plan.sk_iters and last.split_units == plan.split_units
    assert guard_rows_untouched(Cd)
    got = c_to_f64(Cd)
    del Ad, Bd, Cd
    torch.cuda.empty_cache()
    ii, jj = stratified_positions(M, N, plan.tile_n, seed=seed)
    cells = (-(-M // 32)) * sum(-(-min(plan.tile_n, N - t) // 64) for t in range(0, N, plan.tile_n))
    assert len(ii) == 2 * cells
    ref, mag = oracle.gemm_entries(A, B, K, ii, jj, C0=C0, ldc=N, alpha=alpha, beta=beta)
    c0v = c0_values(C0)[ii, jj] if C0 is not None else None
    assert_within(got[ii, jj], ref, gemm_bound(ref, mag, K, alpha, beta, c0v, out_bf16),
                  "%s stratified" % name)


@pytest.mark.parametrize("name", FULL)
@pytest.mark.parametrize("mma", [0, 1, 2])
def test_full_size_workload_sampled(name, mma):
    """mma 0 = the library default (the launch the benchmark times); 1 and 2 = each kind."""
    import torch
    M, N, K, _, _, _, _, seed, out, alpha, beta = gen.GEMM_WORKLOADS[name]
    out_bf16 = out == "bf16"
    A, B, C0 = gen.gemm_inputs(name)
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    Cd = device_c(M, N, N, out_bf16, C0)
    layout = tg.TG_C_BF16 if out_bf16 else tg.TG_C_F32
    if mma == 0:
        st = tg.gemm_bf16(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, Cd.data_ptr(), N, alpha,
                          beta, layout, None)
    else:
        st = tg.gemm_bf16_ex(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, Cd.data_ptr(), N, alpha,
                             beta, layout, tg.make_config(mma=mma), None)
    assert st == tg.TG_OK
    assert tg.tg_status_sync(None) == tg.TG_OK
    got = c_to_f64(Cd)
    del Ad, Bd, Cd
    torch.cuda.empty_cache()
    assert np.isfinite(got).all()
    ii, jj = sample_positions(M, N, seed=seed)
    ref, mag = oracle.gemm_entries(A, B, K, ii, jj, C0=C0, ldc=N, alpha=alpha, beta=beta)
    c0v = c0_values(C0)[ii, jj] if C0 is not None else None
    bound = gemm_bound(ref, mag, K, alpha, beta, c0v, out_bf16)
    assert_within(got[ii, jj], ref, bound, name)
    # two whole rows (first and last) across every column tile
    for r in (0, M - 1):
        ref_r, mag_r = oracle.gemm(A, B, M, N, K, C0=C0, ldc=N, alpha=alpha, beta=beta, rows=(r, r + 1))
        c0r = c0_values(C0)[r:r + 1] if C0 is not None else None
        assert_within(got[r:r + 1], ref_r, gemm_bound(ref_r, mag_r, K, alpha, beta, c0r, out_bf16),
                      "%s row %d" % (name, r))
