"""GPU parity of the two-pair cluster (tg_gemm_config.mma = 3, a cluster of four CTAs):
two CTA pairs stacked along M compute 512 x BN units; each CTA loads a quarter of the
shared B tile and multicasts it to the CTA of the same parity in the other pair ("2 . Le
Tensor Memory Accelerator" 2.5: a tile several blocks of a cluster need is read once and
delivered to all of them), so each SM requests 23 % fewer operand rows per k-block than
with one pair.  Results are checked against the fp64 oracle at the bound
|C - C_ref| <= 2*K*2^-24*|alpha|*(|A||B|) + 2^-8*|C_ref| (bf16 C) + 2^-23*|beta*C0|, and
bit-exactly in the exact-integer regime."""
import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_gb300 import inputs as gen
from tma_pipelined_tensor_gb300 import tg

from gpu_util import assert_within, c0_values, c_to_f64, gemm_bound, to_device_bf16
from test_gemm_gpu import full_check, run_gemm

pytestmark = pytest.mark.gpu


def quad(**kw):
    return tg.make_config(mma=3, **kw)


@pytest.mark.parametrize("tile_n", [128, 224, 256])
@pytest.mark.parametrize("M,N,K", [(520, 1000, 300), (1, 1, 1), (129, 257, 65), (1100, 700, 1030),
                                   (2100, 300, 64)])
def test_quad_ragged(tile_n, M, N, K):
    st, plan = tg.tg_gemm_plan_for(M, N, K, tg.TG_C_BF16, quad(tile_n=tile_n), 0)
    assert st == tg.TG_OK and plan.mma == 3 and plan.cluster == 4 and plan.grid % 4 == 0
    full_check(M, N, K, True, seed=M + N + K + tile_n, beta=0.5, alpha=1.25,
               cfg=quad(tile_n=tile_n))


@pytest.mark.parametrize("stages", [2, 3, 4, 5, 6])
def test_quad_stages(stages):
    full_check(1030, 900, 520, False, seed=stages, cfg=quad(stages=stages))


@pytest.mark.parametrize("pad", [(8, 8, 0), (8, 24, 8), (0, 40, 16)])
def test_quad_misaligned_rows(pad):
    # row strides that are 16-byte but not 128-byte multiples (the case the two-pair
    # cluster is for): every 128-byte TMA row straddles two L2 lines
    full_check(1300, 1100, 1032, True, seed=sum(pad), beta=0.5, pad=pad, cfg=quad())


def test_quad_exact_integers_bit_exact():
    M, N, K = 1024, 896, 2048
    A = gen.small_int_matrix(M, K, 81, 0)
    B = gen.small_int_matrix(N, K, 81, 1)
    ref, _ = oracle.gemm(A, B, M, N, K)
    got = run_gemm(A, B, M, N, K, K, K, N, False, cfg=quad())
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("out", ["f32", "f16"])
def test_quad_other_outputs_and_m_major_a(out):
    import torch
    M, N, K = 704, 640, 384          # M-major A: rows of M elements, a 16-byte multiple
    A = gen.bf16_matrix(M, K, 5, 0, "normal")
    B = gen.bf16_matrix(N, K, 5, 1, "normal")
    # A stored M-major (K rows of M elements): the same values, transposed storage
    At = np.ascontiguousarray(A.reshape(M, K).T)
    Ad, Bd = to_device_bf16(At), to_device_bf16(B)
    dt = torch.float32 if out == "f32" else torch.float16
    Cd = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
    layout = tg.TG_LAYOUT_A_MN_MAJOR | (tg.TG_C_F32 if out == "f32" else tg.TG_C_F16)
    st = tg.gemm_bf16_ex(M, N, K, Ad.data_ptr(), M, Bd.data_ptr(), K, Cd.data_ptr(), N, 1.0, 0.0,
                         layout, quad(), None)
    assert st == tg.TG_OK and tg.tg_status_sync(None) == tg.TG_OK
    got = Cd.float().cpu().numpy().astype(np.float64)
    ref, mag = oracle.gemm(A, B, M, N, K)
    bound = gemm_bound(ref, mag, K, 1.0, 0.0, None, False, out_f16=(out == "f16"))
    assert_within(got, ref, bound, "quad %s M-major A" % out)


def test_quad_stream_k():
    cfg = quad(schedule=2)
    st, plan = tg.tg_gemm_plan_for(1100, 1300, 2000, tg.TG_C_BF16, cfg, 0)
    assert st == tg.TG_OK and plan.sk_iters > 0
    full_check(1100, 1300, 2000, True, seed=91, beta=0.5, cfg=cfg)


def test_quad_refusals():
    import torch
    A = torch.ones((256, 256), dtype=torch.uint8, device="cuda")
    C = torch.zeros((256, 256), dtype=torch.float32, device="cuda")
    # 8-bit operands and an N-major B are not provided by the two-pair cluster
    st = tg.gemm_bf16_ex(256, 256, 256, A.data_ptr(), 256, A.data_ptr(), 256, C.data_ptr(), 256,
                         1.0, 0.0, tg.TG_C_F32 | tg.TG_IN_E4M3, quad(), None)
    assert st == tg.TG_ERR_UNSUPPORTED
    Ab = torch.ones((256, 256), dtype=torch.bfloat16, device="cuda")
    st = tg.gemm_bf16_ex(256, 256, 256, Ab.data_ptr(), 256, Ab.data_ptr(), 256, C.data_ptr(), 256,
                         1.0, 0.0, tg.TG_C_F32 | tg.TG_LAYOUT_B_MN_MAJOR, quad(), None)
    assert st == tg.TG_ERR_UNSUPPORTED


def test_quad_full_size_ragged_sampled():
    """The 3000 x 5000 x 2056 workload (beta = 0.5, bf16 C, its own row strides) on the
    two-pair cluster: every (512-row unit quarter, 64-column chunk) cell sampled."""
    import torch
    from gpu_util import stratified_positions
    M, N, K, _, _, _, _, seed, out, alpha, beta = gen.GEMM_WORKLOADS["ragged"]
    A, B, C0 = gen.gemm_inputs("ragged")
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    Cd = to_device_bf16(C0)
    cfg = quad()
    st = tg.gemm_bf16_ex(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, Cd.data_ptr(), N, alpha, beta,
                         tg.TG_C_BF16, cfg, None)
    assert st == tg.TG_OK and tg.tg_status_sync(None) == tg.TG_OK
    _, last = tg.tg_gemm_last_plan()
    got = c_to_f64(Cd)
    ii, jj = stratified_positions(M, N, last.tile_n, seed=seed)
    ref, mag = oracle.gemm_entries(A, B, K, ii, jj, C0=C0, ldc=N, alpha=alpha, beta=beta)
    bound = gemm_bound(ref, mag, K, alpha, beta, c0_values(C0)[ii, jj], True)
    assert_within(got[ii, jj], ref, bound, "quad ragged")


@pytest.mark.parametrize("lda_pad,expect_quad", [(0, False), (8, True)])
def test_automatic_choice_follows_the_row_strides(lda_pad, expect_quad):
    """The default launch takes the two-pair cluster exactly when A's or B's rows are not
    128-byte multiples (K = 1024: 2048-byte rows; padded by 8 elements: 2064 bytes)."""
    M, N, K = 1024, 768, 1024
    full_check(M, N, K, True, seed=3 + lda_pad, pad=(lda_pad, 0, 0))
    st, last = tg.tg_gemm_last_plan()
    assert st == tg.TG_OK
    assert (last.mma == 3) == expect_quad and (last.cluster == 4) == expect_quad
