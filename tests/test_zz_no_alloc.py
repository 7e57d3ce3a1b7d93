"""gemm_bf16_noalloc: the GEMM entry point for callers that cannot allocate device memory.

Who needs it: code that runs while a CUDA stream is being captured (cudaMalloc is not
permitted there), code whose device memory belongs entirely to another allocator or to
a fixed budget, and code that must not make the implicitly synchronising allocation
calls.  gemm_bf16 allocates its status word on first use of a device; this variant keeps
its status words in a small array inside the library's device image instead.

This file is collected last on purpose, so that a run which stops at its first failure
has already run every other test; it passes alone in a fresh process and after them.
"""
import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_gb300 import build as tgbuild
from tma_pipelined_tensor_gb300 import inputs as gen
from tma_pipelined_tensor_gb300 import tg

FAKE = 0x10000


@pytest.fixture(scope="module", autouse=True)
def _built():
    tgbuild.build()


def test_noalloc_is_exported_and_checks_arguments_on_the_host():
    assert "gemm_bf16_noalloc" in tg.declared_functions()
    assert hasattr(tg.lib(), "gemm_bf16_noalloc")
    call = lambda **kw: tg.gemm_bf16_noalloc(
        kw.get("M", 256), kw.get("N", 256), kw.get("K", 256), kw.get("A", FAKE), kw.get("lda", 256),
        FAKE, 256, kw.get("C", FAKE), kw.get("ldc", 256), 1.0, 0.0, kw.get("layout", tg.TG_C_F32))
    assert call(M=-1) == tg.TG_ERR_INVALID_VALUE
    assert call(layout=1 << 7) == tg.TG_ERR_INVALID_VALUE
    assert call(A=FAKE + 2) == tg.TG_ERR_MISALIGNED
    assert call(lda=100) == tg.TG_ERR_INVALID_VALUE
    assert call(ldc=258) == tg.TG_ERR_MISALIGNED
    assert call(M=0, A=0, C=0) == tg.TG_OK


def _problem(M, N, K, seed, beta):
    A = gen.bf16_matrix(M, K, seed, gen.STREAM_A, "normal")
    B = gen.bf16_matrix(N, K, seed, gen.STREAM_B, "normal")
    C0 = gen.bf16_matrix(M, N, seed, gen.STREAM_C, "uniform") if beta != 0.0 else None
    return A, B, C0


@pytest.mark.gpu
def test_noalloc_matches_gemm_bf16_on_two_calls_in_a_row():
    import torch

    from gpu_util import c_to_f64, gemm_bound, to_device_bf16

    status = torch.full((2,), 0x7777, dtype=torch.int32, device="cuda")
    cases = [(300, 520, 200, 41, 0.5), (1024, 768, 1000, 42, 0.0)]
    for call, (M, N, K, seed, beta) in enumerate(cases):
        A, B, C0 = _problem(M, N, K, seed, beta)
        Ad, Bd = to_device_bf16(A), to_device_bf16(B)
        init = C0 if C0 is not None else np.full((M, N), 0x7FC0, dtype=np.uint16)
        C_ref_dev = to_device_bf16(init)
        C_dp_dev = to_device_bf16(init)
        C_new_dev = to_device_bf16(init)
        st = tg.gemm_bf16(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, C_ref_dev.data_ptr(), N,
                          1.0, beta, tg.TG_C_BF16, None)
        assert st == tg.TG_OK and tg.tg_status_sync(None) == tg.TG_OK
        # the same kernel (the CTA pair) with whole tiles only, which is how this entry
        # point launches; gemm_bf16's own choice may differ with these row strides
        st = tg.gemm_bf16_ex(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, C_dp_dev.data_ptr(), N,
                             1.0, beta, tg.TG_C_BF16, tg.make_config(schedule=1, mma=2), None)
        assert st == tg.TG_OK and tg.tg_status_sync(None) == tg.TG_OK
        st = tg.gemm_bf16_noalloc(M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), K, C_new_dev.data_ptr(),
                                  N, 1.0, beta, tg.TG_C_BF16, status[call:].data_ptr(), None)
        assert st == tg.TG_OK
        torch.cuda.synchronize()
        assert int(status[call].item()) == 0

        existing, dp, new = c_to_f64(C_ref_dev), c_to_f64(C_dp_dev), c_to_f64(C_new_dev)
        ref, mag = oracle.gemm(A, B, M, N, K, C0=C0, beta=beta)
        c0v = gen.bf16_bits_to_f32(C0).astype(np.float64) if C0 is not None else None
        bound = gemm_bound(ref, mag, K, 1.0, beta, c0v, True)
        # gemm_bf16 may split tiles across clusters (stream-K) and so sum in another
        # order: both results lie within the bound of the exact product, hence within
        # twice the bound of each other.
        assert np.all(np.abs(new - existing) <= 2 * bound), "call %d" % call
        assert np.all(np.abs(new - ref) <= bound), "call %d" % call
        assert np.array_equal(new, dp), "call %d" % call
