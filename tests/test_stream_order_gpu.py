"""Stream order with programmatic dependent launch: GEMM and tile-copy kernels may start
their set-up while the kernel before them drains, but read nothing in global memory before
it has completed.  Each test issues a producer and a consumer back to back on one stream,
with no synchronisation between them, into buffers pre-filled with NaN: a consumer that
read early would carry NaNs or stale values into its result.

Results are compared with the fp64 oracle at |C - C_ref| <= 2*K*2^-24*(|A||B|) +
2^-8*|C_ref| (bf16 C)."""
import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_gb300 import inputs as gen
from tma_pipelined_tensor_gb300 import tg

from gpu_util import assert_within, c_to_f64, gemm_bound, to_device_bf16

pytestmark = pytest.mark.gpu

NAN_BF16 = 0x7FC0


@pytest.mark.parametrize("cfg1,cfg2", [
    (dict(), dict()),                       # CTA pair after CTA pair
    (dict(mma=1), dict(mma=2)),             # per-CTA kernel, then the pair
    (dict(mma=2, schedule=2), dict(mma=1)),  # stream-K pair, then the per-CTA kernel
])
def test_gemm_reads_the_previous_gemms_output(cfg1, cfg2):
    import torch
    M, K1, N1, N2 = 1024, 512, 768, 640
    A = gen.bf16_matrix(M, K1, 31, 0, "normal")
    B1 = gen.bf16_matrix(N1, K1, 31, 1, "normal")
    B2 = gen.bf16_matrix(N2, N1, 31, 2, "normal")
    Ad, B1d, B2d = to_device_bf16(A), to_device_bf16(B1), to_device_bf16(B2)
    C1 = torch.full((M, N1), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    C2 = torch.full((M, N2), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    torch.cuda.synchronize()
    for _ in range(3):   # the second product reads the first one's output as its A
        tg.gemm(Ad, B1d, C1, config=tg.make_config(**cfg1) if cfg1 else None)
        tg.gemm(C1, B2d, C2, config=tg.make_config(**cfg2) if cfg2 else None)
        C1.view(torch.int16).fill_(NAN_BF16)
    tg.gemm(Ad, B1d, C1, config=tg.make_config(**cfg1) if cfg1 else None)
    tg.gemm(C1, B2d, C2, config=tg.make_config(**cfg2) if cfg2 else None)
    assert tg.tg_status_sync(None) == tg.TG_OK
    c1 = C1.view(torch.int16).cpu().numpy().view(np.uint16)
    ref1, mag1 = oracle.gemm(A, B1, M, N1, K1)
    assert_within(gen.bf16_bits_to_f32(c1).astype(np.float64), ref1,
                  gemm_bound(ref1, mag1, K1, 1.0, 0.0, None, True), "first product")
    ref2, mag2 = oracle.gemm(c1, B2, M, N2, N1)
    assert_within(c_to_f64(C2), ref2, gemm_bound(ref2, mag2, N1, 1.0, 0.0, None, True),
                  "second product, issued right after the first")


def test_gemm_reads_a_tensor_a_copy_just_wrote():
    """tile_copy_back restores A from its swizzled image; the GEMM issued right after it
    reads that A."""
    import torch
    M, N, K = 512, 384, 640
    A = gen.bf16_matrix(M, K, 37, 0, "normal")
    B = gen.bf16_matrix(N, K, 37, 1, "normal")
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    img = torch.empty(tg.image_bytes(M, K, 2, 64, 128), dtype=torch.uint8, device="cuda")
    tg.tile_copy(Ad, 64, 128, tg.TG_SWZ_128B, img)
    A_back = torch.full((M, K), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    C = torch.full((M, N), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    torch.cuda.synchronize()
    assert tg.tile_copy_back(A_back, [64, 128], tg.TG_SWZ_128B, img) == tg.TG_OK
    tg.gemm(A_back, Bd, C)
    assert tg.tg_status_sync(None) == tg.TG_OK
    assert torch.equal(A_back.view(torch.int16), Ad.view(torch.int16))
    ref, mag = oracle.gemm(A, B, M, N, K)
    assert_within(c_to_f64(C), ref, gemm_bound(ref, mag, K, 1.0, 0.0, None, True),
                  "GEMM right after the copy")


def test_copy_reads_the_previous_gemms_output():
    """A tile copy issued right after a GEMM images the GEMM's C, not the NaNs before it."""
    import torch
    M, N, K = 640, 512, 256
    A = gen.bf16_matrix(M, K, 41, 0, "normal")
    B = gen.bf16_matrix(N, K, 41, 1, "normal")
    Ad, Bd = to_device_bf16(A), to_device_bf16(B)
    C = torch.full((M, N), NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    img = torch.empty(tg.image_bytes(M, N, 2, 64, 128), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    tg.gemm(Ad, Bd, C)
    tg.tile_copy(C, 64, 128, tg.TG_SWZ_128B, img)
    assert tg.tg_status_sync(None) == tg.TG_OK
    c = C.view(torch.int16).cpu().numpy().view(np.uint16)
    want = oracle.tma_box_images(c, M, N, N * 2, 2, 64, 128, tg.TG_SWZ_128B)
    assert np.array_equal(img.cpu().numpy(), want)
    assert not np.isnan(gen.bf16_bits_to_f32(c)).any()
