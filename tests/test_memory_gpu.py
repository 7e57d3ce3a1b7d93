"""Every buffer a kernel reads or writes must be device memory of the current device.

A tensor map encodes a global address; through unified addressing a host or peer-GPU
pointer would be accepted by the encoder and the copies would then fetch that memory
over the interconnect (a cluster-multicast load included).  "2 . Le Tensor Memory
Accelerator" 2.3 lists the descriptor rules the library checks before encoding; this one
is the library's own: the maps cover this GPU's memory only.  Each rejected call must
return TG_ERR_INVALID_VALUE before anything is launched (C keeps its contents)."""
import numpy as np
import pytest

from tma_pipelined_tensor_gb300 import tg

pytestmark = pytest.mark.gpu


def _buffers(M=256, N=256, K=256):
    import torch
    A = torch.ones((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.ones((N, K), dtype=torch.bfloat16, device="cuda")
    C = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    return A, B, C


def _call(entry, A, B, C, M=256, N=256, K=256, cfg=None):
    if entry == "gemm_bf16":
        return tg.gemm_bf16(M, N, K, A, K, B, K, C, N, 1.0, 0.0, tg.TG_C_F32, None)
    if entry == "gemm_bf16_ex":
        return tg.gemm_bf16_ex(M, N, K, A, K, B, K, C, N, 1.0, 0.0, tg.TG_C_F32, cfg, None)
    return tg.gemm_bf16_noalloc(M, N, K, A, K, B, K, C, N, 1.0, 0.0, tg.TG_C_F32)


@pytest.mark.parametrize("entry", ["gemm_bf16", "gemm_bf16_ex", "gemm_bf16_noalloc"])
@pytest.mark.parametrize("which", ["A", "B", "C"])
@pytest.mark.parametrize("host", ["pinned", "pageable"])
def test_gemm_refuses_host_memory(entry, which, host):
    import torch
    A, B, C = _buffers()
    shape = {"A": A.shape, "B": B.shape, "C": C.shape}[which]
    dt = torch.float32 if which == "C" else torch.bfloat16
    h = torch.zeros(shape, dtype=dt, pin_memory=(host == "pinned"))
    ptrs = {"A": A.data_ptr(), "B": B.data_ptr(), "C": C.data_ptr()}
    ptrs[which] = h.data_ptr()
    st = _call(entry, ptrs["A"], ptrs["B"], ptrs["C"])
    assert st == tg.TG_ERR_INVALID_VALUE, tg.tg_status_string(st)
    torch.cuda.synchronize()
    assert tg.tg_status_sync(None) == tg.TG_OK
    assert bool((C == 7.0).all())            # nothing was launched
    assert bool((h == 0).all())


def test_multicast_config_refuses_host_memory_and_runs_on_device_memory():
    import torch
    A, B, C = _buffers()
    cfg = tg.make_config(cluster=2, mma=1)
    h = torch.ones(A.shape, dtype=torch.bfloat16, pin_memory=True)
    st = _call("gemm_bf16_ex", h.data_ptr(), B.data_ptr(), C.data_ptr(), cfg=cfg)
    assert st == tg.TG_ERR_INVALID_VALUE
    # this process sees one device, so the single-GPU multicast option is allowed
    assert torch.cuda.device_count() == 1
    st = _call("gemm_bf16_ex", A.data_ptr(), B.data_ptr(), C.data_ptr(), cfg=cfg)
    assert st == tg.TG_OK
    assert tg.tg_status_sync(None) == tg.TG_OK
    assert bool((C == 256.0).all())          # ones . ones = K


def test_k_zero_checks_only_c():
    import torch
    C = torch.full((64, 64), 2.0, dtype=torch.float32, device="cuda")
    st = tg.gemm_bf16(64, 64, 0, None, 0, None, 0, C.data_ptr(), 64, 1.0, 0.5, tg.TG_C_F32, None)
    assert st == tg.TG_OK and tg.tg_status_sync(None) == tg.TG_OK
    assert bool((C == 1.0).all())
    h = torch.full((64, 64), 2.0, dtype=torch.float32, pin_memory=True)
    st = tg.gemm_bf16(64, 64, 0, None, 0, None, 0, h.data_ptr(), 64, 1.0, 0.5, tg.TG_C_F32, None)
    assert st == tg.TG_ERR_INVALID_VALUE
    assert bool((h == 2.0).all())


@pytest.mark.parametrize("which", ["tensor", "image"])
def test_tile_copy_refuses_host_memory(which):
    import torch
    H, W = 256, 128
    T = torch.arange(H * W, dtype=torch.int32).to(torch.bfloat16).reshape(H, W)
    Td = T.cuda()
    nbytes = tg.image_bytes(H, W, 2, 64, 128)
    img = torch.full((nbytes,), 0x5A, dtype=torch.uint8, device="cuda")
    if which == "tensor":
        src, dst = T.pin_memory(), img
    else:
        src, dst = Td, torch.full((nbytes,), 0x5A, dtype=torch.uint8, pin_memory=True)
    t = tg.make_tensor2d(src.data_ptr(), tg.TG_DTYPE_BF16, W, H, W * 2)
    b = tg.make_box(64, 128)
    st = tg.tma_tile_copy(t, b, tg.TG_SWZ_128B, tg.TG_OOB_ZERO, dst.data_ptr(), nbytes, None)
    assert st == tg.TG_ERR_INVALID_VALUE, tg.tg_status_string(st)
    torch.cuda.synchronize()
    assert bool((dst == 0x5A).all())


def test_rate_probe_refuses_host_timing_words():
    import torch
    h = torch.zeros(2, dtype=torch.int64, pin_memory=True)
    st, _, _ = tg.tensor_rate_probe_timed(h.data_ptr(), tg.TG_IN_BF16, 16)
    assert st == tg.TG_ERR_INVALID_VALUE


def test_driver_symbol_lookup_on_a_gpu():
    # the real encoder is exported; a name the driver lacks is reported as such
    assert tg.tg_driver_symbol_status("cuTensorMapEncodeTiled") == tg.TG_OK
    assert tg.tg_driver_symbol_status("cuTensorMapEncodeTiledThatDoesNotExist") == \
        tg.TG_ERR_NO_DRIVER_SYMBOL


def test_first_call_from_a_new_host_thread():
    """A host thread's first GEMM and tile copy, after the main thread has used the library
    (its attribute and occupancy answers are cached), bind the device's context themselves
    before encoding their tensor maps, and give the same results as the main thread."""
    import threading

    import torch
    M, N, K = 640, 520, 384
    A = torch.randn(M, K, device="cuda").to(torch.bfloat16)
    B = torch.randn(N, K, device="cuda").to(torch.bfloat16)
    C_main = torch.empty(M, N, device="cuda")
    C_thread = torch.full((M, N), float("nan"), device="cuda")
    T = torch.randn(300, 200, device="cuda").to(torch.bfloat16)
    img_main = torch.empty(tg.image_bytes(300, 200, 2, 64, 128), dtype=torch.uint8, device="cuda")
    img_thread = torch.zeros_like(img_main)
    tg.gemm(A, B, C_main)
    tg.tile_copy(T, 64, 128, tg.TG_SWZ_128B, img_main)
    torch.cuda.synchronize()
    out = {}

    def worker():
        out["gemm"] = tg.gemm_bf16_ex(M, N, K, A.data_ptr(), K, B.data_ptr(), K,
                                      C_thread.data_ptr(), N, 1.0, 0.0, tg.TG_C_F32, None, None)
        out["copy"] = tg.tile_copy(T, 64, 128, tg.TG_SWZ_128B, img_thread, check=False)
        out["sync"] = tg.tg_status_sync(None)

    t = threading.Thread(target=worker)
    t.start()
    t.join()
    assert out == {"gemm": tg.TG_OK, "copy": tg.TG_OK, "sync": tg.TG_OK}, out
    torch.cuda.synchronize()
    assert torch.equal(C_main, C_thread)
    assert torch.equal(img_main, img_thread)
