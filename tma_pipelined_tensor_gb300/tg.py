"""Thin ctypes binding of the C ABI in include/tg.h (argument marshalling only).

Every function here forwards to libtg.so; nothing is computed in Python and there is
no fallback: if the library is missing, loading raises.  The names match the C entry
points.  Convenience wrappers at the bottom accept torch tensors and take their
device pointers, leading dimensions and the current CUDA stream.
"""
import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtg.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "tg.h")

# tg_status
TG_OK = 0
TG_ERR_INVALID_VALUE = 1
TG_ERR_MISALIGNED = 2
TG_ERR_UNSUPPORTED = 3
TG_ERR_BUFFER_TOO_SMALL = 4
TG_ERR_CUDA = 5
TG_ERR_NO_DRIVER_SYMBOL = 6
TG_ERR_DEVICE_TIMEOUT = 7

# layout bits
TG_LAYOUT_A_MN_MAJOR = 0x1
TG_LAYOUT_B_MN_MAJOR = 0x2
TG_C_F32 = 0 << 2
TG_C_BF16 = 1 << 2
TG_C_F16 = 2 << 2
TG_IN_BF16 = 0 << 4
TG_IN_F16 = 1 << 4
TG_IN_E4M3 = 2 << 4
TG_IN_E5M2 = 3 << 4
TG_IN_TF32 = 4 << 4
TG_IN_MXE4M3 = 5 << 4
TG_IN_MXE5M2 = 6 << 4

TG_GEMM_FLAG_TEST_SKIP_FIRST_LOAD = 0x1
TG_GEMM_FLAG_NO_SPLIT_TAIL = 0x2

# tg_dtype / tg_swizzle / tg_oob
TG_DTYPE_U8, TG_DTYPE_BF16, TG_DTYPE_F16, TG_DTYPE_F32 = 0, 1, 2, 3
TG_SWZ_NONE, TG_SWZ_32B, TG_SWZ_64B, TG_SWZ_128B = 0, 1, 2, 3
TG_OOB_ZERO, TG_OOB_NAN = 0, 1


class tg_gemm_config(ctypes.Structure):
    _fields_ = [("stages", ctypes.c_uint32), ("cluster", ctypes.c_uint32),
                ("tile_n", ctypes.c_uint32), ("group_m", ctypes.c_uint32),
                ("max_ctas", ctypes.c_uint32), ("flags", ctypes.c_uint32),
                ("timeout_ns", ctypes.c_uint64), ("mma", ctypes.c_uint32),
                ("schedule", ctypes.c_uint32), ("epi_bufs", ctypes.c_uint32),
                ("reserved", ctypes.c_uint32), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_uint64)]


class tg_gemm_plan(ctypes.Structure):
    _fields_ = [("tile_m", ctypes.c_uint32), ("tile_n", ctypes.c_uint32),
                ("tile_k", ctypes.c_uint32), ("stages", ctypes.c_uint32),
                ("cluster", ctypes.c_uint32), ("tiles_m", ctypes.c_uint64),
                ("tiles_n", ctypes.c_uint64), ("k_blocks", ctypes.c_uint64),
                ("grid", ctypes.c_uint32), ("smem_bytes", ctypes.c_uint32),
                ("stage_bytes", ctypes.c_uint32), ("mma", ctypes.c_uint32),
                ("dp_units", ctypes.c_uint32), ("sk_iters", ctypes.c_uint64),
                ("split_units", ctypes.c_uint32), ("workspace_bytes", ctypes.c_uint64),
                ("workspace", ctypes.c_uint32), ("sk_fallback", ctypes.c_uint32)]


class tg_tensor2d(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("dtype", ctypes.c_uint32),
                ("rank", ctypes.c_uint32), ("dims", ctypes.c_uint64 * 2),
                ("stride_bytes", ctypes.c_uint64)]


class tg_box(ctypes.Structure):
    _fields_ = [("inner", ctypes.c_uint32), ("outer", ctypes.c_uint32)]


class tg_copy_config(ctypes.Structure):
    _fields_ = [("stages", ctypes.c_uint32), ("blocks_per_sm", ctypes.c_uint32),
                ("order", ctypes.c_uint32), ("l2_promotion", ctypes.c_uint32)]


class tg_tensor_nd(ctypes.Structure):
    _fields_ = [("base", ctypes.c_void_p), ("dtype", ctypes.c_uint32), ("rank", ctypes.c_uint32),
                ("dims", ctypes.c_uint64 * 5), ("strides", ctypes.c_uint64 * 4)]


class tg_box_nd(ctypes.Structure):
    _fields_ = [("extent", ctypes.c_uint32 * 5), ("element_strides", ctypes.c_uint32 * 5)]


class TgError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = int(status)
        super().__init__("%s%s" % (what + ": " if what else "", tg_status_string(status)))


_LIB = None
_i64, _u32, _f32, _vp = ctypes.c_int64, ctypes.c_uint32, ctypes.c_float, ctypes.c_void_p
_st = ctypes.c_int


def lib():
    """The loaded libtg.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libtg.so is missing (%s): build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    L.tg_status_string.argtypes = [_st]
    L.tg_status_string.restype = ctypes.c_char_p
    L.tg_status_sync.argtypes = [_vp]
    L.tg_status_sync.restype = _st
    L.tg_driver_symbol_status.argtypes = [ctypes.c_char_p]
    L.tg_driver_symbol_status.restype = _st
    L.tg_status_detail.argtypes = []
    L.tg_status_detail.restype = _u32
    L.gemm_bf16.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _f32, _f32,
                            _u32, _vp]
    L.gemm_bf16.restype = _st
    L.gemm_bf16_ex.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _f32, _f32,
                               _u32, ctypes.POINTER(tg_gemm_config), _vp]
    L.gemm_bf16_ex.restype = _st
    L.gemm_bf16_noalloc.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _f32,
                                    _f32, _u32, _vp, _vp]
    L.gemm_bf16_noalloc.restype = _st
    L.gemm_mx.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _vp, _i64, _vp, _vp, _i64, _f32,
                          _f32, _u32, ctypes.POINTER(tg_gemm_config), _vp]
    L.gemm_mx.restype = _st
    L.gemm_mx_scale_bytes.argtypes = [_i64, _i64]
    L.gemm_mx_scale_bytes.restype = ctypes.c_size_t
    L.tg_gemm_config_default.argtypes = [ctypes.POINTER(tg_gemm_config)]
    L.tg_gemm_config_default.restype = None
    L.tg_gemm_plan_for.argtypes = [_i64, _i64, _i64, _u32, ctypes.POINTER(tg_gemm_config), _u32,
                                   ctypes.POINTER(tg_gemm_plan)]
    L.tg_gemm_plan_for.restype = _st
    L.tg_gemm_plan_ld.argtypes = [_i64, _i64, _i64, _i64, _i64, _u32,
                                  ctypes.POINTER(tg_gemm_config), _u32, ctypes.POINTER(tg_gemm_plan)]
    L.tg_gemm_plan_ld.restype = _st
    L.tg_gemm_last_plan.argtypes = [ctypes.POINTER(tg_gemm_plan)]
    L.tg_gemm_last_plan.restype = _st
    L.tma_validate.argtypes = [ctypes.POINTER(tg_tensor2d), ctypes.POINTER(tg_box), _st]
    L.tma_validate.restype = _st
    L.tma_tile_copy_image_bytes.argtypes = [ctypes.POINTER(tg_tensor2d), ctypes.POINTER(tg_box)]
    L.tma_tile_copy_image_bytes.restype = ctypes.c_size_t
    L.tma_tile_copy.argtypes = [ctypes.POINTER(tg_tensor2d), ctypes.POINTER(tg_box), _st, _st, _vp,
                                ctypes.c_size_t, _vp]
    L.tma_tile_copy.restype = _st
    L.tma_tile_copy_ex.argtypes = [ctypes.POINTER(tg_tensor2d), ctypes.POINTER(tg_box), _st, _st,
                                   _vp, ctypes.c_size_t, ctypes.POINTER(tg_copy_config), _vp]
    L.tma_tile_copy_ex.restype = _st
    L.tma_validate_nd.argtypes = [ctypes.POINTER(tg_tensor_nd), ctypes.POINTER(tg_box_nd), _st]
    L.tma_validate_nd.restype = _st
    L.tma_tile_copy_nd_image_bytes.argtypes = [ctypes.POINTER(tg_tensor_nd),
                                               ctypes.POINTER(tg_box_nd)]
    L.tma_tile_copy_nd_image_bytes.restype = ctypes.c_size_t
    L.tma_tile_copy_nd.argtypes = [ctypes.POINTER(tg_tensor_nd), ctypes.POINTER(tg_box_nd), _st,
                                   _st, _vp, ctypes.c_size_t, ctypes.POINTER(tg_copy_config), _vp]
    L.tma_tile_copy_nd.restype = _st
    _i32x5 = ctypes.c_int32 * 5
    _u32x5 = ctypes.c_uint32 * 5
    L.tg_tensor_rate_probe.argtypes = [ctypes.c_uint32, ctypes.c_uint64,
                                       ctypes.POINTER(ctypes.c_uint32), _vp]
    L.tg_tensor_rate_probe.restype = _st
    L.tg_tensor_rate_probe_timed.argtypes = [ctypes.c_uint32, ctypes.c_uint64,
                                             ctypes.POINTER(ctypes.c_uint32), _vp, _vp]
    L.tg_tensor_rate_probe_timed.restype = _st
    L.tma_tile_copy_back_nd.argtypes = [ctypes.POINTER(tg_tensor_nd), ctypes.POINTER(tg_box_nd), _st,
                                        _vp, ctypes.c_size_t, ctypes.POINTER(tg_copy_config), _vp]
    L.tma_tile_copy_back_nd.restype = _st
    L.tma_validate_region_nd.argtypes = [ctypes.POINTER(tg_tensor_nd), ctypes.POINTER(tg_box_nd),
                                         ctypes.POINTER(_i32x5), ctypes.POINTER(_u32x5), _st]
    L.tma_validate_region_nd.restype = _st
    L.tma_tile_copy_region_nd_image_bytes.argtypes = [ctypes.POINTER(tg_tensor_nd),
                                                      ctypes.POINTER(tg_box_nd),
                                                      ctypes.POINTER(_u32x5)]
    L.tma_tile_copy_region_nd_image_bytes.restype = ctypes.c_size_t
    L.tma_tile_copy_region_nd.argtypes = [ctypes.POINTER(tg_tensor_nd), ctypes.POINTER(tg_box_nd),
                                          ctypes.POINTER(_i32x5), ctypes.POINTER(_u32x5), _st, _st,
                                          _vp, ctypes.c_size_t, ctypes.POINTER(tg_copy_config), _vp]
    L.tma_tile_copy_region_nd.restype = _st
    _LIB = L
    return L


def declared_functions():
    """Names of the functions include/tg.h declares (for the export check)."""
    with open(HEADER_PATH, encoding="utf-8") as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


# ------------------------------------------------------------------------------------
# C entry points (same names)
# ------------------------------------------------------------------------------------
def tg_status_string(status):
    return lib().tg_status_string(int(status)).decode()


def tg_status_sync(stream=None):
    return lib().tg_status_sync(stream)


def tg_driver_symbol_status(symbol):
    return lib().tg_driver_symbol_status(None if symbol is None else symbol.encode())


def tg_status_detail():
    return lib().tg_status_detail()


def tg_gemm_config_default():
    c = tg_gemm_config()
    lib().tg_gemm_config_default(ctypes.byref(c))
    return c


def make_config(**kw):
    c = tg_gemm_config()
    for k, v in kw.items():
        setattr(c, k, int(v))
    return c


def gemm_bf16(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, layout, stream=None):
    return lib().gemm_bf16(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, layout, stream)


def gemm_bf16_ex(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, layout, cfg=None, stream=None):
    return lib().gemm_bf16_ex(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, layout,
                              ctypes.byref(cfg) if cfg is not None else None, stream)


def gemm_bf16_noalloc(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, layout, status_out=None,
                      stream=None):
    """The allocation-free GEMM entry point (status_out: device or pinned host address)."""
    return lib().gemm_bf16_noalloc(M, N, K, A, lda, B, ldb, C, ldc, alpha, beta, layout,
                                   status_out, stream)


def gemm_mx_raw(M, N, K, A, lda, sfa, B, ldb, sfb, C, ldc, alpha, beta, layout, cfg=None,
                stream=None):
    """The MX GEMM entry point on raw addresses (named gemm_mx in the C ABI)."""
    return lib().gemm_mx(M, N, K, A, lda, sfa, B, ldb, sfb, C, ldc, alpha, beta, layout,
                         ctypes.byref(cfg) if cfg is not None else None, stream)


def gemm_mx_scale_bytes(rows, K):
    return int(lib().gemm_mx_scale_bytes(rows, K))


def tg_gemm_plan_for(M, N, K, layout=TG_C_BF16, cfg=None, sm_count=0):
    plan = tg_gemm_plan()
    st = lib().tg_gemm_plan_for(M, N, K, layout, ctypes.byref(cfg) if cfg is not None else None,
                                sm_count, ctypes.byref(plan))
    return st, plan


def tg_gemm_plan_ld(M, N, K, lda, ldb, layout=TG_C_BF16, cfg=None, sm_count=0):
    plan = tg_gemm_plan()
    st = lib().tg_gemm_plan_ld(M, N, K, lda, ldb, layout,
                               ctypes.byref(cfg) if cfg is not None else None, sm_count,
                               ctypes.byref(plan))
    return st, plan


def tg_gemm_last_plan():
    plan = tg_gemm_plan()
    st = lib().tg_gemm_last_plan(ctypes.byref(plan))
    return st, plan


def make_tensor2d(base, dtype, inner, outer, stride_bytes, rank=2):
    t = tg_tensor2d()
    t.base = base
    t.dtype = dtype
    t.rank = rank
    t.dims[0] = inner
    t.dims[1] = outer
    t.stride_bytes = stride_bytes
    return t


def make_box(inner, outer):
    b = tg_box()
    b.inner, b.outer = inner, outer
    return b


def tma_validate(tensor, box, swizzle):
    return lib().tma_validate(ctypes.byref(tensor) if tensor is not None else None,
                              ctypes.byref(box) if box is not None else None, swizzle)


def tma_tile_copy_image_bytes(tensor, box):
    return lib().tma_tile_copy_image_bytes(ctypes.byref(tensor), ctypes.byref(box))


def tma_tile_copy(tensor, box, swizzle, oob, out, out_bytes, stream=None):
    return lib().tma_tile_copy(ctypes.byref(tensor), ctypes.byref(box), swizzle, oob, out,
                               out_bytes, stream)


def tma_tile_copy_ex(tensor, box, swizzle, oob, out, out_bytes, cfg=None, stream=None):
    return lib().tma_tile_copy_ex(ctypes.byref(tensor), ctypes.byref(box), swizzle, oob, out,
                                  out_bytes, ctypes.byref(cfg) if cfg is not None else None,
                                  stream)


def make_tensor_nd(base, dtype, dims, strides):
    """dims innermost first; strides = byte strides of dimensions 1.. (len(dims)-1)."""
    t = tg_tensor_nd()
    t.base, t.dtype, t.rank = base, dtype, len(dims)
    for i, d in enumerate(dims):
        t.dims[i] = d
    for i, st in enumerate(strides):
        t.strides[i] = st
    return t


def make_box_nd(extent, element_strides=None):
    b = tg_box_nd()
    element_strides = [1] * len(extent) if element_strides is None else element_strides
    for i, (e, st) in enumerate(zip(extent, element_strides)):
        b.extent[i], b.element_strides[i] = e, st
    return b


def tma_validate_nd(tensor, box, swizzle):
    return lib().tma_validate_nd(ctypes.byref(tensor) if tensor is not None else None,
                                 ctypes.byref(box) if box is not None else None, swizzle)


def tma_tile_copy_nd_image_bytes(tensor, box):
    return lib().tma_tile_copy_nd_image_bytes(ctypes.byref(tensor), ctypes.byref(box))


def tma_tile_copy_nd(tensor, box, swizzle, oob, out, out_bytes, cfg=None, stream=None):
    return lib().tma_tile_copy_nd(ctypes.byref(tensor), ctypes.byref(box), swizzle, oob, out,
                                  out_bytes, ctypes.byref(cfg) if cfg is not None else None,
                                  stream)


def _i32x5(v):
    a = (ctypes.c_int32 * 5)()
    for i, x in enumerate(v):
        a[i] = x
    return a


def _u32x5(v):
    a = (ctypes.c_uint32 * 5)()
    for i, x in enumerate(v):
        a[i] = x
    return a


def tma_tile_copy_back_nd(tensor, box, swizzle, image, image_bytes, cfg=None, stream=None):
    return lib().tma_tile_copy_back_nd(ctypes.byref(tensor), ctypes.byref(box), swizzle, image,
                                       image_bytes, ctypes.byref(cfg) if cfg is not None else None,
                                       stream)


def tma_validate_region_nd(tensor, box, origin, nboxes, swizzle):
    """origin / nboxes: sequences (innermost first), or None to pass NULL."""
    return lib().tma_validate_region_nd(
        ctypes.byref(tensor), ctypes.byref(box),
        ctypes.byref(_i32x5(origin)) if origin is not None else None,
        ctypes.byref(_u32x5(nboxes)) if nboxes is not None else None, swizzle)


def tma_tile_copy_region_nd_image_bytes(tensor, box, nboxes):
    return lib().tma_tile_copy_region_nd_image_bytes(ctypes.byref(tensor), ctypes.byref(box),
                                                     ctypes.byref(_u32x5(nboxes)))


def tma_tile_copy_region_nd(tensor, box, origin, nboxes, swizzle, oob, out, out_bytes, cfg=None,
                            stream=None):
    return lib().tma_tile_copy_region_nd(
        ctypes.byref(tensor), ctypes.byref(box), ctypes.byref(_i32x5(origin)),
        ctypes.byref(_u32x5(nboxes)), swizzle, oob, out, out_bytes,
        ctypes.byref(cfg) if cfg is not None else None, stream)


# ------------------------------------------------------------------------------------
# torch conveniences (marshalling only)
# ------------------------------------------------------------------------------------
_RAW_STREAM = None


def _stream_handle(stream):
    """cudaStream_t of `stream`, or of the current device's current stream."""
    global _RAW_STREAM
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    import torch
    if _RAW_STREAM is None:
        # the raw current-stream query avoids building a Stream object on every call
        _RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", False)
    if _RAW_STREAM:
        return ctypes.c_void_p(_RAW_STREAM(torch.cuda.current_device()))
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _row_major_ld(t, name):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("%s must be a 2-D tensor with unit inner stride" % name)
    return t.stride(0)


def _operand_ld(t, name):
    """(leading dimension, MN-major?) of a 2-D operand view: unit stride along its second
    index is the K-major storage, unit stride along its first index the MN-major one."""
    if t.dim() != 2:
        raise ValueError("%s must be 2-D" % name)
    if t.stride(1) == 1:
        return t.stride(0), False
    if t.stride(0) == 1:
        return t.stride(1), True
    raise ValueError("%s needs a unit stride along one index" % name)


_TYPE_BITS = None


def _gemm_type_bits():
    """(operand dtype -> layout bits 4-6, C dtype -> layout bits 2-3), built once."""
    global _TYPE_BITS
    if _TYPE_BITS is None:
        import torch
        _TYPE_BITS = ({torch.bfloat16: TG_IN_BF16, torch.float16: TG_IN_F16,
                       torch.float8_e4m3fn: TG_IN_E4M3, torch.float8_e5m2: TG_IN_E5M2,
                       torch.float32: TG_IN_TF32},
                      {torch.float32: TG_C_F32, torch.bfloat16: TG_C_BF16,
                       torch.float16: TG_C_F16})
    return _TYPE_BITS


def gemm(A, B, C, alpha=1.0, beta=0.0, config=None, stream=None, check=True):
    """C <- alpha * A @ B^T + beta * C on torch CUDA tensors: A is M x K, B is N x K (the K x N
    operand transposed), both bf16, fp16, float8_e4m3fn, float8_e5m2 or float32 (multiplied
    as tf32); 8-bit and float32 operands K-major;
    C is M x N fp32, bf16 or fp16 with unit inner stride.  A view of
    A with unit stride along M (or of B along N) is passed as the M-major (N-major) storage.
    Raises TgError on a host error."""
    in_bits, c_bits = _gemm_type_bits()
    M, K = A.shape
    N = B.shape[0]
    if A.dtype != B.dtype or A.dtype not in in_bits:
        raise TypeError("A and B must have one type: bf16, fp16, float8_e4m3fn, float8_e5m2 "
                        "or float32 (tf32)")
    if B.shape[1] != K or C.dim() != 2 or C.shape[0] != M or C.shape[1] != N:
        raise ValueError("shape mismatch")
    if C.dtype not in c_bits:
        raise TypeError("C must be fp32, bf16 or fp16")
    lda, a_mn = _operand_ld(A, "A")
    ldb, b_mn = _operand_ld(B, "B")
    layout = (c_bits[C.dtype] | in_bits[A.dtype]
              | (TG_LAYOUT_A_MN_MAJOR if a_mn else 0) | (TG_LAYOUT_B_MN_MAJOR if b_mn else 0))
    st = lib().gemm_bf16_ex(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, C.data_ptr(),
                            _row_major_ld(C, "C"), float(alpha), float(beta), layout,
                            ctypes.byref(config) if config is not None else None,
                            _stream_handle(stream))
    if check and st != TG_OK:
        raise TgError(st, "gemm_bf16")
    return st


def gemm_mx(A, SA, B, SB, C, alpha=1.0, beta=0.0, kind="e4m3", config=None, stream=None,
            check=True):
    """C <- alpha * (A . SA) * (B . SB)^T + beta * C with MX operands on torch CUDA
    tensors: A (M x K) and B (N x K) uint8 or float8 tensors of E4M3 / E5M2 bytes, K-major;
    SA, SB uint8 tensors of E8M0 scales in the atom layout (gemm_mx_scale_bytes each); C
    M x N fp32, bf16 or fp16.  Raises TgError on a host error."""
    c_bits = _gemm_type_bits()[1]
    M, K = A.shape
    N = B.shape[0]
    layout = c_bits[C.dtype] | (TG_IN_MXE5M2 if kind == "e5m2" else TG_IN_MXE4M3)
    st = lib().gemm_mx(M, N, K, A.data_ptr(), _row_major_ld(A, "A"), SA.data_ptr(), B.data_ptr(),
                       _row_major_ld(B, "B"), SB.data_ptr(), C.data_ptr(), _row_major_ld(C, "C"),
                       float(alpha), float(beta), layout,
                       ctypes.byref(config) if config is not None else None,
                       _stream_handle(stream))
    if check and st != TG_OK:
        raise TgError(st, "gemm_mx")
    return st


_TORCH_DTYPES = None


def _dtype_code(t):
    import torch
    global _TORCH_DTYPES
    if _TORCH_DTYPES is None:
        _TORCH_DTYPES = {torch.uint8: TG_DTYPE_U8, torch.bfloat16: TG_DTYPE_BF16,
                         torch.float16: TG_DTYPE_F16, torch.float32: TG_DTYPE_F32}
    return _TORCH_DTYPES[t.dtype]


def tile_copy(T, box_inner, box_outer, swizzle, out, oob=TG_OOB_ZERO, stream=None, check=True,
              stages=0, blocks_per_sm=0, order=0, l2_promotion=0):
    """Raw swizzled shared-memory image of every box of the 2-D CUDA tensor T into the
    uint8 CUDA tensor `out`."""
    ld = _row_major_ld(T, "T")
    t = make_tensor2d(T.data_ptr(), _dtype_code(T), T.shape[1], T.shape[0], ld * T.element_size())
    b = make_box(box_inner, box_outer)
    cfg = None
    if stages or blocks_per_sm or order or l2_promotion:
        cfg = tg_copy_config()
        cfg.stages, cfg.blocks_per_sm = stages, blocks_per_sm
        cfg.order, cfg.l2_promotion = order, l2_promotion
    st = tma_tile_copy_ex(t, b, swizzle, oob, out.data_ptr(), out.numel() * out.element_size(), cfg,
                          _stream_handle(stream))
    if check and st != TG_OK:
        raise TgError(st, "tma_tile_copy")
    return st


def image_bytes(rows, cols, elem_size, box_inner, box_outer):
    nbi = -(-rows // box_outer)
    nbj = -(-cols // box_inner)
    return nbi * nbj * box_inner * box_outer * elem_size


def tile_copy_nd(T, extent, element_strides, swizzle, out, oob=TG_OOB_ZERO, stream=None,
                 check=True):
    """Rank 1..5 tile copy of the CUDA tensor T (torch order: outermost index first, unit
    stride on the last); extent / element_strides are given innermost first."""
    if T.stride(-1) != 1:
        raise ValueError("the innermost dimension must be contiguous")
    dims = list(reversed(T.shape))
    strides = [T.stride(T.dim() - 1 - i) * T.element_size() for i in range(1, T.dim())]
    t = make_tensor_nd(T.data_ptr(), _dtype_code(T), dims, strides)
    b = make_box_nd(extent, element_strides)
    st = tma_tile_copy_nd(t, b, swizzle, oob, out.data_ptr(), out.numel() * out.element_size(),
                          None, _stream_handle(stream))
    if check and st != TG_OK:
        raise TgError(st, "tma_tile_copy_nd")
    return st


def tile_copy_region(T, extent, origin, nboxes, swizzle, out, element_strides=None,
                     oob=TG_OOB_ZERO, stream=None, check=True):
    """Region copy of the CUDA tensor T (torch order: outermost index first, unit stride on
    the last): the box grid starts at index `origin` (may be negative) with `nboxes`
    boxes per dimension; extent, origin, nboxes and element_strides innermost first."""
    if T.stride(-1) != 1:
        raise ValueError("the innermost dimension must be contiguous")
    dims = list(reversed(T.shape))
    strides = [T.stride(T.dim() - 1 - i) * T.element_size() for i in range(1, T.dim())]
    t = make_tensor_nd(T.data_ptr(), _dtype_code(T), dims, strides)
    b = make_box_nd(extent, element_strides)
    st = tma_tile_copy_region_nd(t, b, origin, nboxes, swizzle, oob, out.data_ptr(),
                                 out.numel() * out.element_size(), None, _stream_handle(stream))
    if check and st != TG_OK:
        raise TgError(st, "tma_tile_copy_region_nd")
    return st


def tile_copy_back(T, extent, swizzle, image, stream=None, check=True):
    """Writes the box image `image` (as tile_copy_nd produces it for T, extent and
    swizzle) back into the CUDA tensor T."""
    if T.stride(-1) != 1:
        raise ValueError("the innermost dimension must be contiguous")
    dims = list(reversed(T.shape))
    strides = [T.stride(T.dim() - 1 - i) * T.element_size() for i in range(1, T.dim())]
    t = make_tensor_nd(T.data_ptr(), _dtype_code(T), dims, strides)
    b = make_box_nd(extent)
    st = tma_tile_copy_back_nd(t, b, swizzle, image.data_ptr(),
                               image.numel() * image.element_size(), None, _stream_handle(stream))
    if check and st != TG_OK:
        raise TgError(st, "tma_tile_copy_back_nd")
    return st


def tensor_rate_probe(layout=TG_IN_BF16, iters=1 << 14, stream=None):
    """Runs the tensor-core rate probe; returns (status, pairs, flops of the launch)."""
    pairs = ctypes.c_uint32(0)
    st = lib().tg_tensor_rate_probe(layout, iters, ctypes.byref(pairs), _stream_handle(stream))
    return st, pairs.value, _probe_flops(layout, iters, pairs.value)


def _probe_flops(layout, iters, pairs):
    kind = (layout >> 4) & 7
    k_mma = 8 if kind == 4 else 32 if kind in (2, 3) else 16
    return pairs * iters * 4 * 2 * 256 * 256 * k_mma


def tensor_rate_probe_timed(timing, layout=TG_IN_BF16, iters=1 << 14, stream=None):
    """The probe with its own clock: `timing` is a device address of two uint64 (SM cycles,
    nanoseconds of the first pair's MMA loop), valid after the stream is synchronised.
    Returns (status, pairs, flops of the launch)."""
    pairs = ctypes.c_uint32(0)
    st = lib().tg_tensor_rate_probe_timed(layout, iters, ctypes.byref(pairs), timing,
                                          _stream_handle(stream))
    return st, pairs.value, _probe_flops(layout, iters, pairs.value)
