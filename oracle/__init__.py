"""CPU oracle for the TMA-fed bf16 GEMM and the TMA tile-copy path.

TEST INFRASTRUCTURE ONLY: only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package.  It shares no code with the CUDA library
(`tma_pipelined_tensor_gb300`) and never imports it; inputs reach both sides from the
seeded generators, which hold none of the method's arithmetic.

The arithmetic lives in `oracle.c` (plain C, fp64); this module only marshals numpy
arrays into it.  See the C file's header for the pages it restates and the readings
it takes where they are silent.

Parity status: the GEMM definition and the swizzle/zero-fill model are pinned by the
CPU tests (closed forms, brute force, page bit maps, invariants).  The bit pattern of
the NaN out-of-bounds fill is "parity unpinned": the pages do not state it, so only
`isnan` is checked at those positions.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None

_i64 = ctypes.c_int64
_dbl = ctypes.c_double
_int = ctypes.c_int
_vp = ctypes.c_void_p


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        lib.oracle_gemm_rows.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _int, _vp,
                                         _int, _i64, _dbl, _dbl, _i64, _i64, _vp, _vp]
        lib.oracle_gemm_rows.restype = None
        lib.oracle_gemm_entries.argtypes = [_i64, _vp, _i64, _vp, _i64, _int, _vp, _int, _i64,
                                            _dbl, _dbl, _i64, _vp, _vp, _vp, _vp]
        lib.oracle_gemm_entries.restype = None
        lib.oracle_swizzle.argtypes = [ctypes.c_uint64, _int]
        lib.oracle_swizzle.restype = ctypes.c_uint64
        lib.oracle_tma_box_images.argtypes = [_vp, _i64, _i64, _i64, _int, _i64, _i64,
                                              _int, _int, _i64, _i64, _vp]
        lib.oracle_tma_box_images.restype = None
        lib.oracle_tma_box_images_nd.argtypes = [_vp, _int, _vp, _vp, _int, _vp, _vp, _int,
                                                 _int, _i64, _i64, _vp]
        lib.oracle_tma_box_images_nd.restype = None
        lib.oracle_tma_box_images_region.argtypes = [_vp, _int, _vp, _vp, _int, _vp, _vp, _vp,
                                                     _vp, _int, _int, _i64, _i64, _vp]
        lib.oracle_tma_box_images_region.restype = None
        lib.oracle_tf32_to_double.argtypes = [ctypes.c_uint32]
        lib.oracle_tf32_to_double.restype = _dbl
        lib.oracle_f8_to_double.argtypes = [ctypes.c_uint8, _int]
        lib.oracle_f8_to_double.restype = _dbl
        lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_double.restype = _dbl
        lib.oracle_e8m0_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e8m0_to_double.restype = _dbl
        lib.oracle_mx_scale_offset.argtypes = [_i64, _i64, _i64]
        lib.oracle_mx_scale_offset.restype = _i64
        lib.oracle_gemm_mx_entries.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _vp, _i64, _vp,
                                               _int, _vp, _int, _i64, _dbl, _dbl, _i64, _vp,
                                               _vp, _vp, _vp]
        lib.oracle_gemm_mx_entries.restype = None
        lib.oracle_omp_threads.argtypes = []
        lib.oracle_omp_threads.restype = _int
        _LIB = lib
    return _LIB


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c_dtype(C0, c_f16=False):
    if C0 is None:
        return 0
    if C0.dtype == np.uint16:
        return 2 if c_f16 else 1
    if C0.dtype == np.float32:
        return 0
    raise TypeError("C0 must be 16-bit patterns (uint16) or float32")


def f16_value(bits: int) -> float:
    """The oracle's own decoding of one fp16 pattern."""
    return float(_lib().oracle_f16_to_double(int(bits) & 0xFFFF))


def f8_value(bits: int, e5m2: bool = False) -> float:
    """The oracle's own decoding of one E4M3 (or E5M2) pattern."""
    return float(_lib().oracle_f8_to_double(int(bits) & 0xFF, 1 if e5m2 else 0))


def tf32_value(bits: int) -> float:
    """The oracle's own reading of one binary32 pattern as a tf32 operand."""
    return float(_lib().oracle_tf32_to_double(int(bits) & 0xFFFFFFFF))


IN_KINDS = {"bf16": 0, "f16": 1, "e4m3": 2, "e5m2": 3, "tf32": 4}


def _operand_array(X, kind):
    if kind == 4:
        X = np.ascontiguousarray(X)
        return X.view(np.uint32) if X.dtype == np.float32 else np.ascontiguousarray(X, np.uint32)
    return np.ascontiguousarray(X, dtype=np.uint8 if kind >= 2 else np.uint16)


def threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(_lib().oracle_omp_threads())


def gemm(A, B, M, N, K, lda=None, ldb=None, C0=None, ldc=None, alpha=1.0, beta=0.0,
         rows=None, a_mn=False, b_mn=False, in_f16=False, c_f16=False, in_kind=None):
    """C = alpha * A * B + beta * C0, in fp64 (C_ij = sum_k A_ik B_kj).

    A: uint16 bf16 bits; K-major (default): M rows of lda elements (element (i,k) at
    A[i*lda + k]); a_mn: K rows of lda elements (element (i,k) at A[k*lda + i]).
    B: uint16 bf16 bits of the K x N operand; K-major (default): stored as N rows of ldb
    elements (element (k,j) at B[j*ldb + k]); b_mn: K rows of ldb elements (B[k*ldb + j]).
    in_f16: A and B hold fp16 patterns instead of bf16; in_kind ("bf16", "f16", "e4m3",
    "e5m2", "tf32") names the operand type explicitly (8-bit types as uint8 arrays, tf32
    as float32 or uint32 binary32 patterns, truncated to 10 mantissa bits).
    C0: None, float32, or uint16 patterns (bf16, or fp16 with c_f16), M rows of ldc.
    `rows` = (row0, row1) restricts the computation to a band of rows.  Returns
    (C, absprod) as float64 arrays of shape (row1-row0, N); absprod[i, j] =
    sum_k |A_ik| |B_kj|.
    """
    kind = IN_KINDS[in_kind] if in_kind else (1 if in_f16 else 0)
    A = _operand_array(A, kind)
    B = _operand_array(B, kind)
    lda = (M if a_mn else K) if lda is None else lda
    ldb = (N if b_mn else K) if ldb is None else ldb
    layout = (1 if a_mn else 0) | (2 if b_mn else 0) | (kind << 4)
    if C0 is not None:
        C0 = np.ascontiguousarray(C0)
        ldc = N if ldc is None else ldc
    else:
        ldc = N if ldc is None else ldc
        if beta != 0.0:
            raise ValueError("beta != 0 needs C0")
    row0, row1 = (0, M) if rows is None else rows
    row1 = min(row1, M)
    out = np.empty((max(row1 - row0, 0), N), dtype=np.float64)
    absprod = np.empty_like(out)
    if out.size:
        _lib().oracle_gemm_rows(M, N, K, _ptr(A), lda, _ptr(B), ldb, layout, _ptr(C0),
                                _c_dtype(C0, c_f16), ldc, float(alpha), float(beta),
                                row0, row1, _ptr(out), _ptr(absprod))
    return out, absprod


def gemm_entries(A, B, K, ii, jj, lda=None, ldb=None, C0=None, ldc=None, alpha=1.0,
                 beta=0.0, a_mn=False, b_mn=False, in_f16=False, c_f16=False, in_kind=None):
    """The GEMM definition evaluated at the sampled positions (ii[t], jj[t]); for the
    M-/N-major storages pass lda/ldb (they default to K)."""
    kind = IN_KINDS[in_kind] if in_kind else (1 if in_f16 else 0)
    A = _operand_array(A, kind)
    B = _operand_array(B, kind)
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    lda = K if lda is None else lda
    ldb = K if ldb is None else ldb
    layout = (1 if a_mn else 0) | (2 if b_mn else 0) | (kind << 4)
    if C0 is not None:
        C0 = np.ascontiguousarray(C0)
    if beta != 0.0 and C0 is None:
        raise ValueError("beta != 0 needs C0")
    ldc = 0 if ldc is None else ldc
    out = np.empty(ii.shape[0], dtype=np.float64)
    absprod = np.empty_like(out)
    if out.size:
        _lib().oracle_gemm_entries(K, _ptr(A), lda, _ptr(B), ldb, layout, _ptr(C0),
                                   _c_dtype(C0, c_f16),
                                   ldc, float(alpha), float(beta), ii.shape[0], _ptr(ii),
                                   _ptr(jj), _ptr(out), _ptr(absprod))
    return out, absprod


def e8m0_to_double(x: int) -> float:
    """Value of an E8M0 block scale: 2^(x - 127), NaN for 255."""
    return float(_lib().oracle_e8m0_to_double(int(x) & 0xFF))


def mx_scale_offset(rows: int, r: int, j: int) -> int:
    """Byte offset of the scale of row r, 32-element block j, in an operand of `rows` rows."""
    return int(_lib().oracle_mx_scale_offset(int(rows), int(r), int(j)))


def gemm_mx_entries(A, SA, B, SB, M, N, K, ii, jj, kind="e4m3", lda=None, ldb=None, C0=None,
                    ldc=None, alpha=1.0, beta=0.0):
    """C = alpha * A * B + beta * C0 with MX operands (FP8 elements, E8M0 scales per 32
    elements of K, in the scale atoms' byte layout), evaluated at (ii[t], jj[t]).  Returns
    (values, sum_k |a||b| of the scaled values)."""
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    SA = np.ascontiguousarray(SA, dtype=np.uint8)
    SB = np.ascontiguousarray(SB, dtype=np.uint8)
    ii = np.ascontiguousarray(ii, dtype=np.int64)
    jj = np.ascontiguousarray(jj, dtype=np.int64)
    lda = K if lda is None else lda
    ldb = K if ldb is None else ldb
    if C0 is not None:
        C0 = np.ascontiguousarray(C0)
    if beta != 0.0 and C0 is None:
        raise ValueError("beta != 0 needs C0")
    out = np.empty(ii.shape[0], dtype=np.float64)
    absprod = np.empty_like(out)
    if out.size:
        _lib().oracle_gemm_mx_entries(M, N, K, _ptr(A), lda, _ptr(SA), _ptr(B), ldb, _ptr(SB),
                                      IN_KINDS[kind], _ptr(C0), _c_dtype(C0), 0 if ldc is None else ldc,
                                      float(alpha), float(beta), ii.shape[0], _ptr(ii), _ptr(jj),
                                      _ptr(out), _ptr(absprod))
    return out, absprod


def gemm_mx(A, SA, B, SB, M, N, K, kind="e4m3", lda=None, ldb=None, C0=None, ldc=None,
            alpha=1.0, beta=0.0):
    """All of C (M x N) with MX operands: (values, |a||b| sums), each M x N."""
    ii, jj = np.meshgrid(np.arange(M, dtype=np.int64), np.arange(N, dtype=np.int64),
                         indexing="ij")
    v, m = gemm_mx_entries(A, SA, B, SB, M, N, K, ii.ravel(), jj.ravel(), kind, lda, ldb, C0,
                           ldc, alpha, beta)
    return v.reshape(M, N), m.reshape(M, N)


def swizzle(a: int, mode: int) -> int:
    """Image byte offset of logical byte offset `a` (mode 0 none, 1 32B, 2 64B, 3 128B)."""
    return int(_lib().oracle_swizzle(int(a), int(mode)))


def box_grid(H, W, box_w, box_h):
    """(rows, columns) of the box grid covering an H x W tensor."""
    return (H + box_h - 1) // box_h, (W + box_w - 1) // box_w


def tma_box_images(T, H, W, stride, es, box_w, box_h, mode, oob_nan=False, boxes=None):
    """Raw image of boxes [b0, b1) (default: all) of the H x W tensor in `T`.

    T: uint8 view of the tensor bytes (H rows, `stride` bytes apart, W elements of `es`
    bytes each).  Returns a uint8 array of (b1-b0) * box_h * box_w * es bytes.
    """
    T = np.ascontiguousarray(T).view(np.uint8).reshape(-1)
    nbi, nbj = box_grid(H, W, box_w, box_h)
    b0, b1 = (0, nbi * nbj) if boxes is None else boxes
    box_bytes = box_h * box_w * es
    out = np.empty((b1 - b0) * box_bytes, dtype=np.uint8)
    if out.size:
        _lib().oracle_tma_box_images(_ptr(T), H, W, stride, es, box_w, box_h, mode,
                                     1 if oob_nan else 0, b0, b1, _ptr(out))
    return out


def box_grid_nd(dims, ext):
    """Boxes along each dimension (innermost first)."""
    return [(d + e - 1) // e for d, e in zip(dims, ext)]


def tma_box_images_nd(T, dims, strides, es, ext, estr, mode, oob_nan=False, boxes=None):
    """Raw image of boxes [b0, b1) (default: all) of a rank-1..5 tensor.

    T: the tensor's bytes (the buffer starting at element 0); dims: extents, innermost
    first; strides: byte strides of dimensions 1.. (len rank-1); es: element size; ext:
    traversal box per dimension; estr: element strides (estr[0] = 1)."""
    rank = len(dims)
    T = np.ascontiguousarray(T).view(np.uint8).reshape(-1)
    arr = lambda v: np.ascontiguousarray(np.array(list(v) + [1] * (5 - len(v)), dtype=np.int64))
    stride_all = arr([es] + list(strides))
    nb = box_grid_nd(dims, ext)
    total = int(np.prod(nb))
    b0, b1 = (0, total) if boxes is None else boxes
    L = [(e + s - 1) // s for e, s in zip(ext, estr)]
    box_bytes = int(np.prod(L)) * es
    out = np.empty((b1 - b0) * box_bytes, dtype=np.uint8)
    d, st, ex, sr = arr(dims), stride_all, arr(ext), arr(estr)
    if out.size:
        _lib().oracle_tma_box_images_nd(_ptr(T), rank, _ptr(d), _ptr(st), es, _ptr(ex), _ptr(sr),
                                        mode, 1 if oob_nan else 0, b0, b1, _ptr(out))
    return out


def tma_box_images_region(T, dims, strides, es, ext, estr, origin, nboxes, mode, oob_nan=False,
                          boxes=None):
    """As tma_box_images_nd for the box grid that starts at index origin[i] (may be
    negative) with nboxes[i] boxes along dimension i; indices outside [0, dims[i]) read
    the fill value."""
    rank = len(dims)
    T = np.ascontiguousarray(T).view(np.uint8).reshape(-1)
    arr = lambda v, pad=1: np.ascontiguousarray(np.array(list(v) + [pad] * (5 - len(v)),
                                                         dtype=np.int64))
    total = int(np.prod(nboxes))
    b0, b1 = (0, total) if boxes is None else boxes
    L = [(e + s - 1) // s for e, s in zip(ext, estr)]
    box_bytes = int(np.prod(L)) * es
    out = np.empty((b1 - b0) * box_bytes, dtype=np.uint8)
    d, st, ex, sr = arr(dims), arr([es] + list(strides)), arr(ext), arr(estr)
    og, nb = arr(origin, 0), arr(nboxes)
    if out.size:
        _lib().oracle_tma_box_images_region(_ptr(T), rank, _ptr(d), _ptr(st), es, _ptr(ex),
                                            _ptr(sr), _ptr(og), _ptr(nb), mode,
                                            1 if oob_nan else 0, b0, b1, _ptr(out))
    return out


__all__ = ["gemm", "gemm_entries", "swizzle", "box_grid", "tma_box_images", "threads",
           "f16_value", "f8_value", "tf32_value", "box_grid_nd", "tma_box_images_nd",
           "tma_box_images_region"]
