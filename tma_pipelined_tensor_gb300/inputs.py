"""Seeded synthetic inputs shared by the CUDA path's tests/benchmark and the oracle.

This module holds no GEMM or TMA arithmetic: it only draws numbers.  Everything is
numpy on the host so that the same seed yields the same bytes on any machine:

* a counter-based splitmix64 stream per (seed, stream id) pair;
* uniforms in [lo, hi) from the top 53 bits of each draw;
* normals by the Box-Muller transform on pairs of uniforms;
* rounding to bf16 is round-to-nearest-even from binary32 (the value is first
  rounded double -> binary32 by numpy, then binary32 -> bf16 here).

Workload recipes (sizes, distributions, seeds) follow the benchmark configurations:
square GEMMs, the FFN/projection shapes of a BERT-large-like training step, the ragged
edge case and the 4100 x 8200 TMA tile-copy tensor.
"""
import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

STREAM_A, STREAM_B, STREAM_C = 0, 1, 2
STREAM_SFA, STREAM_SFB = 3, 4


def splitmix64(seed: int, start: int, n: int) -> np.ndarray:
    """Draws start..start+n-1 of the splitmix64 sequence seeded with `seed`."""
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _stream_seed(seed: int, stream: int) -> int:
    return int(splitmix64(seed * 8 + stream, 0, 1)[0])


def uniform(seed: int, stream: int, n: int, lo=-1.0, hi=1.0) -> np.ndarray:
    s = _stream_seed(seed, stream)
    out = np.empty(n, dtype=np.float64)
    for p in range(0, n, _CHUNK):
        q = min(n, p + _CHUNK)
        u = (splitmix64(s, p, q - p) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        out[p:q] = lo + (hi - lo) * u
    return out


def normal(seed: int, stream: int, n: int, mean=0.0, std=1.0) -> np.ndarray:
    s = _stream_seed(seed, stream)
    out = np.empty(n, dtype=np.float64)
    for p in range(0, n, _CHUNK):
        q = min(n, p + _CHUNK)
        m = (q - p + 1) // 2
        z = splitmix64(s, 2 * (p // 2), 2 * m)
        u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        r = np.sqrt(-2.0 * np.log(u1))
        pair = np.empty(2 * m, dtype=np.float64)
        pair[0::2] = r * np.cos(2.0 * np.pi * u2)
        pair[1::2] = r * np.sin(2.0 * np.pi * u2)
        out[p:q] = mean + std * pair[: q - p]
    return out


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round-to-nearest-even binary32 -> bf16; returns the 16-bit patterns."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    w = f.view(np.uint32).astype(np.uint64)
    lsb = (w >> np.uint64(16)) & np.uint64(1)
    r = ((w + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        r[nan] = 0x7FC0
    return r


def f32_to_f16_bits(x) -> np.ndarray:
    """Round-to-nearest-even binary32 -> IEEE binary16 (numpy's conversion); the bits."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def f16_matrix(rows: int, cols: int, seed: int, stream: int, dist: str, ld: int = None,
               a=None, b=None) -> np.ndarray:
    """As bf16_matrix, with fp16 patterns (padding columns hold an fp16 NaN)."""
    ld = cols if ld is None else ld
    n = rows * cols
    if dist == "uniform":
        v = uniform(seed, stream, n, -1.0 if a is None else a, 1.0 if b is None else b)
    else:
        v = normal(seed, stream, n, 0.0 if a is None else a, 1.0 if b is None else b)
    bits = f32_to_f16_bits(v.astype(np.float32)).reshape(rows, cols)
    if ld == cols:
        return bits
    out = np.full((rows, ld), 0x7E00, dtype=np.uint16)
    out[:, :cols] = bits
    return out


def f32_to_f8_bits(x, e5m2: bool = False) -> np.ndarray:
    """Binary32 -> E4M3 / E5M2 patterns (torch's round-to-nearest-even conversion)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    dt = torch.float8_e5m2 if e5m2 else torch.float8_e4m3fn
    return t.to(dt).view(torch.uint8).numpy().copy()


def f8_matrix(rows: int, cols: int, seed: int, stream: int, dist: str, ld: int = None,
              e5m2: bool = False, a=None, b=None) -> np.ndarray:
    """rows x ld uint8 array of E4M3 (or E5M2) patterns; padding columns hold a NaN."""
    ld = cols if ld is None else ld
    n = rows * cols
    if dist == "uniform":
        v = uniform(seed, stream, n, -1.0 if a is None else a, 1.0 if b is None else b)
    else:
        v = normal(seed, stream, n, 0.0 if a is None else a, 1.0 if b is None else b)
    bits = f32_to_f8_bits(v.astype(np.float32), e5m2).reshape(rows, cols)
    if ld == cols:
        return bits
    out = np.full((rows, ld), 0x7F, dtype=np.uint8)
    out[:, :cols] = bits
    return out


def mx_scale_bytes(rows: int, K: int) -> int:
    """Bytes of the E8M0 block scales of an MX operand with `rows` rows and K columns:
    512-byte atoms, one per (128 rows, 128 elements of K), both counts rounded up."""
    return ((rows + 127) // 128) * ((K + 127) // 128) * 512


def mx_pack_scales(logical: np.ndarray, K: int) -> np.ndarray:
    """Stores a rows x ceil(K/32) array of E8M0 scale bytes in the library's atom layout:
    byte of row r, 32-element block j at ((j // 4) * RB + r // 128) * 512 + (r % 32) * 16
    + ((r % 128) // 32) * 4 + j % 4, RB = ceil(rows / 128).  Bytes no scale occupies
    (rows and blocks past the operand's end) hold 127, the scale 1."""
    rows, nblk = logical.shape
    rb = (rows + 127) // 128
    out = np.full(mx_scale_bytes(rows, K), 127, dtype=np.uint8)
    r = np.arange(rows)[:, None]
    j = np.arange(nblk)[None, :]
    off = ((j // 4) * rb + r // 128) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + j % 4
    out[off.ravel()] = logical.astype(np.uint8).ravel()
    return out


def mx_scales(rows: int, K: int, seed: int, stream: int, lo: int = 120, hi: int = 134):
    """Seeded E8M0 block scales: a rows x ceil(K/32) array of integers drawn uniformly
    from [lo, hi] (scales 2^(lo-127) .. 2^(hi-127)) and the same bytes packed in the atom
    layout.  Returns (logical, packed)."""
    nblk = (K + 31) // 32
    u = uniform(seed, stream, rows * nblk, 0.0, 1.0)
    logical = (lo + np.floor(u * (hi - lo + 1))).clip(lo, hi).astype(np.uint8).reshape(rows, nblk)
    return logical, mx_pack_scales(logical, K)


def f32_matrix(rows: int, cols: int, seed: int, stream: int, dist: str, ld: int = None,
               a=None, b=None) -> np.ndarray:
    """rows x ld float32 array (the draws rounded to binary32); padding columns hold NaN."""
    ld = cols if ld is None else ld
    n = rows * cols
    if dist == "uniform":
        v = uniform(seed, stream, n, -1.0 if a is None else a, 1.0 if b is None else b)
    else:
        v = normal(seed, stream, n, 0.0 if a is None else a, 1.0 if b is None else b)
    out = np.full((rows, ld), np.nan, dtype=np.float32)
    out[:, :cols] = v.astype(np.float32).reshape(rows, cols)
    return out


def bf16_bits_to_f32(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_matrix(rows: int, cols: int, seed: int, stream: int, dist: str,
                ld: int = None, a=None, b=None) -> np.ndarray:
    """rows x ld uint16 array of bf16 bits; columns >= cols are padding (bf16 NaN).

    dist "uniform": U[a, b) (default [-1, 1)); "normal": N(a, b) (default (0, 1)).
    """
    ld = cols if ld is None else ld
    n = rows * cols
    if dist == "uniform":
        v = uniform(seed, stream, n, -1.0 if a is None else a, 1.0 if b is None else b)
    elif dist == "normal":
        v = normal(seed, stream, n, 0.0 if a is None else a, 1.0 if b is None else b)
    else:
        raise ValueError(dist)
    bits = f32_to_bf16_bits(v.astype(np.float32)).reshape(rows, cols)
    if ld == cols:
        return bits
    out = np.full((rows, ld), 0x7FC0, dtype=np.uint16)
    out[:, :cols] = bits
    return out


def small_int_matrix(rows: int, cols: int, seed: int, stream: int, lo=-2, hi=2,
                     ld: int = None) -> np.ndarray:
    """bf16 bits of integers uniform in [lo, hi] (exact-integer GEMM regime)."""
    ld = cols if ld is None else ld
    u = uniform(seed, stream, rows * cols, 0.0, 1.0)
    v = np.floor(lo + (hi - lo + 1) * u).clip(lo, hi)
    bits = f32_to_bf16_bits(v.astype(np.float32)).reshape(rows, cols)
    if ld == cols:
        return bits
    out = np.full((rows, ld), 0x7FC0, dtype=np.uint16)
    out[:, :cols] = bits
    return out


def copy_tensor(H: int = 4100, W: int = 8200) -> np.ndarray:
    """The tile-copy tensor: bf16 of (row*W + col) mod 65521, H x W, as uint16 bits."""
    r = np.arange(H, dtype=np.int64)[:, None]
    c = np.arange(W, dtype=np.int64)[None, :]
    v = ((r * W + c) % 65521).astype(np.float32)
    return f32_to_bf16_bits(v)


def unique_bits_tensor(H: int, W: int, seed: int = 7) -> np.ndarray:
    """H x W uint16 patterns from the splitmix stream (raw bits, for byte-exact copies)."""
    z = splitmix64(_stream_seed(seed, 3), 0, H * W)
    return (z >> np.uint64(48)).astype(np.uint16).reshape(H, W)


# --------------------------------------------------------------------------------
# Named workloads (sizes, distributions and seeds of the benchmark configurations).
# --------------------------------------------------------------------------------
GEMM_WORKLOADS = {
    # name: (M, N, K, distA, argsA, distB, argsB, seed, out_dtype, alpha, beta)
    "gemm_256": (256, 256, 256, "uniform", (-1.0, 1.0), "uniform", (-1.0, 1.0), 0,
                 "f32", 1.0, 0.0),
    "gemm_4096": (4096, 4096, 4096, "normal", (0.0, 1.0), "normal", (0.0, 1.0), 1,
                  "bf16", 1.0, 0.0),
    "ffn_up": (16384, 4096, 1024, "normal", (0.0, 1.0), "normal", (0.0, 0.02), 2,
               "bf16", 1.0, 0.0),
    "ffn_down": (16384, 1024, 4096, "normal", (0.0, 1.0), "normal", (0.0, 0.02), 2,
                 "bf16", 1.0, 0.0),
    "dw": (1024, 4096, 16384, "normal", (0.0, 1.0), "normal", (0.0, 1.0), 2,
           "bf16", 1.0, 0.0),
    "ragged": (3000, 5000, 2056, "normal", (0.0, 1.0), "normal", (0.0, 0.02), 2,
               "bf16", 1.0, 0.5),
    "gemm_8192": (8192, 8192, 8192, "uniform", (-1.0, 1.0), "uniform", (-1.0, 1.0), 3,
                  "bf16", 1.0, 0.0),
    "gemm_8192_e4m3": (8192, 8192, 8192, "uniform", (-1.0, 1.0), "uniform", (-1.0, 1.0), 3,
                       "bf16", 1.0, 0.0),
    "gemm_8192_tf32": (8192, 8192, 8192, "uniform", (-1.0, 1.0), "uniform", (-1.0, 1.0), 3,
                       "bf16", 1.0, 0.0),
    "gemm_8192_mxe4m3": (8192, 8192, 8192, "uniform", (-1.0, 1.0), "uniform", (-1.0, 1.0), 3,
                         "bf16", 1.0, 0.0),
}

# Operand element type of each workload (bf16 unless listed).
WORKLOAD_IN_TYPE = {"gemm_8192_e4m3": "e4m3", "gemm_8192_tf32": "tf32",
                    "gemm_8192_mxe4m3": "mxe4m3"}


def gemm_inputs(name: str, lda=None, ldb=None, ldc=None):
    """(A, B, C0) host arrays for a named GEMM workload (A, B: uint16 bf16 patterns, uint8
    E4M3 / E5M2 patterns or float32 tf32 operands for the workloads listed in
    WORKLOAD_IN_TYPE); C0 is None unless beta != 0."""
    M, N, K, da, pa, db, pb, seed, out, alpha, beta = GEMM_WORKLOADS[name]
    in_type = WORKLOAD_IN_TYPE.get(name, "bf16")
    if in_type == "bf16":
        A = bf16_matrix(M, K, seed, STREAM_A, da, lda, *pa)
        B = bf16_matrix(N, K, seed, STREAM_B, db, ldb, *pb)
    elif in_type == "tf32":
        A = f32_matrix(M, K, seed, STREAM_A, da, lda, *pa)
        B = f32_matrix(N, K, seed, STREAM_B, db, ldb, *pb)
    else:
        e5m2 = in_type in ("e5m2", "mxe5m2")
        A = f8_matrix(M, K, seed, STREAM_A, da, lda, e5m2, *pa)
        B = f8_matrix(N, K, seed, STREAM_B, db, ldb, e5m2, *pb)
    C0 = None
    if beta != 0.0:
        ldc = N if ldc is None else ldc
        if out == "bf16":
            C0 = bf16_matrix(M, N, seed, STREAM_C, "uniform", ldc, -1.0, 1.0)
        else:
            C0 = np.full((M, ldc), np.nan, dtype=np.float32)
            C0[:, :N] = uniform(seed, STREAM_C, M * N).astype(np.float32).reshape(M, N)
    return A, B, C0


def gemm_mx_scale_inputs(name: str):
    """Block scales of an MX workload (E8M0 integers drawn from [120, 134], the seed of the
    workload, streams of their own): (SA logical, SA packed, SB logical, SB packed)."""
    M, N, K = GEMM_WORKLOADS[name][:3]
    seed = GEMM_WORKLOADS[name][7]
    sa, sa_packed = mx_scales(M, K, seed, STREAM_SFA)
    sb, sb_packed = mx_scales(N, K, seed, STREAM_SFB)
    return sa, sa_packed, sb, sb_packed
