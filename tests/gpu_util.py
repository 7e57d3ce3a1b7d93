"""Helpers shared by the GPU parity tests (device upload, tolerance check)."""
import numpy as np

from tma_pipelined_tensor_gb300 import inputs as gen


def to_device_bf16(bits):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def to_device(arr):
    import torch
    return torch.from_numpy(np.ascontiguousarray(arr)).cuda()


def c_to_f64(C):
    """Device C (fp32, bf16 or fp16 torch tensor) -> host float64 array."""
    import torch
    if C.dtype == torch.bfloat16:
        bits = C.view(torch.int16).cpu().numpy().view(np.uint16)
        return gen.bf16_bits_to_f32(bits).astype(np.float64)
    return C.cpu().numpy().astype(np.float64)


def to_device_f16(bits):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.float16).cuda()


def gemm_bound(C_ref, absprod, K, alpha, beta, c0_vals, out_bf16, out_f16=False):
    """|C - C_ref| <= 2*K*2^-24*|alpha|*(|A||B|) + 2^-8*|C_ref| (bf16 out) or 2^-10*|C_ref|
    (fp16 out: twice its unit roundoff, as 2^-8 is for bf16) + 2^-23*|beta*C0| (the fp32
    add of the beta term)."""
    bound = 2.0 * K * 2.0 ** -24 * abs(alpha) * absprod
    if out_bf16:
        bound = bound + 2.0 ** -8 * np.abs(C_ref)
    if out_f16:
        bound = bound + 2.0 ** -10 * np.abs(C_ref)
    if beta != 0.0:
        bound = bound + 2.0 ** -23 * np.abs(beta * c0_vals)
    return bound


def assert_within(got, C_ref, bound, what=""):
    err = np.abs(got - C_ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d of %d outside the bound; first %s: got %s want %s bound %s" % (
            what, int(bad.sum()), bad.size, idx.tolist(),
            [got[tuple(i)] for i in idx], [C_ref[tuple(i)] for i in idx],
            [bound[tuple(i)] for i in idx]))


def c0_values(C0, f16=False):
    if C0 is None:
        return None
    if C0.dtype == np.uint16:
        if f16:
            return C0.view(np.float16).astype(np.float64)
        return gen.bf16_bits_to_f32(C0).astype(np.float64)
    return C0.astype(np.float64)


def stratified_positions(M, N, tile_n, per_cell=2, seed=0):
    """`per_cell` random outputs in every (128-row tile, 32-row epilogue quarter, 64-column
    chunk) cell of the launch's tiling: each tile of `tile_n` columns is cut into 64-column
    chunks from its own first column (the last chunk of a 224-wide tile is 32 wide), and
    every 32-row group of rows is one epilogue warp's quarter of a 128-row tile.  Half-width
    tiles of the split tail are 128-column halves of 256-wide tiles, so their chunks are
    cells of the same grid."""
    rng = np.random.default_rng(seed)
    r0 = np.arange(0, M, 32)
    c0 = np.array([c for t in range(0, N, tile_n) for c in range(t, min(t + tile_n, N), 64)])
    cw = np.array([min(64, (c // tile_n) * tile_n + tile_n - c, N - c) for c in c0])
    rh = np.minimum(32, M - r0)
    ii, jj = [], []
    for _ in range(per_cell):
        ri = r0[:, None] + (rng.random((len(r0), len(c0))) * rh[:, None]).astype(np.int64)
        cj = c0[None, :] + (rng.random((len(r0), len(c0))) * cw[None, :]).astype(np.int64)
        ii.append(ri.ravel())
        jj.append(cj.ravel())
    return np.concatenate(ii), np.concatenate(jj)
