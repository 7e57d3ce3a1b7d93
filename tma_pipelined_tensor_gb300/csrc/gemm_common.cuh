// Device pieces shared by the GEMM kernels: the persistent tile order and the epilogue
// of one 128-byte-wide chunk (TMEM -> alpha/beta -> swizzled staging -> TMA store).
#pragma once

#include <cuda_bf16.h>

#include "ptx.cuh"

namespace tg {

// Scheduling unit u -> output tile (m_blk, n_blk).  Units walk down groups of
// `group_m` unit rows, then across the N tiles, so that CTAs running at the same time
// share A and B tiles in L2 ("GEMM: la moltiplicazione di matrici sull'hardware",
// tiling section: blocks launched together reuse the same tiles through L2).  With
// clusters of two, a unit is a pair of vertically adjacent M tiles and `rank` picks one.
__device__ __forceinline__ void unit_coords(uint32_t u, const GemmParams &p, uint32_t rank,
                                            uint32_t &m_blk, uint32_t &n_blk) {
    const uint32_t gsz = p.group_m * p.tiles_n;
    const uint32_t g = u / gsz;
    const uint32_t first = g * p.group_m;
    const uint32_t gh = min(p.units_m - first, p.group_m);
    const uint32_t local = u - g * gsz;
    m_blk = (first + local % gh) * p.cluster + rank;
    n_blk = local / gh;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Epilogue of one 128-byte-wide chunk of a warp's 32 rows: COLS fp32 accumulator
// columns -> alpha*acc + beta*C0 -> staged (row = lane, 16-byte units XOR-swizzled by
// row & 7, matching the C descriptor's 128-byte swizzle) -> TMA store.
// A TMA store writes whole 16-byte units at the right edge of a row, so the C
// descriptor ends at n_store (N rounded down to 16-byte rows) and the last columns
// [n_store, N) are written here with plain stores.  Returns whether the staging
// buffer was used (a TMA store was issued).
template <bool kBf16>
__device__ __forceinline__ bool epilogue_chunk(const GemmParams &p, const CUtensorMap *map_c,
                                               uint32_t taddr, bool have_acc, int32_t row0,
                                               int32_t col0, uint32_t buf, uint32_t lane) {
    constexpr uint32_t COLS = kBf16 ? 64 : 32;
    float v[COLS];
    if (have_acc) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
        if constexpr (kBf16) {
            tmem_ld_32x32b_x32(taddr + 32, r);
            tmem_ld_wait(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[32 + i] = __uint_as_float(r[i]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < int(COLS); ++i) v[i] = 0.0f;
    }
#pragma unroll
    for (int i = 0; i < int(COLS); ++i) v[i] *= p.alpha;
    if (p.beta != 0.0f) {
        const int32_t row = row0 + int32_t(lane);
        if (row < p.M) {
            if constexpr (kBf16) {
                const __nv_bfloat16 *c0 =
                    reinterpret_cast<const __nv_bfloat16 *>(p.C) + int64_t(row) * p.ldc;
#pragma unroll
                for (int i = 0; i < int(COLS); ++i)
                    if (col0 + i < p.N) v[i] = fmaf(p.beta, __bfloat162float(c0[col0 + i]), v[i]);
            } else {
                const float *c0 = reinterpret_cast<const float *>(p.C) + int64_t(row) * p.ldc;
#pragma unroll
                for (int i = 0; i < int(COLS); ++i)
                    if (col0 + i < p.N) v[i] = fmaf(p.beta, c0[col0 + i], v[i]);
            }
        }
    }
    if (col0 + int32_t(COLS) > p.n_store) {
        const int32_t row = row0 + int32_t(lane);
        if (row < p.M) {
            const int32_t lo = max(col0, p.n_store), hi = min(col0 + int32_t(COLS), p.N);
            if constexpr (kBf16) {
                __nv_bfloat16 *c = reinterpret_cast<__nv_bfloat16 *>(const_cast<void *>(p.C)) +
                                   int64_t(row) * p.ldc;
#pragma unroll
                for (int i = 0; i < int(COLS); ++i)
                    if (col0 + i >= lo && col0 + i < hi) c[col0 + i] = __float2bfloat16_rn(v[i]);
            } else {
                float *c = reinterpret_cast<float *>(const_cast<void *>(p.C)) + int64_t(row) * p.ldc;
#pragma unroll
                for (int i = 0; i < int(COLS); ++i)
                    if (col0 + i >= lo && col0 + i < hi) c[col0 + i] = v[i];
            }
        }
        if (col0 >= p.n_store) return false;
    }
    uint32_t w[32];
    if constexpr (kBf16) {
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i]);
    }
    // The buffer was last used two chunks ago; let that store finish reading it.
    if (lane == 0) bulk_wait_read<1>();
    __syncwarp();
    const uint32_t row_addr = buf + lane * 128u;
#pragma unroll
    for (uint32_t j = 0; j < 8; ++j)
        st_shared_v4(row_addr + ((j ^ (lane & 7u)) << 4), w[4 * j], w[4 * j + 1], w[4 * j + 2],
                     w[4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(map_c, buf, col0, row0);
        bulk_commit();
    }
    return true;
}


}  // namespace tg
