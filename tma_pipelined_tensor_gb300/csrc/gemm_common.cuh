// Device pieces shared by the GEMM kernels: the persistent tile order and the epilogue
// (TMEM -> alpha/beta -> swizzled staging -> TMA store).
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

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t &a, uint32_t &b, uint32_t &c,
                                             uint32_t &d) {
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "r"(addr)
                 : "memory");
}

// Per-warp epilogue state: which staging buffer comes next and the phase of each
// buffer's C0-load barrier.
struct EpiState {
    uint32_t chunk = 0;     // staging buffers used so far (buffer = chunk & 1)
    uint32_t c0_phase = 0;  // bit b: parity of the next wait on buffer b's C0 barrier
};

// Epilogue of one 128-byte-wide chunk of a warp's 32 rows (row = lane).  COLS fp32
// accumulator columns -> alpha*acc (+ beta*C0) -> bf16 or fp32 -> staging buffer (16-byte
// units XOR-swizzled by row & 7, matching the C descriptor's 128-byte swizzle, so the
// 8-lane phases of each 16-byte store hit distinct banks) -> TMA store.
//  * With beta != 0 the C0 chunk is brought into the same staging buffer by a TMA load
//    (its own mbarrier), read back row by row, and overwritten with the result.
//  * A TMA store writes whole 16-byte units at the right edge of a row, so the C
//    descriptor ends at n_store (N rounded down to 16-byte rows); the last columns
//    [n_store, N) are read and written here with plain loads and stores.
// Returns whether the staging buffer was used (a TMA store was issued).
template <bool kBf16>
__device__ __forceinline__ bool epilogue_chunk(const GemmParams &p, const CUtensorMap *map_c,
                                               uint32_t taddr, bool have_acc, int32_t row0,
                                               int32_t col0, uint32_t stg, uint32_t c0_bars,
                                               EpiState &es, uint32_t lane) {
    constexpr uint32_t COLS = kBf16 ? 64 : 32;
    const bool tma_part = col0 < p.n_store;
    const bool need_c0 = p.beta != 0.0f;
    const uint32_t bsel = es.chunk & 1u;
    const uint32_t buf = stg + bsel * kEpiBufBytes;
    const uint32_t c0_bar = c0_bars + 8u * bsel;
    if (tma_part) {
        // The buffer was last used two chunks ago; let that store finish reading it.
        if (lane == 0) {
            bulk_wait_read<1>();
            if (need_c0) {
                mbar_arrive_expect_tx(c0_bar, kEpiBufBytes);
                tma_load_2d(buf, map_c, c0_bar, col0, row0);
            }
        }
        __syncwarp();
    }
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

    const uint32_t row_addr = buf + lane * 128u;
    const int32_t row = row0 + int32_t(lane);
    if (need_c0) {
        if (tma_part) {
            // columns at or beyond n_store arrive as zeros (out-of-bounds fill)
            wait_bounded(c0_bar, (es.c0_phase >> bsel) & 1u, p.ctl, ROLE_EPILOGUE, false);
            es.c0_phase ^= 1u << bsel;
#pragma unroll
            for (uint32_t j = 0; j < 8; ++j) {
                uint32_t w0, w1, w2, w3;
                ld_shared_v4(row_addr + ((j ^ (lane & 7u)) << 4), w0, w1, w2, w3);
                const uint32_t w[4] = {w0, w1, w2, w3};
                if constexpr (kBf16) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        v[8 * j + 2 * e] = fmaf(p.beta, __uint_as_float(w[e] << 16), v[8 * j + 2 * e]);
                        v[8 * j + 2 * e + 1] =
                            fmaf(p.beta, __uint_as_float(w[e] & 0xffff0000u), v[8 * j + 2 * e + 1]);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        v[4 * j + e] = fmaf(p.beta, __uint_as_float(w[e]), v[4 * j + e]);
                }
            }
        }
        if (col0 + int32_t(COLS) > p.n_store && row < p.M) {
            const int32_t lo = max(col0, p.n_store), hi = min(col0 + int32_t(COLS), p.N);
            if constexpr (kBf16) {
                const __nv_bfloat16 *c0 =
                    reinterpret_cast<const __nv_bfloat16 *>(p.C) + int64_t(row) * p.ldc;
#pragma unroll
                for (int i = 0; i < int(COLS); ++i)
                    if (col0 + i >= lo && col0 + i < hi)
                        v[i] = fmaf(p.beta, __bfloat162float(c0[col0 + i]), v[i]);
            } else {
                const float *c0 = reinterpret_cast<const float *>(p.C) + int64_t(row) * p.ldc;
#pragma unroll
                for (int i = 0; i < int(COLS); ++i)
                    if (col0 + i >= lo && col0 + i < hi) v[i] = fmaf(p.beta, c0[col0 + i], v[i]);
            }
        }
    }
    if (col0 + int32_t(COLS) > p.n_store && row < p.M) {
        const int32_t lo = max(col0, p.n_store), hi = min(col0 + int32_t(COLS), p.N);
        if constexpr (kBf16) {
            __nv_bfloat16 *c =
                reinterpret_cast<__nv_bfloat16 *>(const_cast<void *>(p.C)) + int64_t(row) * p.ldc;
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
    if (!tma_part) return false;

    uint32_t w[32];
    if constexpr (kBf16) {
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i]);
    }
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
    es.chunk += 1;
    return true;
}

// Epilogue of one output tile for one warp: its 32 accumulator rows (TMEM lanes
// 32*warp .. 32*warp+31 of accumulator buffer `acc`), chunk by chunk.  Chunks that start
// at or beyond column N are skipped.
template <uint32_t BN>
__device__ __forceinline__ void epilogue_tile(const GemmParams &p, const CUtensorMap *map_c,
                                              uint32_t tmem_base, uint32_t acc, uint32_t m_blk,
                                              uint32_t n_blk, uint32_t warp, uint32_t lane,
                                              uint32_t stg, uint32_t c0_bars, EpiState &es) {
    const int32_t row0 = int32_t(m_blk * kTileM + warp * 32);
    if (row0 >= p.M) return;
    const bool have_acc = p.k_blocks != 0;
    const uint32_t taddr = tmem_base + ((warp * 32u) << 16) + acc * BN;
    if (p.out_bf16) {
        for (uint32_t c = 0; c < BN / 64 && int32_t(n_blk * BN + c * 64) < p.N; ++c)
            epilogue_chunk<true>(p, map_c, taddr + c * 64, have_acc, row0,
                                 int32_t(n_blk * BN + c * 64), stg, c0_bars, es, lane);
    } else {
        for (uint32_t c = 0; c < BN / 32 && int32_t(n_blk * BN + c * 32) < p.N; ++c)
            epilogue_chunk<false>(p, map_c, taddr + c * 32, have_acc, row0,
                                  int32_t(n_blk * BN + c * 32), stg, c0_bars, es, lane);
    }
}

}  // namespace tg
