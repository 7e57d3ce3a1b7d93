// Structures shared by the host side of the library and its kernels (not part of the
// public C ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>

#include "tg.h"

namespace tg {

// Bounded-wait control handed to every kernel.
// status[0] latches the first error word (0 = healthy) until the host reads it;
// status[1] holds the sequence number of the launch that is aborting, so that only
// the blocks of that launch stop early.
struct WaitCtl {
    uint32_t *status;    // this device's status words
    uint64_t timeout_ns; // limit of one pipeline wait
    uint32_t seq;        // non-zero sequence number of this launch
};

// ---------------------------------------------------------------------------------
// GEMM: persistent, warp-specialised, 128 x BN output tiles, 64-deep k-blocks.
// ---------------------------------------------------------------------------------
constexpr uint32_t kTileM = 128;
constexpr uint32_t kTileK = 64;            // one 128-byte swizzle row of bf16
constexpr uint32_t kTileKBytes = 128;      // k-block depth in bytes: 64 16-bit or 128 8-bit elements
constexpr uint32_t kEpiWarps = 4;          // TMEM lane quarters
constexpr uint32_t kEpiBufBytes = 4096;    // 32 rows x 128 bytes
constexpr uint32_t kMaxEpiBufs = 4;        // staging buffers per epilogue warp (2 or 4)
constexpr uint32_t kMnBox = 64;            // MN-major operand box: 64 MN elements x 64 k-rows
constexpr uint32_t kMnBoxBytes = kMnBox * kTileK * 2;
constexpr uint32_t kGemmThreads = 192;     // 4 epilogue warps, producer, MMA issuer
constexpr uint32_t kMinGemmSmem = 120 * 1024;  // keeps one CTA per SM (TMEM budget)
constexpr uint32_t kClcSlots = 4;          // dynamic scheduling: responses in flight or unread
constexpr uint32_t kClcBytes = kClcSlots * 16 + 2 * kClcSlots * 8;  // responses, full, empty

struct GemmParams {
    int32_t M, N, K;
    int32_t n_store;    // columns the C descriptor covers: N rounded down to 16-byte rows
    uint32_t tiles_m, tiles_n, k_blocks;
    uint32_t units_m;   // rows of scheduling units: tiles_m / cluster, rounded up
    uint32_t num_units; // units_m * tiles_n
    uint32_t group_m;   // rasterisation group height, in units
    uint32_t stages;
    uint32_t cluster;   // CTAs per cluster: 1, 2, or 4 (two CTA pairs sharing B)
    uint32_t out_kind;  // C element type: 0 = fp32, 1 = bf16, 2 = fp16
    uint32_t in_kind;   // A and B element type: 0 = bf16, 1 = fp16, 2 = E4M3, 3 = E5M2, 4 = tf32,
                        // 5 / 6 = E4M3 / E5M2 with MX block scales
    uint32_t kblk;      // elements per k-block: 64 (16-bit), 128 (8-bit) or 32 (tf32)
    uint32_t epi_bufs;  // staging buffers per epilogue warp: 2 or 4
    uint32_t a_mn;      // A stored M-major (K rows of M elements)
    uint32_t b_mn;      // B stored N-major (K rows of N elements)
    uint32_t flags;
    uint32_t clc;       // 1: dynamic scheduling by cluster launch control (one cluster per unit)
    float alpha, beta;
    const void *C;      // C0 for beta != 0 (read with plain loads)
    int64_t ldc;
    WaitCtl ctl;
    // Schedule: units [0, dp_units) are computed whole, strided over the clusters; the
    // k-blocks of units [dp_units, num_units) form sk_iters stream-K iterations split
    // evenly over the clusters.  A unit split between clusters is finished by the cluster
    // holding its first k-block, after adding the fp32 partials of the others.
    uint32_t dp_units;
    // Data-parallel work items: units [0, split_from) whole, then units
    // [split_from, dp_units) as two half-width tiles each (CTA pairs with 256-wide tiles
    // only); dp_work = split_from + 2 (dp_units - split_from).
    uint32_t split_from;
    uint32_t dp_work;
    uint64_t sk_iters;
    float *ws;          // partials: [cluster slot][rank][128 rows][tile_n] fp32
    uint32_t *sk_flags; // [cluster slot][rank] = launch sequence number once written
    // MX operands: E8M0 block scales of A and B in 512-byte atoms (128 rows x 4 blocks of
    // 32 elements); the atom of row group g and k-block kb is at (kb * sf_rb + g) * 512
    const uint8_t *sfa, *sfb;
    uint32_t sf_rb_a, sf_rb_b;  // 128-row groups of A (M) and of B (N)
};

// Bytes one ring stage of one CTA receives: its 128 rows of A plus its B rows (all
// tile_n of them, or half of them when a CTA pair shares the B tile); with MX operands
// also one 512-byte scale atom for A and one per 128 columns of B.
constexpr uint32_t kSfAtomBytes = 512;
inline uint32_t gemm_stage_bytes(uint32_t tile_n, bool pair, bool mx = false) {
    return (kTileM + (pair ? tile_n / 2 : tile_n)) * kTileKBytes +
           (mx ? kSfAtomBytes * (1 + tile_n / kTileM) : 0u);
}

// Operand element type of a layout word (bits 4-6), its size and its k-block depth in
// elements, and the tcgen05 MMA kind that multiplies it (0 = kind::f16, 1 = kind::f8f6f4,
// 2 = kind::tf32).
inline uint32_t gemm_in_kind(uint32_t layout) { return (layout >> 4) & 7u; }
inline bool gemm_in_mx(uint32_t in_kind) { return in_kind == 5u || in_kind == 6u; }
inline uint32_t gemm_in_bytes(uint32_t layout) {
    const uint32_t k = gemm_in_kind(layout);
    return k == 4u ? 4u : k >= 2u ? 1u : 2u;
}
inline uint32_t gemm_kblk(uint32_t layout) { return kTileKBytes / gemm_in_bytes(layout); }
// 0 = kind::f16, 1 = kind::f8f6f4, 2 = kind::tf32, 3 = kind::mxf8f6f4 with block scales
inline uint32_t gemm_mma_kind(uint32_t in_kind) {
    return in_kind == 4u ? 2u : gemm_in_mx(in_kind) ? 3u : in_kind >= 2u ? 1u : 0u;
}
constexpr uint32_t kMmaF16 = 0, kMmaF8 = 1, kMmaTf32 = 2, kMmaMx = 3;

inline uint32_t gemm_smem_bytes(uint32_t tile_n, uint32_t stages, bool pair, uint32_t epi_bufs,
                                bool mx = false) {
    uint32_t bytes = 1024                                                // alignment slack
                     + (mx && pair ? 512u : 0u)  // scale atoms rounded up to 1024 bytes
                     + stages * gemm_stage_bytes(tile_n, pair, mx)       // operand ring
                     + kEpiWarps * epi_bufs * kEpiBufBytes               // epilogue staging
                     + kClcBytes                                         // dynamic-schedule ring
                     + (2 * stages + 6 + kMaxEpiBufs * kEpiWarps) * 8  // barriers
                     + 8 + 24;  // TMEM address slot, the producers' exit-exchange words
    return bytes < kMinGemmSmem ? kMinGemmSmem : bytes;
}

struct GemmLaunch {
    CUtensorMap map_a, map_b, map_c;
    CUtensorMap map_c2;  // C with 32-column boxes: the last chunk of a 224-wide tile
    // MX on CTA pairs: the scale arrays as rows of 512-byte atoms (128 x 32-bit), boxes of
    // one atom (A) and of tile_n / 128 consecutive atoms (B)
    CUtensorMap map_sfa, map_sfb;
    GemmParams p;
    uint32_t tile_n;
    uint32_t pair;  // 1: CTA-pair kernel (tcgen05 cta_group::2), 0: one CTA per MMA
    uint32_t grid;
    uint32_t smem;
};

// Per-device caches of what every launch would otherwise ask the runtime again (each
// query costs microseconds of host time, as much as a small GEMM takes on the GPU):
// kernel_smem_attr raises a kernel's dynamic shared-memory limit only when a launch needs
// more than was set on this device before; kernel_max_clusters / kernel_max_blocks
// remember the occupancy answer for a (kernel, shared memory, cluster) triple.
cudaError_t kernel_smem_attr(const void *kern, uint32_t smem);
cudaError_t kernel_max_clusters(const void *kern, uint32_t smem, uint32_t threads, uint32_t cluster,
                                int *clusters);
cudaError_t kernel_max_blocks(const void *kern, uint32_t smem, uint32_t threads, int *blocks);

tg_status launch_gemm(const GemmLaunch &L, cudaStream_t stream);
tg_status launch_gemm_pair(const GemmLaunch &L, cudaStream_t stream);
tg_status gemm_max_active_clusters(uint32_t tile_n, uint32_t smem, uint32_t cluster,
                                   int *clusters);
tg_status gemm_pair_max_active_clusters(uint32_t tile_n, uint32_t smem, uint32_t cluster,
                                        int *clusters, bool mx = false);

// ---------------------------------------------------------------------------------
// TMA tile copy
// ---------------------------------------------------------------------------------
struct CopyParams {
    uint32_t rank;        // 1..5
    uint32_t nb[5];       // boxes along each dimension (dimension 0 innermost)
    uint32_t ext[5];      // box traversal extent per dimension (box origin step)
    int32_t origin[5];    // index of box 0 along each dimension (may be negative)
    uint32_t nboxes;      // total boxes
    uint32_t box_bytes;   // bytes of one box image
    uint32_t stage_pitch; // box_bytes rounded up to 1024
    uint32_t stages;
    uint32_t reverse;     // process boxes with the outermost box index fastest
    uint32_t back;        // 1: image -> tensor (bulk load of each box, tensor store)
    uint8_t *out;
    WaitCtl ctl;
};

inline uint32_t copy_smem_bytes(uint32_t stage_pitch, uint32_t stages) {
    return 1024 + stages * stage_pitch + stages * 8;
}

struct CopyLaunch {
    CUtensorMap map;
    CopyParams p;
    uint32_t grid;
    uint32_t smem;
};

// Back-to-back pair MMAs of the given kind (kMma*) on `pairs` CTA pairs, `iters` times
// four MMAs each, on zeroed shared-memory operands.
tg_status launch_mma_probe(uint32_t mma_kind, uint32_t pairs, uint64_t iters, const WaitCtl &ctl,
                           unsigned long long *timing, cudaStream_t stream);
tg_status launch_tile_copy(const CopyLaunch &L, cudaStream_t stream);
tg_status tile_copy_blocks_per_sm(uint32_t smem, int *blocks);

}  // namespace tg
