// Device pieces shared by the GEMM kernels: the persistent tile order and the epilogue
// (TMEM -> alpha/beta -> swizzled staging -> TMA store).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

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

// ---------------------------------------------------------------------------------
// Work segments of one cluster: whole units first (data-parallel part), then its share
// of the stream-K iterations.  Every role of a CTA walks the same sequence.
//
// Dynamic mode (p.clc): the grid holds one cluster per unit; a cluster computes its own
// unit, then units of clusters it cancels before they start (cluster launch control).
// The leader CTA's producer keeps one request in flight, one unit ahead; responses land
// in a ring of kClcSlots 16-byte slots in every CTA of the cluster, each with a `full`
// barrier per CTA (armed for 16 bytes by that CTA's producer) and an `empty` barrier in
// the leader that every consumer warp of the cluster arrives on once it has read the
// slot.  Every role reads every response, so all stop at the same failed response.
// ---------------------------------------------------------------------------------
struct Segment {
    uint32_t u;         // scheduling unit
    uint32_t kb0, kb1;  // k-blocks [kb0, kb1) of the unit
    uint32_t half;      // 0: the whole tile; 1 / 2: its left / right half-width tile
};

// Output columns [col0, col0 + width) of a segment of tile column n_blk.
template <uint32_t BN>
__device__ __forceinline__ void segment_cols(const Segment &g, uint32_t n_blk, int32_t &col0,
                                             uint32_t &width) {
    width = g.half ? BN / 2 : BN;
    col0 = int32_t(n_blk * BN + (g.half == 2 ? BN / 2 : 0));
}

struct ClcRing {
    uint32_t resp;       // shared address of slot 0's response (slot i at +16 i)
    uint32_t full;       // this CTA's full barriers (slot i at +8 i)
    uint32_t empty;      // the leader's empty barriers: shared::cluster address
    uint32_t empty_own;  // the same barriers at a shared::cta address (leader CTA only)
    uint32_t issue;      // non-zero in the lane that arrives and requests
    uint32_t role;       // ROLE_* for the waits
    bool requester;      // the leader CTA's producer
    bool rearm;          // this CTA's producer
};

struct SegIter {
    uint32_t dp_next;
    uint64_t it, it_end;
    uint32_t clc_state;   // 0: own unit next, 1: responses next, 2: done
    uint32_t clc_n;       // responses read
    uint32_t clc_issued;  // requests issued (requester only)
    ClcRing ring;
};

// The dynamic mode's ring: responses and barriers at `s_clc` (16-byte aligned).
__device__ __forceinline__ ClcRing clc_ring(uint32_t s_clc, uint32_t issue, uint32_t role,
                                            bool requester, bool rearm, uint32_t cluster) {
    ClcRing r;
    r.resp = s_clc;
    r.full = s_clc + 16 * kClcSlots;
    r.empty_own = r.full + 8 * kClcSlots;
    r.empty = cluster > 1 ? mapa_shared(r.empty_own, 0) : r.empty_own;
    r.issue = issue;
    r.role = role;
    r.requester = requester;
    r.rearm = rearm;
    return r;
}

// Consumer warps of a cluster that release each ring slot (the leader's empty count).
__device__ __forceinline__ uint32_t clc_consumers(const GemmParams &p, bool pair) {
    return p.cluster * (1u + kEpiWarps) + (pair ? 1u : p.cluster);
}

// Requester: ask for the next unit into the next slot once every consumer has read that
// slot's previous response.
__device__ __forceinline__ bool clc_request(SegIter &s, const GemmParams &p) {
    const uint32_t n = s.clc_issued, slot = n % kClcSlots;
    if (!wait_bounded(s.ring.empty_own + 8 * slot, ((n / kClcSlots) & 1u) ^ 1u, p.ctl, s.ring.role))
        return false;
    clc_try_cancel(s.ring.issue, s.ring.resp + 16 * slot, s.ring.full + 8 * slot, p.cluster > 1);
    s.clc_issued = n + 1;
    return true;
}

// Requester, after its loop: a response still on its way must land before the CTA exits.
__device__ __forceinline__ void clc_drain(SegIter &s, const GemmParams &p) {
    if (!p.clc || !s.ring.requester || s.clc_issued == s.clc_n) return;
    const uint32_t n = s.clc_n, slot = n % kClcSlots;
    wait_bounded(s.ring.full + 8 * slot, (n / kClcSlots) & 1u, p.ctl, s.ring.role, false);
}

// ---------------------------------------------------------------------------------
// Producers' exit protocol.  Every copy into a CTA's shared memory must have landed
// before that CTA leaves, on every exit path.  In a cluster of two, copies land in a CTA
// on behalf of the other one (the CTA-pair kernel's loads count their bytes on the
// leader's full barriers; the per-CTA kernel multicasts each half of B into both CTAs),
// and after an abort the two producers may have issued different numbers of k-blocks.
// So, once its loop has ended:
//  1. each producer publishes what the other CTA needs -- its issued k-block count, and
//     the requester its cluster-launch-control request count -- with a remote store and
//     a release-arrive on the other CTA's exchange barrier;
//  2. a CTA whose full barriers count the other CTA's bytes balances the k-blocks only
//     one side issued (drain_full_ring), so that each phase in flight completes exactly
//     when the copies really issued for it have landed;
//  3. it waits for those phases, and a CTA that receives multicast launch-control
//     responses waits for the ones still on their way (clc_drain_to).
// The peer of the CTA-pair kernel has no barrier of its own to wait on: its copies count
// on the leader's, and it passes the final cluster barrier only after the leader did.
// ---------------------------------------------------------------------------------

// Steps 2 and 3 on this CTA's full barriers.  `own` k-blocks were issued by this CTA and
// `other` by the other CTA, whose copies of a k-block bring `other_bytes` to this CTA's
// barrier of that k-block (other = own, other_bytes = 0 without a peer).  The counts differ
// by at most `S`: issuing k-block j waits for the MMA of k-block j - S, which waited for
// both sides' copies of it; for the same reason the phase of every k-block balanced here
// is the current phase of its barrier.
__device__ __forceinline__ void drain_full_ring(uint32_t b_full, uint32_t S, uint32_t own,
                                                uint32_t other, uint32_t other_bytes,
                                                const WaitCtl &ctl, uint32_t issue) {
    // issued only by the other side: this side's expect_tx arrival never came
    for (uint32_t j = own; j < other; ++j)
        mbar_arrive_expect_tx(issue, b_full + 8 * (j % S), other_bytes);
    // issued only by this side: the other side's bytes will never come
    for (uint32_t j = other; j < own; ++j) mbar_complete_tx(issue, b_full + 8 * (j % S), other_bytes);
    __syncwarp();
    const uint32_t n = max(own, other);
    for (uint32_t j = n > S ? n - S : 0; j < n; ++j)
        wait_bounded(b_full + 8 * (j % S), (j / S) & 1u, ctl, ROLE_PRODUCER, false);
}

// Steps 2 and 3 for a barrier that counts the copies of several producers (the leader of a
// CTA pair in a cluster of two pairs).  Producer p issued n[p] k-blocks and each of its
// k-blocks brings contrib[p] bytes to this barrier; this CTA (whose count is n[own]) arrived
// with expect_tx(expect) for each of its own k-blocks.  For every k-block some producers
// issued and others did not, the phase is made to complete exactly when the bytes really
// issued have landed: the missing bytes are completed where this CTA arrived, and an
// arrival expecting the issued bytes is made where it did not.  The counts differ by at
// most `S` (a k-block is issued only after every pair's MMA consumed k-block j - S, which
// needed every producer's copies of it), so each such phase is its barrier's current one.
template <uint32_t NP>
__device__ __forceinline__ void drain_full_ring_n(uint32_t b_full, uint32_t S, const uint32_t (&n)[NP],
                                                  const uint32_t (&contrib)[NP], uint32_t own,
                                                  uint32_t expect, const WaitCtl &ctl,
                                                  uint32_t issue) {
    uint32_t lo = n[0], hi = n[0];
#pragma unroll
    for (uint32_t q = 1; q < NP; ++q) {
        lo = min(lo, n[q]);
        hi = max(hi, n[q]);
    }
    for (uint32_t j = lo; j < hi; ++j) {
        uint32_t landed = 0;
#pragma unroll
        for (uint32_t q = 0; q < NP; ++q) landed += n[q] > j ? contrib[q] : 0u;
        const uint32_t bar = b_full + 8 * (j % S);
        if (n[own] > j) {
            if (landed < expect) mbar_complete_tx(issue, bar, expect - landed);
        } else if (landed > 0) {
            mbar_arrive_expect_tx(issue, bar, landed);
        }
    }
    __syncwarp();
    for (uint32_t j = hi > S ? hi - S : 0; j < hi; ++j)
        wait_bounded(b_full + 8 * (j % S), (j / S) & 1u, ctl, ROLE_PRODUCER, false);
}

// Step 3 for launch-control responses multicast into a CTA that does not request them:
// its producer armed the full barrier of every response up to `requested` (a request is
// made only once every consumer, this producer included, has released the slot's previous
// response), so each one not yet read is awaited there.
__device__ __forceinline__ void clc_drain_to(const SegIter &s, const GemmParams &p,
                                             uint32_t requested) {
    for (uint32_t n = s.clc_n; n < requested; ++n)
        wait_bounded(s.ring.full + 8 * (n % kClcSlots), (n / kClcSlots) & 1u, p.ctl, s.ring.role,
                     false);
}

__device__ __forceinline__ uint64_t sk_start(const GemmParams &p, uint32_t c, uint32_t ncl) {
    return p.sk_iters * c / ncl;
}

__device__ __forceinline__ void seg_begin(SegIter &s, const GemmParams &p, uint32_t cid,
                                          uint32_t ncl, const ClcRing &ring) {
    s.dp_next = cid;
    s.it = sk_start(p, cid, ncl);
    s.it_end = sk_start(p, cid + 1, ncl);
    s.clc_state = 0;
    s.clc_n = 0;
    s.clc_issued = 0;
    s.ring = ring;
    if (p.clc && ring.requester && !clc_request(s, p)) s.clc_state = 2;
}

__device__ __forceinline__ bool seg_next_dynamic(SegIter &s, const GemmParams &p, Segment &g) {
    g.kb0 = 0;
    g.kb1 = p.k_blocks;
    g.half = 0;
    if (s.clc_state == 0) {  // this cluster's own unit
        s.clc_state = 1;
        g.u = s.dp_next;
        return true;
    }
    if (s.clc_state == 2 || (s.ring.requester && s.clc_n == s.clc_issued)) return false;
    const uint32_t n = s.clc_n, slot = n % kClcSlots;
    if (!wait_bounded(s.ring.full + 8 * slot, (n / kClcSlots) & 1u, p.ctl, s.ring.role)) {
        s.clc_state = 2;
        return false;
    }
    uint32_t x;
    const bool got = clc_query(s.ring.resp + 16 * slot, x);
    s.clc_n = n + 1;
    if (s.ring.rearm) mbar_arrive_expect_tx(s.ring.issue, s.ring.full + 8 * slot, 16u);
    if (p.cluster > 1)
        mbar_arrive_remote(s.ring.issue, s.ring.empty + 8 * slot);
    else if (s.ring.issue)
        mbar_arrive(s.ring.empty_own + 8 * slot);
    if (!got) {
        s.clc_state = 2;
        return false;
    }
    // the requester asks for the following unit before working on this one; if that
    // gives up, this unit is still done and the next call ends the sequence
    if (s.ring.requester && !clc_request(s, p)) s.clc_state = 2;
    g.u = x / p.cluster;
    return true;
}

__device__ __forceinline__ bool seg_next(SegIter &s, const GemmParams &p, uint32_t ncl,
                                         Segment &g) {
    if (p.clc) return seg_next_dynamic(s, p, g);
    // Data-parallel work items: units [0, split_from) whole, then each unit in
    // [split_from, dp_units) as two half-width tiles (items split_from + 2j and +2j+1),
    // so that a last wave at most half full takes half the time.
    if (s.dp_next < p.dp_work) {
        const uint32_t w = s.dp_next;
        if (w < p.split_from) {
            g.u = w;
            g.half = 0;
        } else {
            g.u = p.split_from + (w - p.split_from) / 2;
            g.half = 1 + ((w - p.split_from) & 1u);
        }
        g.kb0 = 0;
        g.kb1 = p.k_blocks;
        s.dp_next += ncl;
        return true;
    }
    if (s.it < s.it_end) {
        const uint64_t uu = s.it / p.k_blocks;
        g.u = p.dp_units + uint32_t(uu);
        g.kb0 = uint32_t(s.it - uu * p.k_blocks);
        const uint64_t left = s.it_end - s.it;
        g.kb1 = uint32_t(min(uint64_t(p.k_blocks), uint64_t(g.kb0) + left));
        g.half = 0;
        s.it += g.kb1 - g.kb0;
        return true;
    }
    return false;
}

// Last cluster holding k-blocks of stream-K unit `u` (the unit's later k-blocks belong
// to the clusters after the one holding its first k-block, up to this one).
__device__ __forceinline__ uint32_t sk_last_contributor(const GemmParams &p, uint32_t u,
                                                        uint32_t ncl) {
    const uint64_t last_it = uint64_t(u - p.dp_units) * p.k_blocks + p.k_blocks - 1;
    return uint32_t(((last_it + 1) * ncl - 1) / p.sk_iters);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// fp16 in the low 16 bits of w -> float
__device__ __forceinline__ float half_lo_to_float(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
}

__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t &a, uint32_t &b, uint32_t &c,
                                             uint32_t &d) {
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "r"(addr)
                 : "memory");
}

// Shared-memory descriptors of stage 0's A and B tiles and their steps, in descriptor
// units (16 bytes): `stage` to the next ring stage, `a_k` / `b_k` per MMA (32 bytes of K:
// +32 B along a K-major row, +2 KiB = two 8-row groups for an MN-major tile).
struct MmaDescs {
    uint64_t a0, b0;
    uint32_t a_k, b_k, stage;
};

__device__ __forceinline__ MmaDescs mma_descs(const GemmParams &p, uint32_t sa0, uint32_t sb0,
                                             uint32_t stage_bytes) {
    MmaDescs m;
    m.a0 = p.a_mn ? umma_desc_mnmajor_sw128(sa0, kMnBoxBytes) : umma_desc_kmajor_sw128(sa0);
    m.b0 = p.b_mn ? umma_desc_mnmajor_sw128(sb0, kMnBoxBytes) : umma_desc_kmajor_sw128(sb0);
    m.a_k = (p.a_mn ? 2048u : 32u) >> 4;
    m.b_k = (p.b_mn ? 2048u : 32u) >> 4;
    m.stage = stage_bytes >> 4;
    return m;
}

// Per-warp epilogue state: which staging buffer comes next, the phase of each buffer's
// C0-load barrier, and how many chunks of the current tile had C0 loaded ahead.
struct EpiState {
    uint32_t chunk = 0;     // staging buffers used so far (buffer = chunk % epi_bufs)
    uint32_t c0_phase = 0;  // bit b: parity of the next wait on buffer b's C0 barrier
    uint32_t c0_ahead = 0;  // chunks of the current tile whose C0 load is already issued
};

// Waits until the staging buffer about to be reused is no longer read by a TMA store
// (all but the epi_bufs-1 most recent stores have read their source).
__device__ __forceinline__ void wait_staging_free(uint32_t epi_bufs) {
    if (epi_bufs == 4)
        bulk_wait_read<3>();
    else
        bulk_wait_read<1>();
}

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
// `add` / `add_n` / `add_stride`: stream-K partials of other clusters to add to the
// accumulator: this thread's row at this chunk's first 4-column group in the partial
// layout of epilogue_partial; add_stride = float4s between two clusters' partials.
// kCols = 32 with a 16-bit C is the last chunk of a tile width that is not a multiple
// of 64 (224): 64-byte staging rows, the 64-byte swizzle, its own C descriptor.
template <uint32_t kOut, uint32_t kCols = (kOut ? 64u : 32u)>
__device__ __forceinline__ bool epilogue_chunk(const GemmParams &p, const CUtensorMap *map_c,
                                               uint32_t taddr, bool have_acc, int32_t row0,
                                               int32_t col0, uint32_t stg, uint32_t c0_bars,
                                               EpiState &es, uint32_t lane, const float4 *add,
                                               uint32_t add_n, size_t add_stride, uint32_t idx) {
    constexpr uint32_t COLS = kCols;
    constexpr uint32_t ROW_BYTES = COLS * (kOut ? 2u : 4u);  // 128, or 64 for the last chunk
    constexpr uint32_t UNITS = ROW_BYTES / 16;                // 16-byte units per staging row
    // unit j of row r sits at j ^ (r & 7) with 128-byte rows, j ^ ((r >> 1) & 3) with 64-byte
    // rows: the swizzles of the C descriptors, which also keep the 16-byte stores of a
    // warp's 8-lane phases on distinct banks
    const uint32_t swz = ROW_BYTES == 128 ? (lane & 7u) : ((lane >> 1) & 3u);
    const bool tma_part = col0 < p.n_store;
    const bool need_c0 = p.beta != 0.0f;
    const uint32_t bsel = es.chunk & (p.epi_bufs - 1u);
    const uint32_t buf = stg + bsel * kEpiBufBytes;
    const uint32_t c0_bar = c0_bars + 8u * bsel;
    if (tma_part && idx >= es.c0_ahead) {
        // The buffer was last used epi_bufs chunks ago; let that store finish reading it.
        if (lane == 0) {
            wait_staging_free(p.epi_bufs);
            if (need_c0) {
                mbar_arrive_expect_tx(c0_bar, 32 * ROW_BYTES);
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
        if constexpr (COLS == 64) {
            tmem_ld_32x32b_x32(taddr + 32, r);
            tmem_ld_wait(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[32 + i] = __uint_as_float(r[i]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < int(COLS); ++i) v[i] = 0.0f;
    }
    for (uint32_t j = 0; j < add_n; ++j) {
        const float4 *src = add + j * add_stride;
#pragma unroll
        for (int q = 0; q < int(COLS) / 4; ++q) {
            const float4 f = __ldcg(src + size_t(q) * kTileM);
            v[4 * q] += f.x;
            v[4 * q + 1] += f.y;
            v[4 * q + 2] += f.z;
            v[4 * q + 3] += f.w;
        }
    }
#pragma unroll
    for (int i = 0; i < int(COLS); ++i) v[i] *= p.alpha;

    const uint32_t row_addr = buf + lane * ROW_BYTES;
    const int32_t row = row0 + int32_t(lane);
    if (need_c0) {
        if (tma_part) {
            // columns at or beyond n_store arrive as zeros (out-of-bounds fill)
            wait_bounded(c0_bar, (es.c0_phase >> bsel) & 1u, p.ctl, ROLE_EPILOGUE, false);
            es.c0_phase ^= 1u << bsel;
#pragma unroll
            for (uint32_t j = 0; j < UNITS; ++j) {
                uint32_t w0, w1, w2, w3;
                ld_shared_v4(row_addr + ((j ^ swz) << 4), w0, w1, w2, w3);
                const uint32_t w[4] = {w0, w1, w2, w3};
                if constexpr (kOut == 1) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        v[8 * j + 2 * e] = fmaf(p.beta, __uint_as_float(w[e] << 16), v[8 * j + 2 * e]);
                        v[8 * j + 2 * e + 1] =
                            fmaf(p.beta, __uint_as_float(w[e] & 0xffff0000u), v[8 * j + 2 * e + 1]);
                    }
                } else if constexpr (kOut == 2) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        v[8 * j + 2 * e] = fmaf(p.beta, half_lo_to_float(w[e]), v[8 * j + 2 * e]);
                        v[8 * j + 2 * e + 1] =
                            fmaf(p.beta, half_lo_to_float(w[e] >> 16), v[8 * j + 2 * e + 1]);
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
            if constexpr (kOut == 1) {
                const __nv_bfloat16 *c0 =
                    reinterpret_cast<const __nv_bfloat16 *>(p.C) + int64_t(row) * p.ldc;
#pragma unroll
                for (int i = 0; i < int(COLS); ++i)
                    if (col0 + i >= lo && col0 + i < hi)
                        v[i] = fmaf(p.beta, __bfloat162float(c0[col0 + i]), v[i]);
            } else if constexpr (kOut == 2) {
                const __half *c0 = reinterpret_cast<const __half *>(p.C) + int64_t(row) * p.ldc;
#pragma unroll
                for (int i = 0; i < int(COLS); ++i)
                    if (col0 + i >= lo && col0 + i < hi)
                        v[i] = fmaf(p.beta, __half2float(c0[col0 + i]), v[i]);
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
        if constexpr (kOut == 1) {
            __nv_bfloat16 *c =
                reinterpret_cast<__nv_bfloat16 *>(const_cast<void *>(p.C)) + int64_t(row) * p.ldc;
#pragma unroll
            for (int i = 0; i < int(COLS); ++i)
                if (col0 + i >= lo && col0 + i < hi) c[col0 + i] = __float2bfloat16_rn(v[i]);
        } else if constexpr (kOut == 2) {
            __half *c = reinterpret_cast<__half *>(const_cast<void *>(p.C)) + int64_t(row) * p.ldc;
#pragma unroll
            for (int i = 0; i < int(COLS); ++i)
                if (col0 + i >= lo && col0 + i < hi) c[col0 + i] = __float2half_rn(v[i]);
        } else {
            float *c = reinterpret_cast<float *>(const_cast<void *>(p.C)) + int64_t(row) * p.ldc;
#pragma unroll
            for (int i = 0; i < int(COLS); ++i)
                if (col0 + i >= lo && col0 + i < hi) c[col0 + i] = v[i];
        }
    }
    if (!tma_part) return false;

    constexpr uint32_t WORDS = ROW_BYTES / 4;
    uint32_t w[WORDS];
    if constexpr (kOut == 1) {
#pragma unroll
        for (int i = 0; i < int(WORDS); ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    } else if constexpr (kOut == 2) {
#pragma unroll
        for (int i = 0; i < int(WORDS); ++i) w[i] = pack_f16x2(v[2 * i], v[2 * i + 1]);
    } else {
#pragma unroll
        for (int i = 0; i < int(WORDS); ++i) w[i] = __float_as_uint(v[i]);
    }
#pragma unroll
    for (uint32_t j = 0; j < UNITS; ++j)
        st_shared_v4(row_addr + ((j ^ swz) << 4), w[4 * j], w[4 * j + 1], w[4 * j + 2],
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

// With beta != 0: issue the C0 loads of the first chunks of a tile (one per staging
// buffer) before the accumulator is ready, so that they arrive during the mainloop.
__device__ __forceinline__ void epilogue_prefetch_c0(const GemmParams &p, const CUtensorMap *map_c,
                                                     const CUtensorMap *map_c2, uint32_t m_blk,
                                                     int32_t col0, uint32_t width, uint32_t warp,
                                                     uint32_t lane, uint32_t stg, uint32_t c0_bars,
                                                     EpiState &es) {
    es.c0_ahead = 0;
    if (p.beta == 0.0f) return;
    const int32_t row0 = int32_t(m_blk * kTileM + warp * 32);
    if (row0 >= p.M) return;
    const uint32_t COLS = p.out_kind ? 64 : 32;
    // chunks of the tile; with a 16-bit C and a width of 224 the last one is 32 wide
    const uint32_t n_chunks = width / COLS + (width % COLS ? 1u : 0u);
    uint32_t n_tma = 0;  // chunks with a TMA part: a prefix of the tile's chunks
    while (n_tma < n_chunks && col0 + int32_t(n_tma * COLS) < p.n_store) ++n_tma;
    const uint32_t pre = min(n_tma, p.epi_bufs);
    if (lane == 0 && pre > 0) {
        bulk_wait_read<0>();  // every staging buffer is free
        for (uint32_t i = 0; i < pre; ++i) {
            const uint32_t b = (es.chunk + i) & (p.epi_bufs - 1u);
            const bool narrow = (i + 1) * COLS > width;
            mbar_arrive_expect_tx(c0_bars + 8u * b, narrow ? kEpiBufBytes / 2 : kEpiBufBytes);
            tma_load_2d(stg + b * kEpiBufBytes, narrow ? map_c2 : map_c, c0_bars + 8u * b,
                        col0 + int32_t(i * COLS), row0);
        }
    }
    __syncwarp();
    es.c0_ahead = pre;
}

// Stream-K partial of one segment: this warp's 32 accumulator rows, all BN columns, to
// the cluster's workspace slot.  Layout: float4 index (column / 4) * 128 + row, so that
// the 32 lanes of a warp (32 consecutive rows) store 512 contiguous bytes at a time.
template <uint32_t BN>
__device__ __forceinline__ void epilogue_partial(uint32_t tmem_base, uint32_t acc, uint32_t warp,
                                                 uint32_t lane, float4 *slot) {
    const uint32_t taddr = tmem_base + ((warp * 32u) << 16) + acc * BN;
    float4 *row = slot + (warp * 32 + lane);
    for (uint32_t c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(taddr + c * 32, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int q = 0; q < 8; ++q)
            __stcg(row + size_t(c * 8 + q) * kTileM,
                   make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                               __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3])));
    }
}

// Bounded wait (one lane) until a stream-K partial is published for this launch.
__device__ __forceinline__ bool wait_partial(const GemmParams &p, const uint32_t *flag) {
    if (ld_acquire_gpu(flag) == p.ctl.seq) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (ld_acquire_gpu(flag) == p.ctl.seq) return true;
        if ((n & 63u) == 0) {
            if (status_peek(p.ctl.status + 1) == p.ctl.seq) return false;
            if (globaltimer_ns() - t0 > p.ctl.timeout_ns) {
                const uint32_t word = uint32_t(TG_ERR_DEVICE_TIMEOUT) | (ROLE_EPILOGUE << 8) |
                                      ((blockIdx.x & 0xffffu) << 16);
                atomicCAS(p.ctl.status, 0u, word);
                atomicExch(p.ctl.status + 1, p.ctl.seq);
                return false;
            }
        }
    }
}

// Epilogue of one segment for one warp (its 32 accumulator rows: TMEM lanes
// 32*warp .. 32*warp+31 of accumulator buffer `acc`).
//  * whole unit: chunk by chunk to C (chunks starting at or beyond column N skipped);
//  * stream-K share that does not hold the unit's first k-block: fp32 partial to this
//    cluster's workspace slot, then publish it (after all four epilogue warps wrote);
//  * share holding the first k-block: wait for the other clusters' partials of the unit,
//    add them, then finish the tile like a whole unit.
// Hands the accumulator buffer back to the MMA warp (all of this warp's TMEM reads of it
// have completed); `remote`: the barrier is the leader CTA's, at cluster address `tempty`.
__device__ __forceinline__ void release_accumulator(uint32_t tempty, bool remote, uint32_t lane) {
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) {
        if (remote)
            mbar_arrive_remote(tempty);
        else
            mbar_arrive(tempty);
    }
}

// Epilogue of a whole tile with beta = 0 and a 16-bit C: one 64-column TMEM load per
// chunk, the load of chunk c+1 in flight while chunk c is converted and staged, and the
// accumulator released as soon as its last columns are in registers.  Each chunk's store
// leaves as soon as it is staged (sending a tile's stores together measured slower).
template <uint32_t kOut, uint32_t BN>
__device__ __forceinline__ void epilogue_fast(const GemmParams &p, const CUtensorMap *map_c,
                                              uint32_t taddr, int32_t row0, int32_t col0,
                                              uint32_t stg, uint32_t lane, EpiState &es,
                                              uint32_t tempty, bool remote) {
    constexpr uint32_t NCH = BN / 64;
    uint32_t r[64];
    tmem_ld_32x32b_x64(taddr, r);
#pragma unroll
    for (uint32_t c = 0; c < NCH; ++c) {
        tmem_ld_wait(r);
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float lo = __uint_as_float(r[2 * i]) * p.alpha;
            const float hi = __uint_as_float(r[2 * i + 1]) * p.alpha;
            w[i] = kOut == 1 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
        }
        if (c + 1 < NCH)
            tmem_ld_32x32b_x64(taddr + (c + 1) * 64, r);
        else
            release_accumulator(tempty, remote, lane);
        const uint32_t buf = stg + ((es.chunk + c) & (p.epi_bufs - 1u)) * kEpiBufBytes;
        if (lane == 0) wait_staging_free(p.epi_bufs);
        __syncwarp();
        const uint32_t row_addr = buf + lane * 128u;
#pragma unroll
        for (uint32_t j = 0; j < 8; ++j)
            st_shared_v4(row_addr + ((j ^ (lane & 7u)) << 4), w[4 * j], w[4 * j + 1], w[4 * j + 2],
                         w[4 * j + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(map_c, buf, col0 + int32_t(c * 64), row0);
            bulk_commit();
        }
    }
    es.chunk += NCH;
}

template <uint32_t BN>
__device__ __forceinline__ bool epilogue_segment(const GemmParams &p, const CUtensorMap *map_c,
                                                 const CUtensorMap *map_c2,
                                                 uint32_t tmem_base, uint32_t acc,
                                                 const Segment &g, uint32_t m_blk, uint32_t n_blk,
                                                 uint32_t cid, uint32_t ncl, uint32_t rank,
                                                 uint32_t warp, uint32_t lane, uint32_t stg,
                                                 uint32_t c0_bars, EpiState &es,
                                                 uint32_t tempty, bool remote) {
    const size_t slot_quads = size_t(p.cluster) * kTileM * BN / 4;  // float4s per cluster
    float4 *ws4 = reinterpret_cast<float4 *>(p.ws);
    if (g.kb0 > 0) {
        float4 *slot = ws4 + size_t(cid) * slot_quads + size_t(rank) * kTileM * BN / 4;
        epilogue_partial<BN>(tmem_base, acc, warp, lane, slot);
        __threadfence();
        named_bar_sync(1, kEpiWarps * 32);
        if (warp == 0 && lane == 0) st_release_gpu(p.sk_flags + cid * p.cluster + rank, p.ctl.seq);
        return false;
    }
    const float4 *add = nullptr;
    uint32_t add_n = 0;
    uint32_t c_first = 0;
    if (g.kb1 < p.k_blocks) {
        c_first = cid + 1;
        const uint32_t c_last = sk_last_contributor(p, g.u, ncl);
        // every cluster in (cid, c_last] published one partial (the host keeps
        // sk_iters >= clusters, so no share is empty).  The owner relies on those
        // clusters running: they have higher indices, so they are dispatched with or after
        // it; if other work keeps one off the GPU past the time limit, the wait gives up
        // (the error is latched) and this tile of C is left unwritten rather than wrong.
        bool all_ok = true;
        for (uint32_t c = c_first; c <= c_last && all_ok; ++c) {
            bool ok = true;
            if (lane == 0) ok = wait_partial(p, p.sk_flags + c * p.cluster + rank);
            all_ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        __syncwarp();
        if (!all_ok) {
            // the C0 chunks requested ahead for this tile land before their buffers are
            // used again (or the CTA leaves)
            for (uint32_t i = 0; i < es.c0_ahead; ++i) {
                const uint32_t b = (es.chunk + i) & (p.epi_bufs - 1u);
                wait_bounded(c0_bars + 8u * b, (es.c0_phase >> b) & 1u, p.ctl, ROLE_EPILOGUE,
                             false);
                es.c0_phase ^= 1u << b;
            }
            es.c0_ahead = 0;
            return false;
        }
        add = ws4 + size_t(c_first) * slot_quads + size_t(rank) * kTileM * BN / 4 +
              (warp * 32 + lane);
        add_n = c_last + 1 - c_first;
    }
    const int32_t row0 = int32_t(m_blk * kTileM + warp * 32);
    if (row0 >= p.M) return false;
    const bool have_acc = p.k_blocks != 0;
    int32_t col0;
    uint32_t width;
    segment_cols<BN>(g, n_blk, col0, width);
    const uint32_t taddr = tmem_base + ((warp * 32u) << 16) + acc * BN;
    // Common case: a whole tile inside the C descriptor, no C0, no partials, 16-bit C.
    const bool fast = add_n == 0 && have_acc && p.beta == 0.0f && p.out_kind != 0 &&
                      col0 + int32_t(width) <= p.n_store;
    if constexpr (BN % 64 == 0) {
        if (fast && g.half == 0 && p.epi_bufs * 64 >= BN) {
            if (p.out_kind == 1)
                epilogue_fast<1, BN>(p, map_c, taddr, row0, col0, stg, lane, es, tempty, remote);
            else
                epilogue_fast<2, BN>(p, map_c, taddr, row0, col0, stg, lane, es, tempty, remote);
            return true;
        }
    }
    if constexpr ((BN / 2) % 64 == 0) {
        if (fast && g.half != 0 && p.epi_bufs * 64 >= BN / 2) {
            if (p.out_kind == 1)
                epilogue_fast<1, BN / 2>(p, map_c, taddr, row0, col0, stg, lane, es, tempty,
                                         remote);
            else
                epilogue_fast<2, BN / 2>(p, map_c, taddr, row0, col0, stg, lane, es, tempty,
                                         remote);
            return true;
        }
    }
    // a width of 224 leaves a last chunk of 32 columns after the 64-column ones (whole
    // tiles only: half-width tiles are made of 256-wide ones)
    const uint32_t c64 = width / 64;
    const bool narrow = width % 64 != 0;
    const int32_t col_narrow = col0 + int32_t(c64 * 64);
    if (p.out_kind == 1) {
        for (uint32_t c = 0; c < c64 && col0 + int32_t(c * 64) < p.N; ++c)
            epilogue_chunk<1>(p, map_c, taddr + c * 64, have_acc, row0, col0 + int32_t(c * 64),
                              stg, c0_bars, es, lane,
                              add ? add + size_t(c * 16) * kTileM : nullptr, add_n, slot_quads, c);
        if (narrow && col_narrow < p.N)
            epilogue_chunk<1, 32>(p, map_c2, taddr + c64 * 64, have_acc, row0, col_narrow, stg,
                                  c0_bars, es, lane,
                                  add ? add + size_t(c64 * 16) * kTileM : nullptr, add_n,
                                  slot_quads, c64);
    } else if (p.out_kind == 2) {
        for (uint32_t c = 0; c < c64 && col0 + int32_t(c * 64) < p.N; ++c)
            epilogue_chunk<2>(p, map_c, taddr + c * 64, have_acc, row0, col0 + int32_t(c * 64),
                              stg, c0_bars, es, lane,
                              add ? add + size_t(c * 16) * kTileM : nullptr, add_n, slot_quads, c);
        if (narrow && col_narrow < p.N)
            epilogue_chunk<2, 32>(p, map_c2, taddr + c64 * 64, have_acc, row0, col_narrow, stg,
                                  c0_bars, es, lane,
                                  add ? add + size_t(c64 * 16) * kTileM : nullptr, add_n,
                                  slot_quads, c64);
    } else {
        for (uint32_t c = 0; c < width / 32 && col0 + int32_t(c * 32) < p.N; ++c)
            epilogue_chunk<0>(p, map_c, taddr + c * 32, have_acc, row0, col0 + int32_t(c * 32),
                              stg, c0_bars, es, lane,
                              add ? add + size_t(c * 8) * kTileM : nullptr, add_n, slot_quads, c);
    }
    return false;
}

// The epilogue warps' loop over this cluster's segments.  The accumulator buffer of
// segment t is t % kAccBufs; after draining it each warp arrives on tmem_empty[acc] (of
// the leader CTA when a CTA pair shares the MMA).
template <uint32_t BN, bool kPair, uint32_t kAccBufs = 2>
__device__ __forceinline__ void epilogue_run(const GemmParams &p, const CUtensorMap *map_c,
                                             const CUtensorMap *map_c2,
                                             uint32_t tmem_base, uint32_t b_tfull,
                                             uint32_t b_tempty, uint32_t cid, uint32_t ncl,
                                             uint32_t rank, uint32_t warp, uint32_t lane,
                                             uint32_t s_epi, uint32_t b_c0, uint32_t s_clc,
                                             uint32_t lead = 0) {
    const uint32_t stg = s_epi + warp * p.epi_bufs * kEpiBufBytes;
    const uint32_t c0_bars = b_c0 + warp * 8u * kMaxEpiBufs;
    EpiState es;
    uint32_t t = 0;
    SegIter si;
    seg_begin(si, p, cid, ncl, clc_ring(s_clc, lane == 0, ROLE_EPILOGUE, false, false, p.cluster));
    Segment g;
    for (; seg_next(si, p, ncl, g); ++t) {
        const uint32_t acc = kAccBufs == 2 ? t & 1u : 0u;
        const uint32_t acc_phase = kAccBufs == 2 ? (t >> 1) & 1u : t & 1u;
        uint32_t m_blk, n_blk;
        unit_coords(g.u, p, rank, m_blk, n_blk);
        if (g.kb0 == 0) {
            int32_t col0;
            uint32_t width;
            segment_cols<BN>(g, n_blk, col0, width);
            epilogue_prefetch_c0(p, map_c, map_c2, m_blk, col0, width, warp, lane, stg, c0_bars,
                                 es);
        } else
            es.c0_ahead = 0;
        const bool ok = wait_bounded(b_tfull + 8 * acc, acc_phase, p.ctl, ROLE_EPILOGUE);
        if (!__all_sync(0xffffffffu, ok)) {
            // C0 loads issued ahead must land before this CTA can leave
            for (uint32_t i = 0; i < es.c0_ahead; ++i) {
                const uint32_t b = (es.chunk + i) & (p.epi_bufs - 1u);
                wait_bounded(c0_bars + 8u * b, (es.c0_phase >> b) & 1u, p.ctl, ROLE_EPILOGUE, false);
            }
            break;
        }
        tc_fence_after_sync();
        // with CTA pairs the accumulator is handed back on the pair leader's barrier
        const uint32_t tempty = kPair ? mapa_shared(b_tempty + 8 * acc, lead) : b_tempty + 8 * acc;
        if (!epilogue_segment<BN>(p, map_c, map_c2, tmem_base, acc, g, m_blk, n_blk, cid, ncl, rank, warp,
                                  lane, stg, c0_bars, es, tempty, kPair))
            release_accumulator(tempty, kPair, lane);
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
}

}  // namespace tg
