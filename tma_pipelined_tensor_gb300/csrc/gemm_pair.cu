// CTA-pair bf16 GEMM for sm_103a: C <- alpha * A * B + beta * C with 256 x BN output
// tiles computed by a cluster of two CTAs through tcgen05.mma.cta_group::2.
//
// Sources (page title, section): "GEMM: la moltiplicazione di matrici sull'hardware"
// (tiling: a larger tile does more work per byte brought in; the register/accumulator
// budget, not shared memory, caps the tile; the tile is loaded once and reused), "2 .
// Le Tensor Memory Accelerator" 2.5 (a tile needed by the blocks of a cluster is read
// once and delivered to all of them), 2.8 (Blackwell: tensor memory), "1 . Asynchronisme
// et mbarrier" 1.5 (full/empty stage ring).
//
// Why a pair: one 128 x 256 x 16 MMA per SM reads 12 KiB of operands from shared
// memory while TMA writes 48 KiB per 64-deep k-block into it.  With the pair MMA each
// SM stages only its 128 rows of A and its half of B (32 KiB per k-block) and the
// tensor cores of both SMs share each CTA's half of B, so operand traffic per SM drops
// by a third and six stages fit in shared memory.
//
// Roles (192 threads per CTA, cluster of 2, leader = rank 0):
//  warp 4  producer, both CTAs: per k-block waits its own empty[s], then TMA-loads its
//          128 x 64 slice of A and its (BN/2) x 64 slice of B into its own shared memory;
//          both loads count their bytes on the LEADER's full[s] (the leader announces
//          the pair's total with expect_tx).
//  warp 5  TMEM owner in both CTAs (pair allocation); in the leader one thread issues
//          four 256 x BN x 16 pair MMAs per k-block and commits to empty[s] of both CTAs,
//          then to tmem_full[acc] of both CTAs.  The accumulator is double-buffered.
//  0-3     epilogue in both CTAs: each CTA drains its 128 accumulator rows (same code as
//          the single-CTA kernel) and then arrives on the leader's tmem_empty[acc],
//          which expects eight warps.
//
// MX operands (KIND = kMmaMx, 256-wide tiles): each stage also brings, by TMA on the
// leader's full barrier, the k-block's scale atom of the CTA's 128 A rows and the two atoms
// of the tile's 256 B rows (both CTAs hold all of B's scales).  The leader copies them into
// TMEM columns above the accumulator (tcgen05.cp.cta_group::2: each CTA's atoms into its
// own TMEM) before the stage's four block-scaled pair MMAs.  The scale columns of a stage
// and a 256-column accumulator do not fit twice in 512 columns, so the accumulator is
// single-buffered: the next tile's first MMA waits until the epilogue has read the last
// columns out of TMEM.
//
// Measured at 8192^3 (MXE4M3): each scale copy costs about 50 tensor-pipe cycles, in line
// with the MMAs (three per 538-cycle k-block, 20 %; without them the kernel runs as fast
// as plain E4M3).  Storing the scales from four extra warps with tcgen05.st instead, so
// that the tensor pipe does not carry them, was 2x slower: those stores wait while MMAs
// are in flight, and every k-block serialised.
#include "gemm_common.cuh"

namespace tg {

template <uint32_t BN, uint32_t KIND, bool QUAD>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_pair_kernel(const __grid_constant__ CUtensorMap map_a,
                          const __grid_constant__ CUtensorMap map_b,
                          const __grid_constant__ CUtensorMap map_c,
                          const __grid_constant__ CUtensorMap map_c2,
                          const __grid_constant__ CUtensorMap map_sfa,
                          const __grid_constant__ CUtensorMap map_sfb, const GemmParams p) {
    constexpr uint32_t A_BYTES = kTileM * kTileKBytes;      // this CTA's 128 rows of A
    constexpr uint32_t B_BYTES = (BN / 2) * kTileKBytes;    // this CTA's half of the B tile
    constexpr uint32_t OPER_BYTES = A_BYTES + B_BYTES;      // one stage of the operand ring
    constexpr bool MX = KIND == kMmaMx;
    // MX: per stage A's scale atom and one atom per 128 B rows, after the operand ring
    constexpr uint32_t SF_ATOMS = MX ? 1 + BN / kTileM : 0;
    constexpr uint32_t SF_BYTES = SF_ATOMS * kSfAtomBytes, SF_COLS = 4 * SF_ATOMS;
    constexpr uint32_t STAGE_BYTES = OPER_BYTES + SF_BYTES;  // bytes one CTA brings per stage
    // QUAD: a cluster of two pairs stacked along M; each CTA loads a quarter of the shared
    // B tile and multicasts it to the same-parity CTA of the other pair
    constexpr uint32_t CL = QUAD ? 4u : 2u;                  // CTAs per cluster
    constexpr uint32_t BQ_ROWS = BN / 4, BQ_BYTES = BQ_ROWS * kTileKBytes;
    constexpr uint32_t ACC_BUFS = MX ? 1u : 2u;  // double-buffered accumulator, except MX
    constexpr uint32_t ACC_COLS = ACC_BUFS * BN;
    // TMEM is allocated in powers of two: 224-wide tiles use 448 of 512 columns
    constexpr uint32_t TMEM_COLS = MX || ACC_COLS > 256 ? 512u : 256u;
    static_assert(!MX || BN == 256, "MX pair tiles are 256 wide");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t S = p.stages;
    // MX: the stages' scale atoms come first, at the lowest addresses, and the operand
    // ring after them on the next 1024-byte boundary.  The pair scale copy read the
    // wrong rows from sources whose address had bit 15 set (a ring of 3 or 5 stages
    // placed them at 0x18000 or 0x28000; 2 and 4 stages, at 0x10000 and 0x20000, were
    // right); here the scale region takes at most 6 x 1536 bytes from the start of
    // shared memory, far below bit 15.
    const uint32_t s_sf = (raw + 1023u) & ~1023u;  // SF_BYTES per stage
    const uint32_t base = s_sf + (MX ? (S * SF_BYTES + 1023u) & ~1023u : 0u);
    const uint32_t s_epi = base + S * OPER_BYTES;
    const uint32_t s_clc = s_epi + kEpiWarps * p.epi_bufs * kEpiBufBytes;  // dynamic-schedule ring
    const uint32_t s_bar = s_clc + kClcBytes;
    const uint32_t b_full = s_bar, b_empty = s_bar + 8 * S;
    const uint32_t b_tfull = s_bar + 16 * S, b_tempty = b_tfull + 16, b_drain = b_tempty + 16;
    const uint32_t b_c0 = b_drain + 8;  // one C0-load barrier per staging buffer slot
    const uint32_t b_xchg = b_c0 + 8 * kMaxEpiBufs * kEpiWarps;  // producers' exit exchange
    const uint32_t s_slot = b_xchg + 8;                           // TMEM base address
    // exit exchange: [0] the peer's k-blocks, [1] CLC requests, [2 + r] k-blocks of rank r
    const uint32_t x_words = s_slot + 8;
    volatile uint32_t *slot_ptr = reinterpret_cast<volatile uint32_t *>(smem_raw + (s_slot - raw));

    const uint32_t warp = warp_id(), lane = lane_id();
    const uint32_t rank = cluster_ctarank();
    const uint32_t lead = rank & ~1u;        // this CTA's pair leader (cluster rank)
    const bool leader = rank == lead;
    const uint16_t pair_mask = uint16_t(0x3u << lead);

    if (warp == 4 && lane == 0) {
        for (uint32_t s = 0; s < S; ++s) {
            mbar_init(b_full + 8 * s, 1);   // leader: its expect_tx arrival + both CTAs' bytes
            mbar_init(b_empty + 8 * s, QUAD ? 2 : 1);  // one commit per pair that read the stage
        }
        for (uint32_t b = 0; b < 2; ++b) {
            mbar_init(b_tfull + 8 * b, 1);
            mbar_init(b_tempty + 8 * b, 2 * kEpiWarps);  // leader: epilogue warps of both CTAs
        }
        mbar_init(b_drain, 1);
        for (uint32_t i = 0; i < kMaxEpiBufs * kEpiWarps; ++i) mbar_init(b_c0 + 8 * i, 1);
        mbar_init(b_xchg, QUAD ? 3 : 1);  // remote arrivals from the other producers
        if (p.clc) {
            const uint32_t clc_full = s_clc + 16 * kClcSlots, clc_empty = clc_full + 8 * kClcSlots;
            for (uint32_t i = 0; i < kClcSlots; ++i) {
                mbar_init(clc_full + 8 * i, 1);
                mbar_init(clc_empty + 8 * i, clc_consumers(p, true));
                mbar_arrive_expect_tx(clc_full + 8 * i, 16u);  // armed for the slot's first use
            }
        }
        fence_mbarrier_init();
        if (p.k_blocks) {
            prefetch_tensormap(&map_a);
            prefetch_tensormap(&map_b);
            if constexpr (MX) {
                prefetch_tensormap(&map_sfa);
                prefetch_tensormap(&map_sfb);
            }
        }
        if (p.n_store > 0) prefetch_tensormap(&map_c);
        if (p.n_store > 0 && BN % 64 != 0) prefetch_tensormap(&map_c2);
    }
    if (warp == 5) {
        tmem_alloc_pair(s_slot, TMEM_COLS);
        tmem_relinquish_alloc_permit_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after_sync();
    const uint32_t tmem_base = *slot_ptr;
    // Launched with programmatic stream serialisation: the set-up above (barriers, TMEM,
    // descriptor prefetch) overlaps the end of the kernel before it on the stream, and
    // nothing in global memory is touched before that kernel has completed.
    griddep_launch_dependents();
    griddep_wait();

    const uint32_t cid = blockIdx.x / CL;
    const uint32_t ncl = gridDim.x / CL;

    if (warp == 4) {
        // ------------------------------ TMA producer ------------------------------
        {
            // The whole warp runs the loop; lane 0 issues (converged, like the MMA warp).
            const uint32_t issue = lane == 0;
            // test hook: the producers of cluster 0 issue nothing, so the MMA issuer's first
            // wait runs out while no copy is in flight in either CTA of the cluster
            const bool hooked = (p.flags & TG_GEMM_FLAG_TEST_SKIP_FIRST_LOAD) && cid == 0;
            uint32_t stage = 0, phase = 0, issued = 0;
            bool ok = !hooked;
            SegIter si;
            seg_begin(si, p, cid, ncl,
                      clc_ring(s_clc, issue, ROLE_PRODUCER, rank == 0, true, p.cluster));
            Segment g;
            while (ok && seg_next(si, p, ncl, g)) {
                uint32_t m_blk, n_blk;
                unit_coords(g.u, p, rank, m_blk, n_blk);
                int32_t col0;
                uint32_t width;
                segment_cols<BN>(g, n_blk, col0, width);
                // this CTA's half of the segment's B rows; a half-width segment uses the
                // first width / 2 of the rows its (BN / 2)-row box brings
                const int32_t b_row = col0 + int32_t((rank & 1u) * (width / 2));
                for (uint32_t kb = g.kb0; kb < g.kb1; ++kb) {
                    if (!wait_bounded(b_empty + 8 * stage, phase ^ 1u, p.ctl, ROLE_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_leader = mapa_shared(b_full + 8 * stage, lead);
                    if (leader) mbar_arrive_expect_tx(issue, b_full + 8 * stage, 2 * STAGE_BYTES);
                    const uint32_t sa = base + stage * OPER_BYTES, sb = sa + A_BYTES;
                    if (p.a_mn) {  // 64-element M boxes, K rows
#pragma unroll
                        for (uint32_t h = 0; h < kTileM / kMnBox; ++h)
                            tma_load_2d_pair(issue, sa + h * kMnBoxBytes, &map_a, full_leader,
                                             int32_t(m_blk * kTileM + h * kMnBox),
                                             int32_t(kb * p.kblk));
                    } else {
                        tma_load_2d_pair(issue, sa, &map_a, full_leader, int32_t(kb * p.kblk),
                                         int32_t(m_blk * kTileM));
                    }
                    if constexpr (QUAD) {
                        // this CTA's quarter of its pair's B half, delivered to it and to the
                        // CTA of the same parity in the other pair (same rows, same offset)
                        const uint32_t q = rank >> 1;
                        tma_load_2d_pair_multicast(issue, sb + q * BQ_BYTES, &map_b, full_leader,
                                                   int32_t(kb * p.kblk),
                                                   b_row + int32_t(q * BQ_ROWS),
                                                   uint16_t(0x5u << (rank & 1u)));
                    } else if (p.b_mn) {
#pragma unroll
                        for (uint32_t h = 0; h < (BN / 2) / kMnBox; ++h)
                            tma_load_2d_pair(issue, sb + h * kMnBoxBytes, &map_b, full_leader,
                                             b_row + int32_t(h * kMnBox), int32_t(kb * p.kblk));
                    } else {
                        tma_load_2d_pair(issue, sb, &map_b, full_leader, int32_t(kb * p.kblk),
                                         b_row);
                    }
                    if constexpr (MX) {
                        // scale atoms: one row of 512 bytes per (k-block, 128-row group);
                        // A's group of this CTA, then the tile's BN / 128 groups of B
                        const uint32_t ssf = s_sf + stage * SF_BYTES;
                        tma_load_2d_pair(issue, ssf, &map_sfa, full_leader, 0,
                                         int32_t(kb * p.sf_rb_a + m_blk));
                        tma_load_2d_pair(issue, ssf + kSfAtomBytes, &map_sfb, full_leader, 0,
                                         int32_t(kb * p.sf_rb_b + n_blk * (BN / kTileM)));
                    }
                    ++issued;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            clc_drain(si, p);
            // Exit protocol (gemm_common.cuh): the leader's full barriers count both CTAs'
            // bytes, so the peer reports its k-block count to the leader, which balances
            // and drains every phase in flight; in dynamic mode the leader reports its
            // launch-control requests, whose responses also land in the peer.
            if constexpr (QUAD) {
                // every producer's copies count on both leaders' barriers: each reports its
                // k-block count to both leaders, which balance and drain with all four
                for (uint32_t l = 0; l < CL; l += 2) {
                    if (l == rank) continue;
                    st_shared_cluster_u32(issue, mapa_shared(x_words + 8 + 4 * rank, l), issued);
                    mbar_arrive_remote(issue, mapa_shared(b_xchg, l));
                }
                if (leader) {
                    uint32_t n[4] = {issued, issued, issued, issued};
                    if (wait_cluster_exit(b_xchg, 0, p.ctl, ROLE_PRODUCER, 2 * p.ctl.timeout_ns)) {
                        for (uint32_t r = 0; r < 4; ++r)
                            if (r != rank) n[r] = ld_shared_u32(x_words + 8 + 4 * r);
                    }
                    // this pair's CTAs bring their A and B quarter; the other pair's CTAs
                    // their multicast B quarter
                    uint32_t contrib[4];
                    for (uint32_t r = 0; r < 4; ++r)
                        contrib[r] = (r & ~1u) == lead ? A_BYTES + BQ_BYTES : BQ_BYTES;
                    drain_full_ring_n<4>(b_full, S, n, contrib, rank, 2 * STAGE_BYTES, p.ctl, issue);
                }
            } else {
                if (!leader) st_shared_cluster_u32(issue, mapa_shared(x_words, 0), issued);
                if (leader && p.clc)
                    st_shared_cluster_u32(issue, mapa_shared(x_words + 4, 1), si.clc_issued);
                if (!leader || p.clc) mbar_arrive_remote(issue, mapa_shared(b_xchg, rank ^ 1u));
                if (leader) {
                    uint32_t other = issued;
                    if (wait_cluster_exit(b_xchg, 0, p.ctl, ROLE_PRODUCER, 2 * p.ctl.timeout_ns))
                        other = ld_shared_u32(x_words);
                    drain_full_ring(b_full, S, issued, other, STAGE_BYTES, p.ctl, issue);
                } else if (p.clc) {
                    if (wait_cluster_exit(b_xchg, 0, p.ctl, ROLE_PRODUCER, 2 * p.ctl.timeout_ns))
                        clc_drain_to(si, p, ld_shared_u32(x_words + 4));
                }
            }
        }
    } else if (warp == 5) {
        // ----------------------- MMA issuer (leader CTA only) ----------------------
        if (leader) {
            // The whole warp runs the loop; lane 0 issues (see umma_bf16).
            const uint32_t issue = lane == 0;
            const uint32_t idesc_full = umma_idesc_f32(2 * kTileM, BN, p.in_kind, p.a_mn, p.b_mn);
            const uint32_t idesc_half = umma_idesc_f32(2 * kTileM, BN / 2, p.in_kind, p.a_mn, p.b_mn);
            // The tensor core takes MMAs from a short queue, so everything this thread does
            // between them can leave it idle: descriptors are built once for stage 0 and
            // then only stepped (by a stage, or by 32 bytes of K per MMA).
            const MmaDescs md = mma_descs(p, base, base + A_BYTES, OPER_BYTES);
            uint32_t stage = 0, phase = 0, t = 0;
            uint64_t ad = md.a0, bd = md.b0;
            bool ok = true;
            SegIter si;
            seg_begin(si, p, cid, ncl, clc_ring(s_clc, issue, ROLE_MMA, false, false, p.cluster));
            Segment g;
            for (; ok && seg_next(si, p, ncl, g); ++t) {
                const uint32_t acc = ACC_BUFS == 2 ? t & 1u : 0u;
                const uint32_t acc_phase = ACC_BUFS == 2 ? (t >> 1) & 1u : t & 1u;
                if (!wait_bounded_cluster(b_tempty + 8 * acc, acc_phase ^ 1u, p.ctl, ROLE_MMA)) break;
                tc_fence_after_sync();
                const uint32_t d = tmem_base + acc * BN;
                const uint32_t idesc = g.half ? idesc_half : idesc_full;  // N = BN or BN / 2
                for (uint32_t kb = g.kb0; kb < g.kb1; ++kb) {
                    if (!wait_bounded(b_full + 8 * stage, phase, p.ctl, ROLE_MMA)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    if constexpr (MX) {
                        // the stage's scale atoms into its TMEM columns (in both CTAs), then
                        // one MMA per 32-element block taking its byte of the scale words
                        const uint32_t ssf = s_sf + stage * SF_BYTES;
                        const uint32_t sf_t = tmem_base + ACC_COLS + stage * SF_COLS;
#pragma unroll
                        for (uint32_t h = 0; h < SF_ATOMS; ++h)
                            tmem_cp_sf_atom_pair(issue, sf_t + 4 * h,
                                                 sf_atom_desc(ssf + h * kSfAtomBytes));
                        const uint32_t fmt = p.in_kind == 6u ? 1u : 0u;
#pragma unroll
                        for (uint32_t k = 0; k < kTileKBytes / 32; ++k)
                            umma_mx_pair(issue, d, ad + k * md.a_k, bd + k * md.b_k,
                                         umma_idesc_mx(2 * kTileM, BN, fmt, k), sf_t, sf_t + 4,
                                         (kb != g.kb0 || k > 0) ? 1u : 0u);
                    } else if constexpr (KIND == kMmaF8) {
                        umma_f8_pair(issue, d, ad, bd, idesc, kb != g.kb0);
#pragma unroll
                        for (uint32_t k = 1; k < kTileKBytes / 32; ++k)  // 32 bytes of K per MMA
                            umma_f8_pair(issue, d, ad + k * md.a_k, bd + k * md.b_k, idesc, 1u);
                    } else if constexpr (KIND == kMmaTf32) {
                        umma_tf32_pair(issue, d, ad, bd, idesc, kb != g.kb0);
#pragma unroll
                        for (uint32_t k = 1; k < kTileKBytes / 32; ++k)
                            umma_tf32_pair(issue, d, ad + k * md.a_k, bd + k * md.b_k, idesc, 1u);
                    } else {
                        umma_bf16_pair(issue, d, ad, bd, idesc, kb != g.kb0);
#pragma unroll
                        for (uint32_t k = 1; k < kTileKBytes / 32; ++k)
                            umma_bf16_pair(issue, d, ad + k * md.a_k, bd + k * md.b_k, idesc, 1u);
                    }
                    // the stage is free again in every CTA whose copies it holds
                    umma_commit_pair_multicast(issue, b_empty + 8 * stage,
                                               QUAD ? uint16_t(0xF) : pair_mask);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                        ad = md.a0;
                        bd = md.b0;
                    } else {
                        ad += md.stage;
                        bd += md.stage;
                    }
                }
                if (!ok) break;
                umma_commit_pair_multicast(issue, b_tfull + 8 * acc, pair_mask);
            }
            // All pair MMAs complete before either CTA releases its TMEM.
            umma_commit_pair_multicast(issue, b_drain, uint16_t(1u << lead));
            wait_bounded(b_drain, 0, p.ctl, ROLE_MMA, false);
        }
    } else {
        // ---------------------- epilogue (both CTAs) -----------------------------
        epilogue_run<BN, true, ACC_BUFS>(p, &map_c, &map_c2, tmem_base, b_tfull, b_tempty, cid, ncl,
                                         rank, warp, lane, s_epi, b_c0, s_clc, lead);
    }

    // ---------------------------------- teardown ----------------------------------
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();
    if (warp == 5) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

template <uint32_t BN, uint32_t KIND, bool QUAD>
static cudaError_t launch_pair_bn(const GemmLaunch &L, cudaStream_t stream) {
    auto kern = gemm_bf16_pair_kernel<BN, KIND, QUAD>;
    cudaError_t e = kernel_smem_attr(reinterpret_cast<const void *>(kern), L.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.grid, 1, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = L.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = QUAD ? 4 : 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, L.map_a, L.map_b, L.map_c, L.map_c2, L.map_sfa,
                              L.map_sfb, L.p);
}

tg_status launch_gemm_pair(const GemmLaunch &L, cudaStream_t stream) {
    cudaError_t e;
    if (gemm_mma_kind(L.p.in_kind) == kMmaMx) {  // MX: 256-wide tiles, one pair per cluster
        if (L.tile_n != 256 || L.p.cluster != 2) return TG_ERR_UNSUPPORTED;
        e = launch_pair_bn<256, kMmaMx, false>(L, stream);
        return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
    }
    const uint32_t w = L.tile_n == 256 ? 2u : L.tile_n == 224 ? 1u : 0u;
    if (L.p.cluster == 4) {  // two pairs sharing B (16-bit operands only)
        if (gemm_mma_kind(L.p.in_kind) != kMmaF16) return TG_ERR_UNSUPPORTED;
        e = w == 2   ? launch_pair_bn<256, kMmaF16, true>(L, stream)
            : w == 1 ? launch_pair_bn<224, kMmaF16, true>(L, stream)
                     : launch_pair_bn<128, kMmaF16, true>(L, stream);
        return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
    }
    switch (gemm_mma_kind(L.p.in_kind) * 3 + w) {
    case 0: e = launch_pair_bn<128, kMmaF16, false>(L, stream); break;
    case 1: e = launch_pair_bn<224, kMmaF16, false>(L, stream); break;
    case 2: e = launch_pair_bn<256, kMmaF16, false>(L, stream); break;
    case 3: e = launch_pair_bn<128, kMmaF8, false>(L, stream); break;
    case 4: e = launch_pair_bn<224, kMmaF8, false>(L, stream); break;
    case 5: e = launch_pair_bn<256, kMmaF8, false>(L, stream); break;
    case 6: e = launch_pair_bn<128, kMmaTf32, false>(L, stream); break;
    case 7: e = launch_pair_bn<224, kMmaTf32, false>(L, stream); break;
    default: e = launch_pair_bn<256, kMmaTf32, false>(L, stream); break;
    }
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

// The MMA kinds without block scales share the launch shape, registers aside; the 16-bit
// one stands for them.
template <uint32_t BN, uint32_t KIND, bool QUAD>
static cudaError_t pair_clusters_bn(uint32_t smem, int *clusters) {
    auto kern = gemm_bf16_pair_kernel<BN, KIND, QUAD>;
    return kernel_max_clusters(reinterpret_cast<const void *>(kern), smem, kGemmThreads,
                               QUAD ? 4u : 2u, clusters);
}

tg_status gemm_pair_max_active_clusters(uint32_t tile_n, uint32_t smem, uint32_t cluster,
                                        int *clusters, bool mx) {
    const bool quad = cluster == 4;
    if (mx) {
        if (tile_n != 256 || quad) return TG_ERR_UNSUPPORTED;
        return pair_clusters_bn<256, kMmaMx, false>(smem, clusters) == cudaSuccess ? TG_OK
                                                                                   : TG_ERR_CUDA;
    }
    cudaError_t e = tile_n == 256 ? (quad ? pair_clusters_bn<256, kMmaF16, true>(smem, clusters)
                                          : pair_clusters_bn<256, kMmaF16, false>(smem, clusters))
                    : tile_n == 224 ? (quad ? pair_clusters_bn<224, kMmaF16, true>(smem, clusters)
                                            : pair_clusters_bn<224, kMmaF16, false>(smem, clusters))
                                    : (quad ? pair_clusters_bn<128, kMmaF16, true>(smem, clusters)
                                            : pair_clusters_bn<128, kMmaF16, false>(smem, clusters));
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

}  // namespace tg
