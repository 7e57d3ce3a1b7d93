// Persistent, warp-specialised bf16 GEMM for sm_103a:  C <- alpha * A * B + beta * C.
//
// Sources (page title, section):
//  - "GEMM: la moltiplicazione di matrici sull'hardware": tiling (a tile of C is built
//    from a strip of A and a strip of B walked in K blocks, each block loaded once into
//    shared memory and reused for the whole tile), L2-aware launch order ("blocks that
//    run together share the same tiles"), tensor cores (16-bit inputs, fp32 accumulator,
//    C <- alpha*A*B + beta*C), wave quantisation.
//  - "2 . Le Tensor Memory Accelerator": 2.2/2.4 (one thread issues TMA copies by
//    coordinates and announces the expected bytes on an mbarrier), 2.5 (TMA store for
//    the epilogue; multicast of a tile shared by the CTAs of a cluster; zero fill of the
//    out-of-bounds part of edge tiles), 2.6 (warp specialisation: one warp feeds TMA,
//    others compute; data never passes through registers between HBM and the tensor
//    core), 2.8 (Blackwell keeps TMA and adds tensor memory).
//  - "1 . Asynchronisme et mbarrier": 1.4 (mbarrier: byte count + phase bit), 1.5 (an
//    N-stage ring with a "full" and an "empty" barrier per stage).
//
// Roles (192 threads, one CTA per SM):
//  warps 0-3  epilogue: TMEM -> registers (each warp owns one 32-lane quarter of the
//             128-row accumulator), alpha/beta in fp32, convert, stage in swizzled shared
//             memory, TMA store of 32-row boxes.
//  warp 4     TMA producer (one thread): waits empty[s], expect_tx on full[s], issues
//             the A box (128 x 64) and the B box (BN x 64, or its half with multicast).
//  warp 5     MMA issuer (one thread) and TMEM owner: waits full[s], issues four
//             128 x BN x 16 tcgen05.mma per k-block, commits to empty[s]; after the last
//             k-block commits to tmem_full[acc].  The accumulator is double-buffered in
//             TMEM (2 x BN columns) so the epilogue of tile i overlaps the MMAs of i+1.
// Cluster 2: the two CTAs compute vertically adjacent tiles that share one B tile; each
// loads one half of it and multicasts it to both, and each MMA issuer releases a stage
// in both CTAs (empty[s] expects two arrivals).
#include "gemm_common.cuh"

namespace tg {

template <uint32_t BN, uint32_t KIND>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap map_a,
                     const __grid_constant__ CUtensorMap map_b,
                     const __grid_constant__ CUtensorMap map_c,
                     const __grid_constant__ CUtensorMap map_c2, const GemmParams p) {
    constexpr uint32_t A_BYTES = kTileM * kTileKBytes;
    constexpr uint32_t B_BYTES = BN * kTileKBytes;
    // MX operands: each stage also holds A's scale atom and one per 128 columns of B
    constexpr bool MX = KIND == kMmaMx;
    constexpr uint32_t SF_ATOMS = MX ? 1 + BN / kTileM : 0;
    constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES + SF_ATOMS * kSfAtomBytes;
    constexpr uint32_t ACC_COLS = 2 * BN;  // double-buffered fp32 accumulator
    // TMEM: the accumulators, then (MX) four scale columns per atom per stage
    constexpr uint32_t SF_COLS = 4 * SF_ATOMS;
    constexpr uint32_t TMEM_COLS = MX ? 512u : ACC_COLS;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t S = p.stages;
    const uint32_t s_epi = base + S * STAGE_BYTES;
    const uint32_t s_clc = s_epi + kEpiWarps * p.epi_bufs * kEpiBufBytes;  // dynamic-schedule ring
    const uint32_t s_bar = s_clc + kClcBytes;
    const uint32_t b_full = s_bar, b_empty = s_bar + 8 * S;
    const uint32_t b_tfull = s_bar + 16 * S, b_tempty = b_tfull + 16, b_drain = b_tempty + 16;
    const uint32_t b_c0 = b_drain + 8;  // one C0-load barrier per staging buffer slot
    const uint32_t b_xchg = b_c0 + 8 * kMaxEpiBufs * kEpiWarps;  // producers' exit exchange
    const uint32_t s_slot = b_xchg + 8;                           // TMEM base address
    const uint32_t x_words = s_slot + 8;  // exit exchange: [0] k-blocks, [1] CLC requests
    volatile uint32_t *slot_ptr = reinterpret_cast<volatile uint32_t *>(smem_raw + (s_slot - raw));

    const uint32_t warp = warp_id(), lane = lane_id();
    const uint32_t rank = p.cluster > 1 ? cluster_ctarank() : 0u;

    if (warp == 4 && lane == 0) {
        for (uint32_t s = 0; s < S; ++s) {
            mbar_init(b_full + 8 * s, 1);
            mbar_init(b_empty + 8 * s, p.cluster);
        }
        for (uint32_t b = 0; b < 2; ++b) {
            mbar_init(b_tfull + 8 * b, 1);
            mbar_init(b_tempty + 8 * b, kEpiWarps);
        }
        mbar_init(b_drain, 1);
        for (uint32_t i = 0; i < kMaxEpiBufs * kEpiWarps; ++i) mbar_init(b_c0 + 8 * i, 1);
        mbar_init(b_xchg, 1);  // one remote arrival from the other CTA's producer
        if (p.clc) {
            const uint32_t clc_full = s_clc + 16 * kClcSlots, clc_empty = clc_full + 8 * kClcSlots;
            for (uint32_t i = 0; i < kClcSlots; ++i) {
                mbar_init(clc_full + 8 * i, 1);
                mbar_init(clc_empty + 8 * i, clc_consumers(p, false));
                mbar_arrive_expect_tx(clc_full + 8 * i, 16u);  // armed for the slot's first use
            }
        }
        fence_mbarrier_init();
        if (p.k_blocks) {
            prefetch_tensormap(&map_a);
            prefetch_tensormap(&map_b);
        }
        if (p.n_store > 0) prefetch_tensormap(&map_c);
    }
    if (warp == 5) {
        tmem_alloc(s_slot, TMEM_COLS);
        tmem_relinquish_alloc_permit();
    }
    tc_fence_before_sync();
    __syncthreads();
    if (p.cluster > 1) cluster_sync_all();
    tc_fence_after_sync();
    const uint32_t tmem_base = *slot_ptr;
    // Launched with programmatic stream serialisation: the set-up above (barriers, TMEM,
    // descriptor prefetch) overlaps the end of the kernel before it on the stream, and
    // nothing in global memory is touched before that kernel has completed.
    griddep_launch_dependents();
    griddep_wait();

    const uint32_t cid = blockIdx.x / p.cluster;
    const uint32_t ncl = gridDim.x / p.cluster;

    if (warp == 4) {
        // ------------------------------ TMA producer ------------------------------
        {
            // The whole warp runs the loop; lane 0 issues (converged, like the MMA warp).
            const uint32_t issue = lane == 0;
            // test hook: the producers of cluster 0 issue nothing, so the MMA issuers' first
            // waits run out while no copy is in flight in any CTA of the cluster
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
                for (uint32_t kb = g.kb0; kb < g.kb1; ++kb) {
                    if (!wait_bounded(b_empty + 8 * stage, phase ^ 1u, p.ctl, ROLE_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    {
                        const uint32_t full = b_full + 8 * stage;
                        const uint32_t sa = base + stage * STAGE_BYTES, sb = sa + A_BYTES;
                        mbar_arrive_expect_tx(issue, full, STAGE_BYTES);
                        if (p.a_mn) {  // 64-element M boxes, K rows
#pragma unroll
                            for (uint32_t h = 0; h < kTileM / kMnBox; ++h)
                                tma_load_2d(issue, sa + h * kMnBoxBytes, &map_a, full,
                                            int32_t(m_blk * kTileM + h * kMnBox), int32_t(kb * p.kblk));
                        } else {
                            tma_load_2d(issue, sa, &map_a, full, int32_t(kb * p.kblk), int32_t(m_blk * kTileM));
                        }
                        // B rows this CTA loads: all BN, or its half (multicast to both CTAs)
                        const uint32_t rows = p.cluster == 1 ? BN : BN / 2;
                        const uint32_t row0 = n_blk * BN + (p.cluster == 1 ? 0 : rank * rows);
                        const uint32_t dst = sb + (p.cluster == 1 ? 0 : rank * rows * kTileKBytes);
                        if (p.b_mn) {
                            for (uint32_t h = 0; h < rows / kMnBox; ++h) {
                                if (p.cluster == 1)
                                    tma_load_2d(issue, dst + h * kMnBoxBytes, &map_b, full,
                                                int32_t(row0 + h * kMnBox), int32_t(kb * p.kblk));
                                else
                                    tma_load_2d_multicast(issue, dst + h * kMnBoxBytes, &map_b, full,
                                                          int32_t(row0 + h * kMnBox),
                                                          int32_t(kb * p.kblk), uint16_t(0x3));
                            }
                        } else if (p.cluster == 1) {
                            tma_load_2d(issue, dst, &map_b, full, int32_t(kb * p.kblk), int32_t(row0));
                            if constexpr (MX) {
                                // the k-block's scale atoms: A's row group, then B's
                                const uint32_t ssf = sb + B_BYTES;
                                bulk_load(issue, ssf,
                                          p.sfa + (size_t(kb) * p.sf_rb_a + m_blk) * kSfAtomBytes,
                                          kSfAtomBytes, full);
#pragma unroll
                                for (uint32_t h = 0; h < BN / kTileM; ++h)
                                    bulk_load(issue, ssf + (1 + h) * kSfAtomBytes,
                                              p.sfb + (size_t(kb) * p.sf_rb_b + n_blk * (BN / kTileM) + h) *
                                                          kSfAtomBytes,
                                              kSfAtomBytes, full);
                            }
                        } else {
                            tma_load_2d_multicast(issue, dst, &map_b, full, int32_t(kb * p.kblk),
                                                  int32_t(row0), uint16_t(0x3));
                        }
                    }
                    ++issued;
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            clc_drain(si, p);
            // Exit protocol (gemm_common.cuh).  With a cluster of two each CTA's full barrier
            // also counts the half of B that the other CTA multicasts into it: the CTAs
            // exchange their k-block counts (and the requester its launch-control requests,
            // whose responses land in both), then each balances and drains its own ring.
            if (p.cluster > 1) {
                const uint32_t peer = rank ^ 1u;
                st_shared_cluster_u32(issue, mapa_shared(x_words, peer), issued);
                if (rank == 0 && p.clc)
                    st_shared_cluster_u32(issue, mapa_shared(x_words + 4, peer), si.clc_issued);
                mbar_arrive_remote(issue, mapa_shared(b_xchg, peer));
                uint32_t other = issued, requested = 0;
                const bool got =
                    wait_cluster_exit(b_xchg, 0, p.ctl, ROLE_PRODUCER, 2 * p.ctl.timeout_ns);
                if (got) {
                    other = ld_shared_u32(x_words);
                    requested = ld_shared_u32(x_words + 4);
                }
                drain_full_ring(b_full, S, issued, other, B_BYTES / 2, p.ctl, issue);
                if (rank != 0 && p.clc && got) clc_drain_to(si, p, requested);
            } else {
                drain_full_ring(b_full, S, issued, issued, 0, p.ctl, issue);
            }
        }
    } else if (warp == 5) {
        // ------------------------------ MMA issuer --------------------------------
        {
            // The whole warp runs the loop; lane 0 issues (see umma_bf16).
            const uint32_t issue = lane == 0;
            const uint32_t idesc = umma_idesc_f32(kTileM, BN, p.in_kind, p.a_mn, p.b_mn);
            // Descriptors built once and stepped, as in the pair kernel.
            const MmaDescs md = mma_descs(p, base, base + A_BYTES, STAGE_BYTES);
            uint32_t stage = 0, phase = 0, t = 0;
            uint64_t ad = md.a0, bd = md.b0;
            bool ok = true;
            SegIter si;
            seg_begin(si, p, cid, ncl, clc_ring(s_clc, issue, ROLE_MMA, false, false, p.cluster));
            Segment g;
            for (; ok && seg_next(si, p, ncl, g); ++t) {
                const uint32_t acc = t & 1u, acc_phase = (t >> 1) & 1u;
                if (!wait_bounded(b_tempty + 8 * acc, acc_phase ^ 1u, p.ctl, ROLE_MMA)) break;
                tc_fence_after_sync();
                const uint32_t d = tmem_base + acc * BN;
                for (uint32_t kb = g.kb0; kb < g.kb1; ++kb) {
                    if (!wait_bounded(b_full + 8 * stage, phase, p.ctl, ROLE_MMA)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    if constexpr (MX) {
                        // scales into this stage's TMEM columns, then one MMA per 32-element
                        // block, each taking its byte of the 32-bit scale words
                        const uint32_t ssf = base + stage * STAGE_BYTES + A_BYTES + B_BYTES;
                        const uint32_t sfa_t = tmem_base + ACC_COLS + stage * SF_COLS;
#pragma unroll
                        for (uint32_t h = 0; h < SF_ATOMS; ++h)
                            tmem_cp_sf_atom(issue, sfa_t + 4 * h, sf_atom_desc(ssf + h * kSfAtomBytes));
                        const uint32_t fmt = p.in_kind == 6u ? 1u : 0u;
#pragma unroll
                        for (uint32_t k = 0; k < kTileKBytes / 32; ++k)
                            umma_mx(issue, d, ad + k * md.a_k, bd + k * md.b_k,
                                    umma_idesc_mx(kTileM, BN, fmt, k), sfa_t, sfa_t + 4,
                                    (kb != g.kb0 || k > 0) ? 1u : 0u);
                    } else if constexpr (KIND == kMmaF8) {
                        umma_f8(issue, d, ad, bd, idesc, kb != g.kb0);
#pragma unroll
                        for (uint32_t k = 1; k < kTileKBytes / 32; ++k)  // 32 bytes of K per MMA
                            umma_f8(issue, d, ad + k * md.a_k, bd + k * md.b_k, idesc, 1u);
                    } else if constexpr (KIND == kMmaTf32) {
                        umma_tf32(issue, d, ad, bd, idesc, kb != g.kb0);
#pragma unroll
                        for (uint32_t k = 1; k < kTileKBytes / 32; ++k)
                            umma_tf32(issue, d, ad + k * md.a_k, bd + k * md.b_k, idesc, 1u);
                    } else {
                        umma_bf16(issue, d, ad, bd, idesc, kb != g.kb0);
#pragma unroll
                        for (uint32_t k = 1; k < kTileKBytes / 32; ++k)
                            umma_bf16(issue, d, ad + k * md.a_k, bd + k * md.b_k, idesc, 1u);
                    }
                    if (p.cluster == 1)
                        umma_commit(issue, b_empty + 8 * stage);
                    else
                        umma_commit_multicast(issue, b_empty + 8 * stage, uint16_t(0x3));
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
                umma_commit(issue, b_tfull + 8 * acc);
            }
            // All MMAs issued by this warp complete before TMEM is released.
            umma_commit(issue, b_drain);
            wait_bounded(b_drain, 0, p.ctl, ROLE_MMA, false);
        }
    } else {
        // ------------------------------ epilogue ----------------------------------
        epilogue_run<BN, false>(p, &map_c, &map_c2, tmem_base, b_tfull, b_tempty, cid, ncl, rank, warp, lane,
                                 s_epi, b_c0, s_clc);
    }

    // ---------------------------------- teardown ----------------------------------
    tc_fence_before_sync();
    __syncthreads();
    if (p.cluster > 1) cluster_sync_all();
    if (warp == 5) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <uint32_t BN, uint32_t KIND>
static cudaError_t launch_bn(const GemmLaunch &L, cudaStream_t stream) {
    auto kern = gemm_bf16_kernel<BN, KIND>;
    cudaError_t e = kernel_smem_attr(reinterpret_cast<const void *>(kern), L.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.grid, 1, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = L.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = L.p.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, L.map_a, L.map_b, L.map_c, L.map_c2, L.p);
}

tg_status launch_gemm(const GemmLaunch &L, cudaStream_t stream) {
    if (L.pair) return launch_gemm_pair(L, stream);
    // one kernel per MMA kind: kind::f16, kind::f8f6f4 or kind::tf32
    cudaError_t e;
    if (gemm_mma_kind(L.p.in_kind) == kMmaMx) {  // MX operands: 128-wide tiles, one CTA each
        if (L.tile_n != 128 || L.p.cluster != 1) return TG_ERR_UNSUPPORTED;
        e = launch_bn<128, kMmaMx>(L, stream);
        return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
    }
    switch (gemm_mma_kind(L.p.in_kind) * 2 + (L.tile_n == 256 ? 1 : 0)) {
    case 0: e = launch_bn<128, kMmaF16>(L, stream); break;
    case 1: e = launch_bn<256, kMmaF16>(L, stream); break;
    case 2: e = launch_bn<128, kMmaF8>(L, stream); break;
    case 3: e = launch_bn<256, kMmaF8>(L, stream); break;
    case 4: e = launch_bn<128, kMmaTf32>(L, stream); break;
    default: e = launch_bn<256, kMmaTf32>(L, stream); break;
    }
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

// All MMA kinds share the launch shape, registers aside; the 16-bit one stands for all.
template <uint32_t BN>
static cudaError_t clusters_bn(uint32_t smem, uint32_t cluster, int *clusters) {
    auto kern = gemm_bf16_kernel<BN, kMmaF16>;
    return kernel_max_clusters(reinterpret_cast<const void *>(kern), smem, kGemmThreads, cluster,
                               clusters);
}

tg_status gemm_max_active_clusters(uint32_t tile_n, uint32_t smem, uint32_t cluster,
                                   int *clusters) {
    cudaError_t e = tile_n == 256 ? clusters_bn<256>(smem, cluster, clusters)
                                  : clusters_bn<128>(smem, cluster, clusters);
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

}  // namespace tg
