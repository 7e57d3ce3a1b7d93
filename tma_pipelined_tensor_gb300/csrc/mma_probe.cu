// Tensor-core rate probe for sm_103a: CTA pairs issue back-to-back tcgen05 pair MMAs
// (256 x 256 x K per instruction) on operand tiles already in shared memory, with no
// data movement and no epilogue, so that the measured time is the tensor cores' own
// dense rate.  It gives the per-SM FLOP per clock of the nameplate peak (SM count x rate
// x clock), which the pages do not state for this part ("GEMM: la moltiplicazione di
// matrici sull'hardware", tensor-core section: the peaks quoted are per generation, and
// none is GB300's).
#include "ptx.cuh"

namespace tg {

namespace {

constexpr uint32_t kProbeN = 256;                         // MMA N (pair M = 256)
constexpr uint32_t kProbeTileBytes = 128 * kTileKBytes;   // one 128-row, 128-byte-deep tile
// the GEMM's shared-memory floor keeps one CTA per SM, so every pair has its two SMs alone
constexpr uint32_t kProbeSmem = kMinGemmSmem;
static_assert(1024 + 2 * kProbeTileBytes + 64 <= kProbeSmem, "probe tiles fit");

// `timing` (may be null): CTA 0 (the first pair's leader, which issues its MMAs) writes
// the SM cycles and the nanoseconds from just before its first MMA to the completion of
// its last one, so that the rate can be divided by the clock the SMs actually ran at.
template <uint32_t KIND>
__global__ void __launch_bounds__(128, 1) mma_rate_kernel(uint64_t iters, WaitCtl ctl,
                                                          unsigned long long *timing) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sa = base, sb = base + kProbeTileBytes;
    const uint32_t b_drain = sb + kProbeTileBytes, s_slot = b_drain + 8;
    volatile uint32_t *slot_ptr = reinterpret_cast<volatile uint32_t *>(smem_raw + (s_slot - raw));
    const uint32_t warp = warp_id(), lane = lane_id();
    const bool leader = cluster_ctarank() == 0;

    // zero operands: the products are exact and no value can become a NaN
    for (uint32_t i = threadIdx.x * 16; i < 2 * kProbeTileBytes; i += blockDim.x * 16)
        st_shared_v4(base + i, 0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) {
        mbar_init(b_drain, 1);
        fence_mbarrier_init();
    }
    fence_proxy_async_smem();
    if (warp == 0) {
        tmem_alloc_pair(s_slot, kProbeN);
        tmem_relinquish_alloc_permit_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after_sync();
    const uint32_t tmem = *slot_ptr;

    if (warp == 0 && leader) {
        const uint32_t issue = lane == 0;
        const uint32_t kind = KIND == kMmaTf32 ? 4u : KIND == kMmaF8 ? 2u : 0u;
        const uint32_t idesc = umma_idesc_f32(2 * kTileM, kProbeN, kind, 0, 0);
        const uint64_t ad = umma_desc_kmajor_sw128(sa), bd = umma_desc_kmajor_sw128(sb);
        const long long c0 = clock64();
        const uint64_t t0 = globaltimer_ns();
        for (uint64_t it = 0; it < iters; ++it) {
#pragma unroll
            for (uint32_t k = 0; k < kTileKBytes / 32; ++k) {
                const uint32_t acc = (it | k) != 0;
                if constexpr (KIND == kMmaF8)
                    umma_f8_pair(issue, tmem, ad + 2 * k, bd + 2 * k, idesc, acc);
                else if constexpr (KIND == kMmaTf32)
                    umma_tf32_pair(issue, tmem, ad + 2 * k, bd + 2 * k, idesc, acc);
                else
                    umma_bf16_pair(issue, tmem, ad + 2 * k, bd + 2 * k, idesc, acc);
            }
        }
        umma_commit_pair_multicast(issue, b_drain, uint16_t(0x1));
        wait_bounded(b_drain, 0, ctl, ROLE_MMA, false);
        if (timing && blockIdx.x == 0 && lane == 0) {
            timing[0] = static_cast<unsigned long long>(clock64() - c0);
            timing[1] = globaltimer_ns() - t0;
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem, kProbeN);
    }
}

template <uint32_t KIND>
cudaError_t launch_probe(uint32_t pairs, uint64_t iters, const WaitCtl &ctl,
                         unsigned long long *timing, cudaStream_t stream) {
    auto kern = mma_rate_kernel<KIND>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kProbeSmem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = kProbeSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, iters, ctl, timing);
}

}  // namespace

tg_status launch_mma_probe(uint32_t mma_kind, uint32_t pairs, uint64_t iters, const WaitCtl &ctl,
                           unsigned long long *timing, cudaStream_t stream) {
    cudaError_t e;
    switch (mma_kind) {
    case kMmaF8: e = launch_probe<kMmaF8>(pairs, iters, ctl, timing, stream); break;
    case kMmaTf32: e = launch_probe<kMmaTf32>(pairs, iters, ctl, timing, stream); break;
    default: e = launch_probe<kMmaF16>(pairs, iters, ctl, timing, stream); break;
    }
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

}  // namespace tg
