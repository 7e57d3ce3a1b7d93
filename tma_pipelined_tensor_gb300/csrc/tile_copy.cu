// TMA tile copy for sm_103a: every box of a rank 1..5 tensor goes global -> shared memory
// through the tensor descriptor (hardware swizzle, out-of-bounds fill, transaction
// counted on an mbarrier) and its raw shared-memory image goes back to global memory
// with one untiled bulk store.
//
// Sources: "2 . Le Tensor Memory Accelerator" 2.2 (one thread issues the copy by
// coordinates, the hardware computes addresses, edges, swizzle and byte counts), 2.4
// (expect_tx then wait for the bytes); "1 . Asynchronisme et mbarrier" 1.5 (a ring of
// stages so that the load of box n+1 overlaps the store of box n).
//
// The box grid starts at `origin` (0 for the whole-tensor copy; negative coordinates and
// boxes past the end read the fill value, the copy engine's out-of-bounds rule).
// With `back` set the copy runs the other way: each box image is brought in by an
// untiled bulk load and written to the tensor by a tensor store through the same
// descriptor (the pages' TMA store), which restores the dense layout.
// Work split: persistent CTAs of one warp each; CTA b handles boxes b, b + grid, ...
// One elected thread runs the whole pipeline: S loads in flight, and a stage is
// reloaded only after the bulk store that drains it has finished reading it.
#include "ptx.cuh"

namespace tg {

__global__ void __launch_bounds__(32) tma_tile_copy_kernel(const __grid_constant__ CUtensorMap map,
                                                           const CopyParams p) {
    extern __shared__ uint8_t smem_raw[];
    if (threadIdx.x != 0) return;

    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t S = p.stages;
    const uint32_t bars = base + S * p.stage_pitch;
    auto stage = [&](uint32_t s) { return base + s * p.stage_pitch; };
    auto full = [&](uint32_t s) { return bars + 8u * s; };

    for (uint32_t s = 0; s < S; ++s) mbar_init(full(s), 1);
    fence_mbarrier_init();
    prefetch_tensormap(&map);
    // Launched with programmatic stream serialisation: the set-up above overlaps the end
    // of the kernel before it on the stream; nothing in global memory is touched before
    // that kernel has completed.  The next kernel may be scheduled as this one's CTAs leave.
    griddep_launch_dependents();
    griddep_wait();

    const uint32_t first = blockIdx.x, step = gridDim.x;
    const uint32_t n_mine = p.nboxes > first ? (p.nboxes - first + step - 1) / step : 0;

    // Processing index -> box coordinates and image index.  The image always follows the
    // box grid row-major (dimension 0 fastest); `reverse` only changes the order in which
    // the CTAs take the boxes (outermost box index fastest).
    // Dimensions at or beyond the rank have one box (nb = 1), so every loop runs over
    // five dimensions with compile-time indices.
    auto coords = [&](uint32_t pidx, int32_t (&c)[5], uint32_t &image_idx) {
        uint32_t bi[5];
        uint32_t q = pidx;
        if (p.reverse) {
#pragma unroll
            for (int k = 4; k >= 0; --k) {
                bi[k] = q % p.nb[k];
                q /= p.nb[k];
            }
        } else {
#pragma unroll
            for (int k = 0; k < 5; ++k) {
                bi[k] = q % p.nb[k];
                q /= p.nb[k];
            }
        }
        image_idx = 0;
#pragma unroll
        for (int k = 4; k >= 0; --k) image_idx = image_idx * p.nb[k] + bi[k];
#pragma unroll
        for (int k = 0; k < 5; ++k) c[k] = p.origin[k] + int32_t(bi[k] * p.ext[k]);
    };
    auto issue = [&](uint32_t i) {
        int32_t c[5];
        uint32_t image_idx;
        coords(first + i * step, c, image_idx);
        const uint32_t s = i % S;
        mbar_arrive_expect_tx(full(s), p.box_bytes);
        if (p.back)
            bulk_load(stage(s), p.out + size_t(image_idx) * p.box_bytes, p.box_bytes, full(s));
        else
            tma_load_nd(stage(s), &map, full(s), p.rank, c);
    };

    uint32_t issued = 0;
    for (; issued < n_mine && issued < S; ++issued) issue(issued);

    uint32_t i = 0;
    for (; i < n_mine; ++i) {
        const uint32_t s = i % S;
        if (!wait_bounded(full(s), (i / S) & 1u, p.ctl, ROLE_COPY)) break;
        if (p.back) fence_proxy_async_smem();
        int32_t c[5];
        uint32_t image_idx;
        coords(first + i * step, c, image_idx);
        if (p.back)  // the descriptor's tensor store undoes the swizzle and clips at the edge
            tma_store_nd(&map, stage(s), p.rank, c);
        else
            bulk_store(p.out + size_t(image_idx) * p.box_bytes, stage(s), p.box_bytes);
        bulk_commit();
        // Refill the stage drained one iteration ago, once its store has read it.
        if (i >= 1 && issued < n_mine) {
            bulk_wait_read<1>();
            issue(issued);
            ++issued;
        }
    }
    // On an early exit, let the loads already in flight land before the CTA leaves.
    for (uint32_t j = i; j < issued; ++j)
        wait_bounded(full(j % S), (j / S) & 1u, p.ctl, ROLE_COPY, false);
    bulk_wait<0>();
}

tg_status tile_copy_blocks_per_sm(uint32_t smem, int *blocks) {
    cudaError_t e =
        kernel_max_blocks(reinterpret_cast<const void *>(tma_tile_copy_kernel), smem, 32, blocks);
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

tg_status launch_tile_copy(const CopyLaunch &L, cudaStream_t stream) {
    cudaError_t e = kernel_smem_attr(reinterpret_cast<const void *>(tma_tile_copy_kernel), L.smem);
    if (e != cudaSuccess) return TG_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.grid, 1, 1);
    cfg.blockDim = dim3(32, 1, 1);
    cfg.dynamicSmemBytes = L.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, tma_tile_copy_kernel, L.map, L.p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return TG_ERR_CUDA;
    }
    return TG_OK;
}

}  // namespace tg
