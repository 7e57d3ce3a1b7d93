// Inline-PTX primitives for sm_103a: mbarrier, TMA (cp.async.bulk.tensor), bulk
// copies, cluster helpers and the 5th-generation tensor core (tcgen05 + TMEM).
//
// Every wait in the kernels goes through wait_bounded(), which gives up after a
// time limit and latches TG_ERR_DEVICE_TIMEOUT in the device status word instead of
// spinning forever.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "tg.h"
#include "tg_internal.h"

namespace tg {

// ----------------------------------------------------------------------------------
// Addresses, clocks, warps
// ----------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ uint32_t warp_id() {
    return __shfl_sync(0xffffffffu, threadIdx.x >> 5, 0);
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// All threads of all CTAs of the cluster (every thread must execute it).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ----------------------------------------------------------------------------------
// mbarrier: 8 bytes in shared memory with an arrival count, a transaction-byte count
// and a phase bit.
// ----------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy and to the cluster.
__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

// Converged-warp form: performed only by the lane whose `issue` is non-zero.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t issue, uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .pred e;\n\t"
                 "setp.ne.b32 e, %2, 0;\n\t"
                 "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar),
                 "r"(bytes), "r"(issue)
                 : "memory");
}

// Converged-warp form: completes `bytes` transaction bytes of the current phase of a local
// barrier, as if an asynchronous copy of that size had landed on it.
__device__ __forceinline__ void mbar_complete_tx(uint32_t issue, uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .pred e;\n\t"
                 "setp.ne.b32 e, %2, 0;\n\t"
                 "@e mbarrier.complete_tx.shared::cta.b64 [%0], %1;\n\t}" ::"r"(bar),
                 "r"(bytes), "r"(issue)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Same wait with cluster-scope acquire: for barriers that threads of the peer CTA
// arrive on remotely.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Shared::cluster address of the object at shared offset `addr` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrive (release at cluster scope) on a barrier given by its shared::cluster address.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

// Converged-warp form: performed only by the lane whose `issue` is non-zero.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t issue, uint32_t cluster_addr) {
    asm volatile("{\n\t.reg .pred e;\n\t"
                 "setp.ne.b32 e, %1, 0;\n\t"
                 "@e mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n\t}" ::"r"(
                     cluster_addr),
                 "r"(issue)
                 : "memory");
}

// Converged-warp form: stores a 32-bit word at a shared::cluster address (a word of this
// or the peer CTA's shared memory); performed only by the lane whose `issue` is non-zero.
__device__ __forceinline__ void st_shared_cluster_u32(uint32_t issue, uint32_t cluster_addr,
                                                      uint32_t v) {
    asm volatile("{\n\t.reg .pred e;\n\t"
                 "setp.ne.b32 e, %2, 0;\n\t"
                 "@e st.shared::cluster.u32 [%0], %1;\n\t}" ::"r"(cluster_addr), "r"(v),
                 "r"(issue)
                 : "memory");
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// ----------------------------------------------------------------------------------
// Cluster launch control: a running cluster asks the hardware to cancel the launch of
// a cluster of the same grid that has not started yet, and takes over its work.  The
// 16-byte response lands at `resp` (in every CTA of the cluster when `multicast`) and
// completes 16 transaction bytes on the barrier at `bar` (same offset in every CTA).
// A request must not be issued once a response has reported failure.
// ----------------------------------------------------------------------------------
__device__ __forceinline__ void clc_try_cancel(uint32_t issue, uint32_t resp, uint32_t bar,
                                               bool multicast) {
    if (multicast)
        asm volatile("{\n\t.reg .pred e;\n\t"
                     "setp.ne.b32 e, %2, 0;\n\t"
                     "@e clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes"
                     ".multicast::cluster::all.b128 [%0], [%1];\n\t}" ::"r"(resp),
                     "r"(bar), "r"(issue)
                     : "memory");
    else
        asm volatile("{\n\t.reg .pred e;\n\t"
                     "setp.ne.b32 e, %2, 0;\n\t"
                     "@e clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes"
                     ".b128 [%0], [%1];\n\t}" ::"r"(resp),
                     "r"(bar), "r"(issue)
                     : "memory");
}

// Reads the response at `resp`: true, and the x index of the cancelled cluster's first
// CTA, when a cluster was cancelled; false when none was left to cancel.
__device__ __forceinline__ bool clc_query(uint32_t resp, uint32_t &ctaid_x) {
    uint32_t ok, x = 0;
    asm volatile("{\n\t.reg .pred p;\n\t.reg .b128 r;\n\t"
                 "ld.shared.b128 r, [%2];\n\t"
                 "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
                 "selp.u32 %1, 1, 0, p;\n\t"
                 "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %0, r;\n\t}"
                 : "+r"(x), "=r"(ok)
                 : "r"(resp)
                 : "memory");
    ctaid_x = x;
    return ok != 0;
}

// Roles reported in bits 8-11 of the status word when a wait gives up.
enum : uint32_t { ROLE_PRODUCER = 1, ROLE_MMA = 2, ROLE_EPILOGUE = 3, ROLE_COPY = 4 };

__device__ __forceinline__ uint32_t status_peek(const uint32_t *status) {
    return *reinterpret_cast<const volatile uint32_t *>(status);
}

// Slow path of wait_bounded (kept out of line so the hot loops stay small).
static __device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, uint32_t *status,
                                              uint64_t timeout_ns, uint32_t seq, uint32_t role,
                                              bool obey_abort) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((n & 63u) == 0) {
            if (obey_abort && status_peek(status + 1) == seq) return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                const uint32_t word = uint32_t(TG_ERR_DEVICE_TIMEOUT) | (role << 8) |
                                      ((blockIdx.x & 0xffffu) << 16);
                atomicCAS(status, 0u, word);
                atomicExch(status + 1, seq);
                return false;
            }
        }
    }
}

static __device__ __noinline__ bool wait_slow_cluster(uint32_t bar, uint32_t parity,
                                                      uint32_t *status, uint64_t timeout_ns,
                                                      uint32_t seq, uint32_t role) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((n & 63u) == 0) {
            if (status_peek(status + 1) == seq) return false;
            if (globaltimer_ns() - t0 > timeout_ns) {
                const uint32_t word = uint32_t(TG_ERR_DEVICE_TIMEOUT) | (role << 8) |
                                      ((blockIdx.x & 0xffffu) << 16);
                atomicCAS(status, 0u, word);
                atomicExch(status + 1, seq);
                return false;
            }
        }
    }
}

// Cluster-scope wait that ignores other threads' failures (used once a launch is leaving,
// to collect what the peer CTA publishes): gives up after `limit_ns` and latches
// TG_ERR_DEVICE_TIMEOUT like any other wait.
static __device__ __noinline__ bool wait_cluster_exit(uint32_t bar, uint32_t parity,
                                                      const WaitCtl &ctl, uint32_t role,
                                                      uint64_t limit_ns) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((n & 63u) == 0 && globaltimer_ns() - t0 > limit_ns) {
            const uint32_t word = uint32_t(TG_ERR_DEVICE_TIMEOUT) | (role << 8) |
                                  ((blockIdx.x & 0xffffu) << 16);
            atomicCAS(ctl.status, 0u, word);
            atomicExch(ctl.status + 1, ctl.seq);
            return false;
        }
    }
}

// Bounded wait with cluster-scope acquire (see mbar_try_wait_cluster).
static __device__ __forceinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                            const WaitCtl &ctl, uint32_t role) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    return wait_slow_cluster(bar, parity, ctl.status, ctl.timeout_ns, ctl.seq, role);
}

// Waits until the phase with parity `parity` of `bar` has completed.  Returns false
// (and latches TG_ERR_DEVICE_TIMEOUT) after ctl.timeout_ns, or returns false as soon
// as another thread of the same launch has given up.  `obey_abort` = false ignores
// other threads' failures (used when draining copies that are already in flight).
static __device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                                    const WaitCtl &ctl, uint32_t role,
                                                    bool obey_abort = true) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, ctl.status, ctl.timeout_ns, ctl.seq, role, obey_abort);
}

// ----------------------------------------------------------------------------------
// TMA: tensor copies by coordinates (x = innermost, in elements)
// ----------------------------------------------------------------------------------
// Programmatic dependent launch: let the next kernel of the stream (launched with
// programmatic stream serialisation) be scheduled before this grid ends, and wait until
// the grids this one depends on have completed and their memory is visible.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

// Converged-warp form of tma_load_2d (see mbar_arrive_expect_tx).
__device__ __forceinline__ void tma_load_2d(uint32_t issue, uint32_t dst, const CUtensorMap *map,
                                            uint32_t bar, int32_t x, int32_t y) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "setp.ne.b32 e, %5, 0;\n\t"
        "@e cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(issue)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map,
                                                 uint32_t bar, int32_t x, int32_t y,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// Rank 1..5 load by coordinates c[0..rank-1] (c[0] innermost).
__device__ __forceinline__ void tma_load_nd(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            uint32_t rank, const int32_t (&c)[5]) {
    const uint64_t m = reinterpret_cast<uint64_t>(map);
    switch (rank) {
    case 1:
        asm volatile("cp.async.bulk.tensor.1d.shared::cluster.global.mbarrier::complete_tx::bytes"
                     " [%0], [%1, {%3}], [%2];" ::"r"(dst), "l"(m), "r"(bar), "r"(c[0])
                     : "memory");
        break;
    case 2:
        asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
                     " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst), "l"(m), "r"(bar), "r"(c[0]),
                     "r"(c[1])
                     : "memory");
        break;
    case 3:
        asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
                     " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst), "l"(m), "r"(bar), "r"(c[0]),
                     "r"(c[1]), "r"(c[2])
                     : "memory");
        break;
    case 4:
        asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
                     " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst), "l"(m), "r"(bar), "r"(c[0]),
                     "r"(c[1]), "r"(c[2]), "r"(c[3])
                     : "memory");
        break;
    default:
        asm volatile("cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
                     " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst), "l"(m), "r"(bar),
                     "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(c[4])
                     : "memory");
        break;
    }
}

// The box lands at offset `dst` of every CTA in `mask`, and each destination CTA's
// barrier at offset `bar` receives the transaction bytes of its copy.
__device__ __forceinline__ void tma_load_2d_multicast(uint32_t issue, uint32_t dst,
                                                      const CUtensorMap *map, uint32_t bar,
                                                      int32_t x, int32_t y, uint16_t mask) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "setp.ne.b32 e, %6, 0;\n\t"
        "@e cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".multicast::cluster [%0], [%1, {%3, %4}], [%2], %5;\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "h"(mask), "r"(issue)
        : "memory");
}

// CTA-pair form: the box lands in this CTA's shared memory at `dst`, and the
// transaction bytes are counted on the barrier at shared::cluster address `bar`, which
// may belong to the peer CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t issue, uint32_t dst, const CUtensorMap *map,
                                                 uint32_t bar, int32_t x, int32_t y) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "setp.ne.b32 e, %5, 0;\n\t"
        "@e cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(issue)
        : "memory");
}

// CTA-pair form with cluster multicast: the box lands at offset `dst` of every CTA in
// `mask`, and the bytes landing in each destination CTA are counted on the barrier at the
// same offset in that CTA's pair leader (the even rank of its pair); `bar` is the
// executing CTA's pair leader's barrier as a shared::cluster address.
__device__ __forceinline__ void tma_load_2d_pair_multicast(uint32_t issue, uint32_t dst,
                                                           const CUtensorMap *map, uint32_t bar,
                                                           int32_t x, int32_t y, uint16_t mask) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "setp.ne.b32 e, %6, 0;\n\t"
        "@e cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".multicast::cluster [%0], [%1, {%3, %4}], [%2], %5;\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "h"(mask), "r"(issue)
        : "memory");
}

// Tensor store of a rank 1..5 box from shared memory (bulk group; coordinates >= 0).
__device__ __forceinline__ void tma_store_nd(const CUtensorMap *map, uint32_t src, uint32_t rank,
                                             const int32_t (&c)[5]) {
    const uint64_t m = reinterpret_cast<uint64_t>(map);
    switch (rank) {
    case 1:
        asm volatile("cp.async.bulk.tensor.1d.global.shared::cta.bulk_group [%0, {%2}], [%1];" ::"l"(m),
                     "r"(src), "r"(c[0])
                     : "memory");
        break;
    case 2:
        asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                         m),
                     "r"(src), "r"(c[0]), "r"(c[1])
                     : "memory");
        break;
    case 3:
        asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                         m),
                     "r"(src), "r"(c[0]), "r"(c[1]), "r"(c[2])
                     : "memory");
        break;
    case 4:
        asm volatile(
            "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(m),
            "r"(src), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3])
            : "memory");
        break;
    default:
        asm volatile(
            "cp.async.bulk.tensor.5d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5, %6}], [%1];" ::"l"(
                m),
            "r"(src), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(c[4])
            : "memory");
        break;
    }
}

// Untiled bulk load global -> shared memory, counted on `bar` (addresses and size
// multiples of 16 bytes).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *gsrc, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst),
                 "l"(gsrc), "r"(bytes), "r"(bar)
                 : "memory");
}

// Converged-warp form of bulk_load: performed only by the lane whose `issue` is non-zero.
__device__ __forceinline__ void bulk_load(uint32_t issue, uint32_t dst, const void *gsrc,
                                          uint32_t bytes, uint32_t bar) {
    asm volatile("{\n\t.reg .pred e;\n\t"
                 "setp.ne.b32 e, %4, 0;\n\t"
                 "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}"
                 ::"r"(dst), "l"(gsrc), "r"(bytes), "r"(bar), "r"(issue)
                 : "memory");
}

// The GEMM's C tiles are written once and not read again by the launch: the store asks L2
// to evict them first, so that they do not push out A and B lines still to be reused
// (8192^3: 6 % less DRAM read; 16384 x 4096 x 1024, whose C is 128 MiB: 1731 -> 1760
// TFLOP/s).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int32_t x,
                                             int32_t y) {
    asm volatile("{\n\t.reg .b64 pol;\n\t"
                 "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
                 "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint"
                 " [%0, {%2, %3}], [%1], pol;\n\t}" ::"l"(reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(x), "r"(y)
                 : "memory");
}

// Untiled bulk copy shared -> global (16-byte aligned addresses, size multiple of 16).
__device__ __forceinline__ void bulk_store(void *gdst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(src), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until at most N bulk groups still read their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Waits until at most N bulk groups are incomplete (writes performed).
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later async-proxy
// (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------------------------
// tcgen05: tensor memory (TMEM) and the 5th-generation MMA
// ----------------------------------------------------------------------------------
// Whole-warp operations.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_alloc_permit() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes (64 bf16 along K), groups of 8 rows 1024 bytes
// apart.  `saddr` is the shared address of the first element the MMA reads; stepping
// K by 16 elements inside the 128-byte row adds 32 bytes to it.
__device__ __forceinline__ uint64_t umma_desc_kmajor_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= uint64_t((saddr & 0x3FFFFu) >> 4);  // bits  0-13: start address >> 4
    d |= uint64_t(1) << 16;                  // bits 16-29: leading offset (unused here)
    d |= uint64_t(1024u >> 4) << 32;         // bits 32-45: stride offset, 8 rows x 128 B
    d |= uint64_t(1) << 46;                  // bits 46-48: fixed 0b001
    d |= uint64_t(2) << 61;                  // bits 61-63: 128-byte swizzle
    return d;
}

// Shared-memory matrix descriptor of an MN-major operand tile written by TMA with the
// 128-byte swizzle: each 128-byte row holds 64 consecutive M (or N) elements of one k,
// groups of 8 k-rows are 1024 bytes apart, and the next 64 M (N) elements start `mn_stride`
// bytes further (the next TMA box).  Stepping K by 16 adds 2048 bytes (two 8-row groups).
__device__ __forceinline__ uint64_t umma_desc_mnmajor_sw128(uint32_t saddr, uint32_t mn_stride) {
    uint64_t d = 0;
    d |= uint64_t((saddr & 0x3FFFFu) >> 4);  // bits  0-13: start address >> 4
    d |= uint64_t(mn_stride >> 4) << 16;     // bits 16-29: leading offset: next 64 MN elements
    d |= uint64_t(1024u >> 4) << 32;         // bits 32-45: stride offset: next 8 k-rows
    d |= uint64_t(1) << 46;                  // bits 46-48: fixed 0b001
    d |= uint64_t(2) << 61;                  // bits 61-63: 128-byte swizzle
    return d;
}

// Instruction descriptor with an fp32 accumulator.  `in_kind` names the operand type:
// 0 bf16 and 1 fp16 (kind::f16, formats 1 and 0), 2 E4M3 and 3 E5M2 (kind::f8f6f4,
// formats 0 and 1), 4 tf32 (kind::tf32, format 2); A and B share it.  Bit 15 / bit 16
// select an MN-major A / B.
__host__ __device__ constexpr uint32_t umma_in_format(uint32_t in_kind) {
    return in_kind == 4u ? 2u : (in_kind == 0u || in_kind == 3u) ? 1u : 0u;
}

__host__ __device__ constexpr uint32_t umma_idesc_f32(uint32_t m, uint32_t n, uint32_t in_kind,
                                                      uint32_t a_mn, uint32_t b_mn) {
    return (1u << 4)                                         // D format: fp32
           | (umma_in_format(in_kind) << 7)                  // A format
           | (umma_in_format(in_kind) << 10)                 // B format
           | (a_mn << 15) | (b_mn << 16)                     // operand majors
           | ((n >> 3) << 17)                                // N / 8
           | ((m >> 4) << 24);                               // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]^T; `accumulate` = 0 overwrites.  The MMA and commit
// forms below are executed by a whole converged warp and performed only by the lane whose
// `issue` is non-zero: the warp never branches around them (a warp left with one active
// lane issued MMAs measurably more slowly).
__device__ __forceinline__ void umma_bf16(uint32_t issue, uint32_t d_tmem, uint64_t adesc,
                                   uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p, e;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "setp.ne.b32 e, %5, 0;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(issue)
                 : "memory");
}

// The same with 8-bit operands (kind::f8f6f4, K = 32 per instruction: 32 bytes, as for
// kind::f16 with K = 16).
__device__ __forceinline__ void umma_f8(uint32_t issue, uint32_t d_tmem, uint64_t adesc,
                                   uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p, e;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "setp.ne.b32 e, %5, 0;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(issue)
                 : "memory");
}

// tf32 operands (kind::tf32, K = 8 per instruction: again 32 bytes).
__device__ __forceinline__ void umma_tf32(uint32_t issue, uint32_t d_tmem, uint64_t adesc,
                                   uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p, e;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "setp.ne.b32 e, %5, 0;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(issue)
                 : "memory");
}

// Arrives once on `bar` when all tcgen05 MMAs previously issued by the issuing lane finish.
__device__ __forceinline__ void umma_commit(uint32_t issue, uint32_t bar) {
    asm volatile("{\n\t.reg .pred e;\n\t"
                 "setp.ne.b32 e, %1, 0;\n\t"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
                 ::"r"(bar), "r"(issue)
                 : "memory");
}

// Same, arriving on the barrier at offset `bar` of every CTA in `mask`.
__device__ __forceinline__ void umma_commit_multicast(uint32_t issue, uint32_t bar, uint16_t mask) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "setp.ne.b32 e, %2, 0;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;\n\t}" ::"r"(bar),
        "h"(mask), "r"(issue)
        : "memory");
}

// ---- MX block-scaled MMA (kind::mxf8f6f4 with E8M0 scales, one per 32 elements of K)
//
// Instruction descriptor of the block-scaled kinds: bits 4-5 = which byte of B's 32-bit
// scale word this MMA uses, 7-9 / 10-12 = A / B element format (0 = E4M3, 1 = E5M2), 15 /
// 16 = A / B MN-major, 17-22 = N / 8, 23 = scale type (1 = E8M0), 24-28 = M / 16, 29-30 =
// which byte of A's scale word.  The accumulator is fp32.
__host__ __device__ constexpr uint32_t umma_idesc_mx(uint32_t m, uint32_t n, uint32_t fmt,
                                                     uint32_t sf_id) {
    return (sf_id << 4)          // B scale byte
           | (fmt << 7)          // A format
           | (fmt << 10)         // B format
           | ((n >> 3) << 17)    // N / 8
           | (1u << 23)          // E8M0 scales
           | ((m >> 4) << 24)    // M / 16
           | (sf_id << 29);      // A scale byte
}

// Shared-memory descriptor of one 512-byte scale atom as tcgen05.cp's 32x128b source:
// 32 rows of 16 bytes, no swizzle, 8-row core matrices 128 bytes apart.
__device__ __forceinline__ uint64_t sf_atom_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= uint64_t((saddr & 0x3FFFFu) >> 4);  // bits  0-13: start address >> 4
    d |= uint64_t(16u >> 4) << 16;           // bits 16-29: leading offset (one 16-byte column)
    d |= uint64_t(128u >> 4) << 32;          // bits 32-45: stride offset, 8 rows x 16 B
    d |= uint64_t(1) << 46;                  // bits 46-48: fixed 0b001
    return d;                                // bits 61-63: 0 = no swizzle
}

// Copies a scale atom from shared memory into four TMEM columns starting at `taddr`: its
// 32 rows of 16 bytes land in lanes 0-31 and again in lanes 32-63, 64-95 and 96-127, so
// lane 32q + r, column c holds the four block scales of atom row r, quarter c.  Ordered
// with the issuing thread's later tcgen05.mma; completion is tracked by tcgen05.commit.
__device__ __forceinline__ void tmem_cp_sf_atom(uint32_t issue, uint32_t taddr, uint64_t sdesc) {
    asm volatile("{\n\t.reg .pred e;\n\t"
                 "setp.ne.b32 e, %2, 0;\n\t"
                 "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr),
                 "l"(sdesc), "r"(issue)
                 : "memory");
}

// D[tmem] (+)= (A * scales of A) * (B * scales of B), one 32-element block of K.
__device__ __forceinline__ void umma_mx(uint32_t issue, uint32_t d_tmem, uint64_t adesc,
                                        uint64_t bdesc, uint32_t idesc, uint32_t sfa_tmem,
                                        uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p, e;\n\t"
                 "setp.ne.b32 p, %6, 0;\n\t"
                 "setp.ne.b32 e, %7, 0;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
                 " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
                 "r"(accumulate), "r"(issue)
                 : "memory");
}

// ---- CTA-pair (cta_group::2) forms: one warp of each CTA of the pair allocates and
// releases the same TMEM columns; one thread of the leader CTA issues MMAs whose A rows
// and B columns are split across the two CTAs' shared memory and whose D rows land in
// both CTAs' TMEM. ----
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_alloc_permit_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void umma_bf16_pair(uint32_t issue, uint32_t d_tmem, uint64_t adesc,
                                   uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p, e;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "setp.ne.b32 e, %5, 0;\n\t"
                 "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(issue)
                 : "memory");
}

__device__ __forceinline__ void umma_f8_pair(uint32_t issue, uint32_t d_tmem, uint64_t adesc,
                                   uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p, e;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "setp.ne.b32 e, %5, 0;\n\t"
                 "@e tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(issue)
                 : "memory");
}

__device__ __forceinline__ void umma_tf32_pair(uint32_t issue, uint32_t d_tmem, uint64_t adesc,
                                   uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p, e;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "setp.ne.b32 e, %5, 0;\n\t"
                 "@e tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(issue)
                 : "memory");
}

// Pair forms of the scale copy and the block-scaled MMA, issued by the pair leader.  The
// copy moves the atom at shared-memory offset `sdesc` of each CTA of the pair into the
// same TMEM columns of that CTA; the MMA scales the D rows held by each CTA with that
// CTA's A-scale columns, and every column of D with the B-scale columns (all N of them,
// held in both CTAs).
__device__ __forceinline__ void tmem_cp_sf_atom_pair(uint32_t issue, uint32_t taddr,
                                                     uint64_t sdesc) {
    asm volatile("{\n\t.reg .pred e;\n\t"
                 "setp.ne.b32 e, %2, 0;\n\t"
                 "@e tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr),
                 "l"(sdesc), "r"(issue)
                 : "memory");
}

__device__ __forceinline__ void umma_mx_pair(uint32_t issue, uint32_t d_tmem, uint64_t adesc,
                                             uint64_t bdesc, uint32_t idesc, uint32_t sfa_tmem,
                                             uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p, e;\n\t"
                 "setp.ne.b32 p, %6, 0;\n\t"
                 "setp.ne.b32 e, %7, 0;\n\t"
                 "@e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
                 " [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
                 "r"(accumulate), "r"(issue)
                 : "memory");
}

// Arrives once on the barrier at offset `bar` of every CTA in `mask` when all earlier
// pair MMAs of this thread finish.
__device__ __forceinline__ void umma_commit_pair_multicast(uint32_t issue, uint32_t bar,
                                                           uint16_t mask) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "setp.ne.b32 e, %2, 0;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;\n\t}" ::"r"(bar),
        "h"(mask), "r"(issue)
        : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp receives lane
// (base lane + t), columns [col, col+32).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
        " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
        " [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

// Waits for this thread's outstanding tcgen05.ld; the registers pass through the asm
// statement so that no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]),
                   "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]),
                   "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// 32 lanes x 64 consecutive 32-bit columns in one instruction.
__device__ __forceinline__ void tmem_ld_32x32b_x64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
        " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31,"
        " %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47,"
        " %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63},"
        " [%64];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
          "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
          "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
          "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]),
          "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]),
          "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]),
          "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]),
          "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[64]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31]), "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]),
                   "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]),
                   "+r"(r[42]), "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]),
                   "+r"(r[48]), "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]),
                   "+r"(r[54]), "+r"(r[55]), "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]),
                   "+r"(r[60]), "+r"(r[61]), "+r"(r[62]), "+r"(r[63])
                 :
                 : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

}  // namespace tg
