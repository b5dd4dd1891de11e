// Thin inline-PTX wrappers for sm_100-family asynchronous copies and
// barriers (bulk TMA copies, mbarriers, proxy fences), written from the PTX
// ISA.  Every wait is bounded: it gives up after a fixed number of polls,
// records a bit in the caller's error word and returns false, so no kernel
// can spin forever.
#pragma once

#include <stdint.h>

namespace kda {
namespace ptx {

// Bits of the per-context error word (read back by kda_sync_status).
constexpr int kErrDecodeLoadWait = 1 << 0;
constexpr int kErrPrefillWait = 1 << 1;
constexpr int kErrTestingWait = 1 << 2;
constexpr int kErrLowrankWait = 1 << 3;
constexpr int kErrProjWait = 1 << 4;

// Longest a kernel waits on one barrier phase before it reports an error.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // 1 s

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* m, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(m)), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* m, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_u32(m)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* m) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(m)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* m, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(m)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Bounded in wall
// time (limit_ns) and, when `abort` is given, cut short as soon as another
// thread of the CTA has set *abort.  Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait_timed(uint64_t* m, uint32_t parity, const int* abort = nullptr,
                                                unsigned long long limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(m, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (unsigned i = 1;; ++i) {
        if (mbar_try_wait(m, parity)) return true;
        if ((i & 63) == 0) {
            if (abort && *(volatile const int*)abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) return false;
        }
    }
}

// As mbar_wait_timed, recording `bit` in the error word when it gives up.
__device__ __forceinline__ bool mbar_wait(uint64_t* m, uint32_t parity, int* err, int bit) {
    if (mbar_wait_timed(m, parity)) return true;
    atomicOr(err, bit);
    return false;
}

// Programmatic dependent launch.  A kernel launched with the programmatic
// stream-serialisation attribute may start while the kernel before it in the
// stream is still running, once every CTA of that kernel has executed
// griddep_launch_dependents() (or exited); griddep_wait() returns once the
// kernel before has completed and its memory operations are visible.  In a
// kernel launched the ordinary way both are no-ops in effect (the kernel
// before has already completed).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Thread-block clusters.  The address, in the cluster's shared window, of
// the location at shared-memory address `saddr` of CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// Arrive on an mbarrier of another CTA of the cluster (release at cluster
// scope: this thread's earlier memory operations are visible to the CTA that
// waits on it).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// 16-byte and 4-byte stores into another CTA's shared memory (cluster
// addresses), each completing its bytes on an mbarrier of that CTA.
__device__ __forceinline__ void st_async_v4(uint32_t cluster_addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                            uint32_t cluster_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
                 ::"r"(cluster_addr), "r"(a), "r"(b), "r"(c), "r"(d), "r"(cluster_bar)
                 : "memory");
}

__device__ __forceinline__ void st_async_b32(uint32_t cluster_addr, uint32_t a, uint32_t cluster_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
                 ::"r"(cluster_addr), "r"(a), "r"(cluster_bar)
                 : "memory");
}

// Barrier over every thread of every CTA of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Bulk (non-tensor) TMA copy global -> this CTA's shared memory, completing
// `bytes` of transaction count on mbarrier m.  Addresses 16-byte aligned,
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* m) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(m))
        : "memory");
}

// Bulk TMA copy shared -> global, tracked by the bulk-group mechanism.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 ::"l"(dst), "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until every committed bulk store has finished READING shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until every committed bulk store has fully completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Tiled TMA load of a 4-D box (coordinates innermost first) into shared
// memory, completing its bytes on mbarrier m.  tmap is the address of a
// CUtensorMap kernel parameter (__grid_constant__).
__device__ __forceinline__ void tma_load_4d(void* dst, const void* tmap, int c0, int c1, int c2, int c3,
                                            uint64_t* m) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];"
        ::"r"(smem_u32(dst)), "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(m))
        : "memory");
}

// Tiled TMA load of a 2-D box (coordinates innermost first) into shared
// memory, completing its bytes on mbarrier m.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int c0, int c1, uint64_t* m) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(smem_u32(dst)), "l"(tmap), "r"(c0), "r"(c1), "r"(smem_u32(m))
        : "memory");
}

// Prefetch of a 4-D box into L2 (no shared memory, no completion to wait on).
__device__ __forceinline__ void tma_prefetch_4d(const void* tmap, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];"
                 ::"l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}

// Tiled TMA store of a 4-D box from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_4d(const void* tmap, int c0, int c1, int c2, int c3, const void* src) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];"
        ::"l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(src))
        : "memory");
}

// 16-byte asynchronous copy global -> shared (cp.async, L2 only); when !ok
// the destination is zero-filled and nothing is read.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool ok) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(ok ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace ptx
}  // namespace kda
