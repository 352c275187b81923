// dec_ptx.cuh -- PTX helpers shared by the decode kernels (mbarrier waits,
// TMA loads, legacy-path tensor-core MMA, cluster barriers, cp.async).
#pragma once

#include "wl_internal.cuh"

namespace wl {

// ------------------------------------------------------------------------
// PTX helpers: mbarrier, TMA, cluster, tensor cores, dependent launch
// ------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t *bar, unsigned parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_test_cluster(uint64_t *bar, unsigned parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded waits: false after kWaitLimitCycles (the status word is then set).
static __device__ __noinline__ bool mbar_wait(uint64_t *bar, unsigned parity, unsigned *status, unsigned site)
{
    if (mbar_test(bar, parity)) return true;
    const long long t0 = wait_clock();
    while (!mbar_test(bar, parity)) {
        if (wait_clock() - t0 > kWaitLimitCycles) {
            atomicOr(status, kStatusTimeout | site);
            return false;
        }
    }
    return true;
}

static __device__ __noinline__ bool mbar_wait_cluster(uint64_t *bar, unsigned parity, unsigned *status)
{
    if (mbar_test_cluster(bar, parity)) return true;
    const long long t0 = wait_clock();
    while (!mbar_test_cluster(bar, parity)) {
        if (wait_clock() - t0 > kWaitLimitCycles) {
            atomicOr(status, kStatusTimeout | kWaitExchange);
            return false;
        }
    }
    return true;
}

// Arrive on the mbarrier at the same shared-memory offset in CTA `rank` of
// this cluster, with release semantics at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint64_t *bar, unsigned rank)
{
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(bar)), "r"(rank));
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}

// One 2D tile of a tensor map into shared memory; c0 = column (inner), c1 =
// row.  Completion is counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// One box of a 3D tensor map (c0 innermost).
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t a[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
                 : "r"(addr));
}

// Shared-memory loads by shared address.  Data reached through a generic
// pointer into dynamic shared memory is loaded by generic loads, measured
// several times slower on the critical paths of these kernels.
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ float lds_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ float lds_bf16(uint32_t addr)
{
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return __uint_as_float((uint32_t)v << 16);
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t a[2], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(a[0]), "=r"(a[1]) : "r"(addr));
}

// D += A (16x16 bf16, row) * B (16x8 bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma_16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Cluster barrier split in two: every thread arrives once right after the
// barriers are initialised (the producer then never waits), and the consumer
// threads wait only before their first access to a peer CTA.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Barrier among the 256 consumer threads only (the producer never joins).
__device__ __forceinline__ void consumer_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Start copying nbytes (even) from global `src` into the shared buffer `dst`
// (16-byte aligned, nbytes + 16 bytes long) and return where src's first byte
// lands (dst + src % 16, so 16-byte alignment carries over).  The aligned body
// is copied with cp.async, the unaligned head and tail with 2-byte loads; no
// byte outside [src, src + nbytes) is read.  Finish with cp_async_wait_all()
// and a consumer barrier.
__device__ __forceinline__ const char *prefetch(char *dst, const void *src, int nbytes)
{
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(src);
    const uintptr_t s1 = s0 + (uintptr_t)nbytes;
    char *d = dst + (s0 & 15);
    uintptr_t b0 = (s0 + 15) & ~uintptr_t(15), b1 = s1 & ~uintptr_t(15);
    if (b1 <= b0) b0 = b1 = s1;  // no whole 16-byte chunk: all by elements
    for (uintptr_t c = b0 + 16 * threadIdx.x; c < b1; c += 16 * kThreads)
        cp_async16(d + (c - s0), reinterpret_cast<const void *>(c));
    const int nhead = (int)((b0 < s1 ? b0 : s1) - s0) >> 1;
    const int ntail = (int)(s1 - (b1 > s0 ? b1 : s0)) >> 1;
    const uint16_t *g = reinterpret_cast<const uint16_t *>(src);
    uint16_t *o = reinterpret_cast<uint16_t *>(d);
    const int tail0 = (int)((b1 > s0 ? b1 : s0) - s0) >> 1;
    for (int e = threadIdx.x; e < nhead; e += kThreads) o[e] = g[e];
    if (b1 > b0)
        for (int e = threadIdx.x; e < ntail; e += kThreads) o[tail0 + e] = g[tail0 + e];
    return d;
}

// Ring wait: a non-blocking test first (the stage is usually loaded long
// before its consumer reaches it), then the bounded wait.
__device__ __forceinline__ bool ring_wait(uint64_t *bar, unsigned parity, unsigned *status)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    return mbar_wait(bar, parity, status, kWaitRingFull);
}

__device__ __forceinline__ bool ring_wait_empty(uint64_t *bar, unsigned parity, unsigned *status)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    return mbar_wait(bar, parity, status, kWaitRingEmpty);
}

// A 2D tile copy addressed by a shared-memory offset (no address conversion
// per copy).
// Prefetch of a 2D box of `map` into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int c0, int c1)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void tma_load_2d_u32(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ float gelu_tanh_f32(float v)
{
    const float c = 0.7978845608028654f;  // sqrt(2/pi)
    return 0.5f * v * (1.0f + tanhf(c * (v + 0.044715f * v * v * v)));
}

}  // namespace wl
