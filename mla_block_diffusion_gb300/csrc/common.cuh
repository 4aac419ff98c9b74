// Device helpers shared by the DSpark kernels: inline PTX for mbarriers, TMA
// (cp.async.bulk.tensor), the 5th-generation tensor core (tcgen05 + TMEM), a
// bounded wait, and the error word. sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/dspark.h"

#define DS_DEVINL __device__ __forceinline__

namespace ds {

// Bounded waits give up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Error word (first int of the workspace). The first recorded error wins.
DS_DEVINL void set_error(int *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

DS_DEVINL unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

DS_DEVINL uint32_t smem_u32(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
DS_DEVINL void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
DS_DEVINL void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

DS_DEVINL void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
DS_DEVINL void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
DS_DEVINL bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
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

// Wait for the phase of the given parity to complete. Returns false (and raises
// *abort) once the wait has run longer than kWaitLimitNs, or if another role of
// the CTA has raised *abort already.
DS_DEVINL bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0) {
            if (*abort) return false;
            if (globaltimer() - t0 > kWaitLimitNs) {
                *abort = 1;
                return false;
            }
        }
    }
}

// Wait without the abort shortcut (drains copies after an abort), still bounded.
DS_DEVINL void mbar_drain(uint64_t *bar, uint32_t parity) {
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer() - t0 > kWaitLimitNs) break;
}

// ---------------------------------------------------------------------------
// TMA: 2D tiled bulk tensor load into shared memory, completing on an mbarrier.
// x is the innermost (contiguous) coordinate in elements, y the row.
// ---------------------------------------------------------------------------
DS_DEVINL void tma_prefetch_desc(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

DS_DEVINL void tma_load_2d(void *smem_dst, const CUtensorMap *m, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// 3D form: x innermost (elements), y the row, z the outer index.
DS_DEVINL void tma_load_3d(void *smem_dst, const CUtensorMap *m, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// Same, with an L2 cache-policy hint (used to mark streamed weights evict-first).
DS_DEVINL void tma_load_2d_hint(void *smem_dst, const CUtensorMap *m, int x, int y, uint64_t *bar,
                                uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

DS_DEVINL uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------------------
// tcgen05 / TMEM
// ---------------------------------------------------------------------------
DS_DEVINL void tmem_alloc(uint32_t *smem_slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
DS_DEVINL void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
DS_DEVINL void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DS_DEVINL void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand stored in the
// 128-byte-swizzled layout TMA writes (8 rows x 128 B atoms, atoms 1024 B apart).
DS_DEVINL uint64_t sdesc_k_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
    d |= (uint64_t)1 << 16;                    // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024u >> 4) << 32;         // stride byte offset: 8-row groups 1024 B apart
    d |= (uint64_t)1 << 46;                    // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;                    // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulator, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor for an MN-major operand in the 128-byte
// swizzled layout: rows of 128 bytes hold 64 consecutive MN elements of one k,
// 8 consecutive k rows form a 1024-byte atom; atoms repeat along k every
// sbo_bytes and along MN every lbo_bytes.
DS_DEVINL uint64_t sdesc_mn_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
// Instruction-descriptor bit that reads the B operand MN-major.
constexpr uint32_t kIdescBMajorMN = 1u << 16;

// Instruction descriptor, kind::f16: f16 A and B, fp32 accumulator, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

DS_DEVINL void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on an mbarrier once every previously issued tcgen05.mma of this thread completes.
DS_DEVINL void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 lanes x 16 columns of 32-bit accumulators: lane = thread, 16 consecutive columns.
DS_DEVINL void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// MMA with the A operand (M x K, 16-bit, two K elements per 32-bit cell, row = lane)
// taken from tensor memory.
DS_DEVINL void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 32 lanes x 32 columns of 32-bit cells from registers (lane = thread).
// 16 consecutive 32-bit columns of the warp's lane quadrant (one row per lane), raw.
DS_DEVINL void tmem_ld16u(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

DS_DEVINL void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
                 : "memory");
}
DS_DEVINL void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

DS_DEVINL void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

// Split form of tmem_ld16u for double buffering: the load is issued without a
// wait, and the wait names the destination registers so that no use of them
// can be scheduled above it.
DS_DEVINL void tmem_ld16_issue(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
DS_DEVINL void tmem_ld8_issue(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}
DS_DEVINL void tmem_ld_wait_tied(uint32_t (&r)[8]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7])
                 :
                 : "memory");
}
DS_DEVINL void tmem_ld_wait_tied(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15])
                 :
                 : "memory");
}

// Relaxed 64-bit store / load at GPU scope: a word that is its own payload
// (no other data is published with it).
DS_DEVINL void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
DS_DEVINL unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Bulk prefetch of bytes (16-byte aligned address, multiple of 16) into L2.
DS_DEVINL void prefetch_l2_bulk(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Up to two byte ranges (16-byte aligned starts, sizes multiples of 16) that a
// kernel pulls into L2 for the kernel that consumes them next: weights that do
// not depend on anything, streamed while this kernel leaves HBM idle.
struct L2Prefetch {
    const uint8_t *ptr[2];
    unsigned long long bytes[2];
};

// One thread per CTA: the CTA's share of the ranges, in 64 KB prefetches.
DS_DEVINL void l2_prefetch_range(const uint8_t *ptr, unsigned long long bytes, unsigned int cta, unsigned int ctas) {
    constexpr unsigned long long kChunk = 65536;
#pragma unroll 1
    for (unsigned long long off = (unsigned long long)cta * kChunk; off < bytes; off += (unsigned long long)ctas * kChunk)
        prefetch_l2_bulk(ptr + off, (uint32_t)(bytes - off < kChunk ? bytes - off : kChunk));
}
DS_DEVINL void l2_prefetch_share(const L2Prefetch &pf, unsigned int cta, unsigned int ctas) {
    l2_prefetch_range(pf.ptr[0], pf.bytes[0], cta, ctas);
    l2_prefetch_range(pf.ptr[1], pf.bytes[1], cta, ctas);
}

DS_DEVINL void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// AND of a predicate over the n threads arriving at named barrier id.
DS_DEVINL bool named_bar_and(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

DS_DEVINL float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue now; wait until the previous kernel's results are visible.
DS_DEVINL void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
DS_DEVINL void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch with programmatic stream serialization (overlaps this kernel's
// prologue with the tail of the previous kernel on the stream).
// Every kernel runs with the largest shared-memory carveout. An SM holds CTAs
// of several kernels at once only under one L1 / shared-memory split, and the
// weight GEMMs and the attention need the largest; a small kernel that let the
// driver pick a smaller split could not become resident beside them (and so
// could not start early under programmatic dependent launch). Set once per kernel.
inline void carveout_max(const void *kern) {
    static std::mutex mu;
    static const void *seen[128];
    static int n = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
        if (seen[i] == kern) return;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
        cudaSuccess)
        (void)cudaGetLastError();  // a hint: the launch proceeds without it
    if (n < 128) seen[n++] = kern;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args &&...args) {
    carveout_max((const void *)kern);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

DS_DEVINL unsigned long long ldcg_u64(const unsigned long long *p) { return __ldcg(p); }
DS_DEVINL int ld_volatile_i32(const int *p) { return *(const volatile int *)p; }
DS_DEVINL void st_volatile_i32(int *p, int v) { *(volatile int *)p = v; }

// Same, with thread-block clusters of cx CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                      int cx, Args &&...args) {
    carveout_max((const void *)kern);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cx;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------
// Thread-block clusters: rank, barrier (every CTA of a cluster is resident at
// once, so the barrier always completes), and loads from a peer's shared memory.
// ---------------------------------------------------------------------------
DS_DEVINL uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
DS_DEVINL void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Split cluster barrier without memory ordering (ordering comes from elsewhere):
// arrive early, wait before the CTA may stop being a target of its peers.
DS_DEVINL void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory"); }
DS_DEVINL void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// Asynchronous store of two floats into the same shared-memory location of CTA
// `rank`, counted as 8 transaction bytes on that CTA's mbarrier at local_bar.
DS_DEVINL void st_async_peer_f2(float2 *local_dst, uint64_t *local_bar, uint32_t rank, float2 v) {
    uint32_t a, b;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local_dst)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(b) : "r"(smem_u32(local_bar)), "r"(rank));
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(a),
                 "f"(v.x), "f"(v.y), "r"(b)
                 : "memory");
}

// Store into the same shared-memory location of CTA `rank` of the cluster
// (visible to it after the next cluster barrier).
DS_DEVINL void st_peer_f2(float2 *local, uint32_t rank, float2 v) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(v.x), "f"(v.y) : "memory");
}

// ---------------------------------------------------------------------------
// Split-K bookkeeping of the weight GEMMs: CTA c owns units [begin(c), begin(c+1))
// of the (tile, k-block) order; a tile is split over the CTAs whose ranges meet it.
// ---------------------------------------------------------------------------
__host__ __device__ inline long long gemm_unit_begin(int c, long long units, int grid) {
    return (long long)c * units / grid;
}

// CTA whose unit range contains unit u (ranges are non-empty: grid <= units).
__host__ __device__ inline int gemm_cta_of_unit(long long u, long long units, int grid) {
    int c = (int)((u * grid) / units);
    if (c >= grid) c = grid - 1;
    while (c + 1 < grid && gemm_unit_begin(c + 1, units, grid) <= u) ++c;
    while (c > 0 && gemm_unit_begin(c, units, grid) > u) --c;
    return c;
}

// A GEMM output left unreduced (pending): CTA c wrote the rows of its first tile
// in slot 2c and of its second tile in slot 2c + 1 (a pending GEMM gives every
// CTA at most one tile of units), row m of channel tile * 128 + r at
// part[(slot * BN + m) * 128 + r]. The output is the sum over the tile's CTAs in
// increasing order, so it does not depend on timing. part == nullptr: none.
// units * grid < 2^31 (32-bit bookkeeping).
struct GemmPending {
    const float *part;
    int units, grid, KB, BN;
};

// The CTAs of one tile: c_lo .. c_hi; c_lo wrote slot lo_slot, the others 2c.
struct PendTile {
    int c_lo, c_hi, lo_slot;
};

DS_DEVINL int pend_begin(const GemmPending &g, int c) {
    return (int)((unsigned)c * (unsigned)g.units / (unsigned)g.grid);
}
DS_DEVINL int pend_cta_of(const GemmPending &g, int u) {
    int c = (int)((unsigned)u * (unsigned)g.grid / (unsigned)g.units);
    if (c >= g.grid) c = g.grid - 1;
    while (c + 1 < g.grid && pend_begin(g, c + 1) <= u) ++c;
    while (c > 0 && pend_begin(g, c) > u) --c;
    return c;
}
DS_DEVINL PendTile pend_tile(const GemmPending &g, int t) {
    PendTile r;
    r.c_lo = pend_cta_of(g, t * g.KB);
    r.c_hi = pend_cta_of(g, (t + 1) * g.KB - 1);
    r.lo_slot = 2 * r.c_lo + (pend_begin(g, r.c_lo) < t * g.KB ? 1 : 0);
    return r;
}

// Channels r .. r + 3 (r a multiple of 4) of row m of a tile: contributors in
// batches of eight loads issued before any is added (the sum stays in CTA order).
constexpr int kPendBatch = 8;
template <int BATCH = kPendBatch>
DS_DEVINL float4 pending_sum4(const GemmPending &g, const PendTile &pt, int m, int r) {
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = pt.c_lo; c0 <= pt.c_hi; c0 += BATCH) {
        float4 v[BATCH];
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const int c = c0 + u;
            const int sl = c == pt.c_lo ? pt.lo_slot : 2 * c;
            v[u] = c <= pt.c_hi ? __ldcg((const float4 *)(g.part + ((size_t)sl * g.BN + m) * 128 + r))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            if (c0 + u <= pt.c_hi) {
                s.x += v[u].x;
                s.y += v[u].y;
                s.z += v[u].z;
                s.w += v[u].w;
            }
        }
    }
    return s;
}
// NP positions at once (channels r[j] .. r[j] + 3 of row m[j] of tile pt[j]): the
// first CMAX contributors of every position are loaded before any is added, so
// the positions share one round trip; contributors past CMAX follow in order.
// Each sum runs over its tile's CTAs in increasing order (as pending_sum4).
template <int NP, int CMAX>
DS_DEVINL void pending_sum4_multi(const GemmPending &g, const PendTile (&pt)[NP], const int (&m)[NP],
                                  const int (&r)[NP], const bool (&live)[NP], float4 (&out)[NP]) {
    float4 v[NP][CMAX];
#pragma unroll
    for (int j = 0; j < NP; ++j) {
#pragma unroll
        for (int u = 0; u < CMAX; ++u) {
            const int c = pt[j].c_lo + u;
            const int sl = u == 0 ? pt[j].lo_slot : 2 * c;
            v[j][u] = (live[j] && c <= pt[j].c_hi)
                          ? __ldcg((const float4 *)(g.part + ((size_t)sl * g.BN + m[j]) * 128 + r[j]))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
#pragma unroll
    for (int j = 0; j < NP; ++j) {
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < CMAX; ++u) {
            if (live[j] && pt[j].c_lo + u <= pt[j].c_hi) {
                s.x += v[j][u].x;
                s.y += v[j][u].y;
                s.z += v[j][u].z;
                s.w += v[j][u].w;
            }
        }
        for (int c = pt[j].c_lo + CMAX; live[j] && c <= pt[j].c_hi; ++c) {
            const float4 w = __ldcg((const float4 *)(g.part + ((size_t)(2 * c) * g.BN + m[j]) * 128 + r[j]));
            s.x += w.x;
            s.y += w.y;
            s.z += w.z;
            s.w += w.w;
        }
        out[j] = s;
    }
}

// Channel r of row m of a tile (same order).
DS_DEVINL float pending_sum1(const GemmPending &g, const PendTile &pt, int m, int r) {
    float s = 0.f;
    for (int c0 = pt.c_lo; c0 <= pt.c_hi; c0 += kPendBatch) {
        float v[kPendBatch];
#pragma unroll
        for (int u = 0; u < kPendBatch; ++u) {
            const int c = c0 + u;
            const int sl = c == pt.c_lo ? pt.lo_slot : 2 * c;
            v[u] = c <= pt.c_hi ? __ldcg(g.part + ((size_t)sl * g.BN + m) * 128 + r) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kPendBatch; ++u)
            if (c0 + u <= pt.c_hi) s += v[u];
    }
    return s;
}

}  // namespace ds
