// Shared host and device helpers of the h32 library (sm_103a only).
//
// Device side: bounded waits on mbarriers (a wait that gives up records a
// status bit instead of trapping), and thin inline-PTX wrappers for the
// Blackwell data movers and tensor-core instructions the GEMM uses
// (mbarrier, cp.async.bulk.tensor, tcgen05.*).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/h32.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ != 1030)
#error "h32 kernels are written for sm_103a only"
#endif

namespace h32 {

// status bits recorded by kernels
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusGuard = 2u;

// default bound on polling iterations of a spin wait (each poll backs off a
// little, so this is of the order of a second)
constexpr uint64_t kDefaultWaitPolls = 1ull << 22;

// host side -----------------------------------------------------------------
uint64_t wait_limit();                    // current bound (never 0)
h32_status check_device(int *sm_count);   // an sm_103 device is current
h32_status launch_status(cudaError_t e);  // map a CUDA error (and remember its text)
void note_error(const char *what);        // remember a non-CUDA failure text

// per-translation-unit status readers (each .cu file owns its status word)
h32_status quant_read_and_clear_status(cudaStream_t s);
h32_status gemm_read_and_clear_status(cudaStream_t s);
h32_status tc_read_and_clear_status(cudaStream_t s);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#if defined(__CUDACC__)
// launch `kernel` so that it may overlap the tail of the previous kernel of the
// stream (programmatic dependent launch; the kernel calls pdl_wait() first)
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}
#endif

#if defined(__CUDACC__)
// Read and clear a kernel status word in one atomic step: `take` is a
// one-thread kernel that swaps the word with 0 and leaves the old value in the
// device word `taken`, which is then copied out.  A bit that a kernel on
// another stream sets meanwhile is reported by this call or by the next one,
// never lost.  `*ok` is false when a launch, copy or synchronization failed.
// Not reentrant (one `taken` word per status word): h32_device_status
// serializes its callers.
template <typename T>
uint32_t take_status(void (*take)(), const T &taken, cudaStream_t s, bool *ok) {
    uint32_t v = 0;
    take<<<1, 1, 0, s>>>();
    *ok = cudaGetLastError() == cudaSuccess &&
          cudaMemcpyFromSymbolAsync(&v, taken, 4, 0, cudaMemcpyDeviceToHost, s) == cudaSuccess &&
          cudaStreamSynchronize(s) == cudaSuccess;
    return v;
}
#endif

#define H32_TRY(expr)                  \
    do {                               \
        h32_status _st = (expr);       \
        if (_st != H32_OK) return _st; \
    } while (0)

// device side ---------------------------------------------------------------
#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// programmatic dependent launch ---------------------------------------------
// A kernel launched with the programmatic-serialization attribute may start
// while the previous kernel of its stream is still finishing; it must not touch
// global memory (read or write) before pdl_wait(), which returns once that
// kernel has completed and its writes are visible.  pdl_trigger() lets the next
// kernel of the stream start early in the same way.  Both are no-ops for a
// kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// mbarrier ------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile(
        "{\n.reg .b64 st;\nmbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile(
        "{\n.reg .b64 st;\nmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(
            smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

// > 0: each try_wait may suspend the thread for up to this many ns while the
// phase is incomplete (it resumes as soon as the phase completes)
#ifndef H32_WAIT_HINT_NS
#define H32_WAIT_HINT_NS 0
#endif

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
#if H32_WAIT_HINT_NS > 0
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(static_cast<uint32_t>(H32_WAIT_HINT_NS))
        : "memory");
#else
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
#endif
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after
// `limit` polls, or as soon as *abort is set by another role of the CTA.
// Returns false when it gave up.
// 1: back off with a short sleep once a wait has polled 64 times
#ifndef H32_WAIT_SLEEP
#define H32_WAIT_SLEEP 1
#endif

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t limit,
                                                  volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    for (uint64_t i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort && *abort) return false;
#if H32_WAIT_SLEEP
        if (i > 64) __nanosleep(64);
#endif
    }
    return false;
}

// Every lane of a warp waits for a phase; the outcome is warp-uniform, so the
// warp-wide instructions after it (tcgen05.ld, votes) are reached by all lanes
// or none.  The common case, the phase already complete for every lane, costs
// one test and one vote (measured 2-3% faster on every pp512 shape of the
// tensor-core GEMM than entering the bounded loop first).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t limit,
                                          volatile int *abort) {
    uint32_t all;
    asm volatile(
        "{\n.reg .pred p, q;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "vote.sync.all.pred q, p, 0xffffffff;\nselp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(all)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (all) return true;
    const bool ok = mbar_wait_bounded(bar, parity, limit, abort);
    return __all_sync(0xFFFFFFFFu, ok);
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// make generic-proxy writes to shared memory visible to the async proxy
// (tensor-core operand reads, TMA)
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMA -----------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const void *tmap, uint64_t *bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// tcgen05 -------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (=|+=) A[smem desc] x B[smem desc]^T, kind::f8f6f4, issued by one thread
__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// arrive on an mbarrier once all previously issued tcgen05.mma of this thread complete
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 lanes x 32 bit, 16 consecutive columns per thread
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for tcgen05 (no swizzle, K-major canonical
// layout of 8-row x 16-byte core matrices).  lbo = byte distance between core
// matrices adjacent in K, sbo = byte distance between core matrices adjacent
// in M/N.
__device__ __forceinline__ uint64_t smem_desc_noswizzle(uint32_t saddr, uint32_t lbo,
                                                        uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo & 0x3FFFFu) >> 4) << 16;
    d |= static_cast<uint64_t>((sbo & 0x3FFFFu) >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // fixed constant 0b001 (descriptor version)
    // base offset 0, relative LBO mode, swizzle mode 0 (none)
    return d;
}

// Instruction descriptor: kind::f8f6f4, A = B = E4M3, D = F32, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(uint32_t M, uint32_t N) {
    return (1u << 4)            // D format: F32
           | (0u << 7)          // A format: E4M3
           | (0u << 10)         // B format: E4M3
           | ((N >> 3) << 17)   // N / 8
           | ((M >> 4) << 24);  // M / 16
}

// The same with A = E4M3 and B = E5M2 (kind::f8f6f4 takes any pair of its types)
__host__ __device__ constexpr uint32_t idesc_e4m3_e5m2_f32(uint32_t M, uint32_t N) {
    return idesc_e4m3_f32(M, N) | (1u << 10);   // B format: E5M2
}

#endif  // __CUDACC__

}  // namespace h32
