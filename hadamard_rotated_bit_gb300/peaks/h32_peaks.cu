// Microbenchmarks behind the roofline denominators of the h32 kernels on one
// GB300 (sm_103a).  Each prints one JSON line with its rate per SM per clock
// (clock64 cycles, one resident CTA per SM unless noted, every SM running):
//   fp32      scalar fma.f32, fma.f32x2, and mul.f32x2 + fma.f32x2 (the tc
//             GEMM epilogue's mix): fp32 lane operations per clock
//   mma_sync  mma.sync.m16n8k32 s8 (the legacy integer tensor path): MACs per clock
//   tcgen05   tcgen05.mma kind::f8f6f4 M=128, K=32, N=128 and 256, back to back:
//             MACs per clock; and the issue-to-commit latency of one MMA
//   tmem      tcgen05.ld 32x32b.x16 by 16 warps: TMEM bytes read per clock
//   lds       ld.shared.v4 with one address for the whole warp (a broadcast),
//             16 warps: clocks per instruction per SM
//   mbarrier  arrive on one warp -> observed by another: clocks per hop
//   quantizer_launch_floor  an empty kernel and a copy with the activation
//             quantizer's access pattern on its grid at the pp512 sizes
//             (512 x 5120 and 512 x 17408 bf16), L2 flushed before each launch
//   tma_read  bulk asynchronous copies (the TMA engine) of 16 KB chunks from a
//             buffer held in L2 (32 MB) and from one in HBM (2 GB) into a ring of
//             shared-memory stages, one thread a CTA, every SM: bytes per clock
//             per SM and the aggregate rate (the operand stream of the tc GEMM)
// Every wait is bounded; nothing here depends on another kernel or rank.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#define CK(x)                                                                          \
    do {                                                                               \
        cudaError_t e_ = (x);                                                          \
        if (e_ != cudaSuccess) {                                                       \
            printf("{\"error\": \"%s: %s\"}\n", #x, cudaGetErrorString(e_));           \
            exit(1);                                                                   \
        }                                                                              \
    } while (0)

__device__ volatile int g_err;

__device__ __forceinline__ uint32_t su32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm volatile("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm volatile("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ float fma1(float a, float b, float c) {
    float d;
    asm volatile("fma.rn.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n) : "memory");
}
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t par) {
    for (int i = 0; i < (1 << 22); ++i) {
        uint32_t ok;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            "selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(su32(b)), "r"(par)
            : "memory");
        if (ok) return true;
    }
    g_err = 1;
    return false;
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
    asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(su32(b))
                 : "memory");
}

// ---------------------------------------------------------------- fp32 pipe
template <int MODE>
__global__ void __launch_bounds__(512) k_fp32(int iters, float *out, long long *cyc) {
    const int tid = threadIdx.x;
    const float s = 1.0f + tid * 1e-7f;
    const uint64_t a2 = (static_cast<uint64_t>(__float_as_uint(1.0000001f)) << 32) |
                        __float_as_uint(0.9999999f);
    uint64_t acc[8];
    float accs[16];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        acc[i] = (static_cast<uint64_t>(__float_as_uint(s + i)) << 32) | __float_as_uint(s - i);
#pragma unroll
    for (int i = 0; i < 16; ++i) accs[i] = s + i;
    __syncthreads();
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
        if constexpr (MODE == 0) {
#pragma unroll
            for (int i = 0; i < 16; ++i) accs[i] = fma1(accs[i], 0.9999999f, 1e-7f);
        } else if constexpr (MODE == 1) {
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fma2(acc[i], a2, a2);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fma2(mul2(a2, acc[i ^ 1]), a2, acc[i]);
        }
    }
    const long long t1 = clock64();
    float r = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        r += __uint_as_float(static_cast<uint32_t>(acc[i])) +
             __uint_as_float(static_cast<uint32_t>(acc[i] >> 32));
#pragma unroll
    for (int i = 0; i < 16; ++i) r += accs[i];
    out[blockIdx.x * 512 + tid] = r;
    if (tid == 0) cyc[blockIdx.x] = t1 - t0;
}

// ---------------------------------------------------------------- mma.sync s8
__global__ void __launch_bounds__(256) k_mma_sync(int iters, int *out, long long *cyc) {
    const int tid = threadIdx.x;
    uint32_t a[4] = {0x01020304u + tid, 0x05060708u, 0x01010101u, 0x02020202u};
    uint32_t b[2] = {0x01010101u, 0x03030303u + tid};
    int c[4][4] = {};
    __syncthreads();
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                "{%8,%9}, {%0,%1,%2,%3};"
                : "+r"(c[k][0]), "+r"(c[k][1]), "+r"(c[k][2]), "+r"(c[k][3])
                : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
    }
    const long long t1 = clock64();
    int r = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) r += c[k][0] + c[k][1] + c[k][2] + c[k][3];
    out[blockIdx.x * 256 + tid] = r;
    if (tid == 0) cyc[blockIdx.x] = t1 - t0;
}

// ------------------------------------------ tcgen05 MMA, TMEM loads, LDS, mbarrier
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// MODE 0: MMA throughput (N given), batches of 32 MMAs per commit; 1: MMA latency;
// 2: TMEM loads; 3: broadcast ld.shared.v4; 4: mbarrier hops
template <int MODE, int N>
__global__ void __launch_bounds__(512, 1) k_sm(int iters, long long *cyc, uint32_t *sink) {
    extern __shared__ __align__(1024) uint8_t smr[];
    uint8_t *sm = smr + ((1024u - (su32(smr) & 1023u)) & 1023u);
    uint8_t *sA = sm, *sB = sm + 16384;                       // 16 KB + 32 KB operands
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + 49152);
    uint32_t *tb = reinterpret_cast<uint32_t *>(sm + 49152 + 64);
    float *sx = reinterpret_cast<float *>(sm + 49152 + 128);  // 512 floats
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < 49152 / 4; i += blockDim.x) reinterpret_cast<uint32_t *>(sm)[i] = 0;
    for (int i = tid; i < 512; i += blockDim.x) sx[i] = 1.0f + i;
    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                         su32(tb))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tm = *tb;
    uint32_t x = 0;
    long long dt = 0;
    if constexpr (MODE <= 1) {
        if (tid == 0) {
            const uint32_t idesc = (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | ((128u >> 4) << 24);
            const uint64_t da = desc_sw128(su32(sA)), db = desc_sw128(su32(sB));
            uint32_t ph = 0;
            const long long t0 = clock64();
            for (int it = 0; it < iters; ++it) {
                const int nb = MODE == 0 ? 32 : 1;
                for (int k = 0; k < nb; ++k)
                    asm volatile(
                        "{\n.reg .pred p;\nsetp.ne.b32 p, 0, 0;\n"
                        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(
                            tm + static_cast<uint32_t>((k & 1) * 256)),
                        "l"(da + ((32 * (k & 3)) >> 4)), "l"(db + ((32 * (k & 3)) >> 4)), "r"(idesc)
                        : "memory");
                asm volatile(
                    "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                        su32(&bar[0]))
                    : "memory");
                if (!mbar_wait(&bar[0], ph)) break;
                ph ^= 1;
            }
            dt = clock64() - t0;
        }
    } else if constexpr (MODE == 2) {
        // 16 warps, 4 per lane quarter, each two x16 loads (32 columns) per step
        const uint32_t la = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t c0 = (warp >> 2) * 32;
        const long long t0 = clock64();
        for (int it = 0; it < iters; ++it) {
            uint32_t r0[16], r1[16];
            const uint32_t buf = (it & 3) * 128;
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
                "%13,%14,%15}, [%16];"
                : "=r"(r0[0]), "=r"(r0[1]), "=r"(r0[2]), "=r"(r0[3]), "=r"(r0[4]), "=r"(r0[5]),
                  "=r"(r0[6]), "=r"(r0[7]), "=r"(r0[8]), "=r"(r0[9]), "=r"(r0[10]), "=r"(r0[11]),
                  "=r"(r0[12]), "=r"(r0[13]), "=r"(r0[14]), "=r"(r0[15])
                : "r"(tm + la + buf + c0));
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
                "%13,%14,%15}, [%16];"
                : "=r"(r1[0]), "=r"(r1[1]), "=r"(r1[2]), "=r"(r1[3]), "=r"(r1[4]), "=r"(r1[5]),
                  "=r"(r1[6]), "=r"(r1[7]), "=r"(r1[8]), "=r"(r1[9]), "=r"(r1[10]), "=r"(r1[11]),
                  "=r"(r1[12]), "=r"(r1[13]), "=r"(r1[14]), "=r"(r1[15])
                : "r"(tm + la + buf + c0 + 16));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            // consume one register of each load (static indices: no local-memory copy)
            x ^= r0[0] ^ r1[15];
        }
        dt = clock64() - t0;
    } else if constexpr (MODE == 3) {
        // 16 warps, each 8 broadcast 16-byte loads per step (one address per warp)
        const long long t0 = clock64();
        for (int it = 0; it < iters; ++it) {
            const float *p = sx + ((it * 32 + warp * 16) & 448);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint4 v = *reinterpret_cast<const uint4 *>(p + 4 * q);
                x ^= v.x;
            }
        }
        dt = clock64() - t0;
    } else {
        if (lane == 0 && warp < 2) {
            const long long t0 = clock64();
            for (int it = 0; it < iters; ++it) {
                const uint32_t ph = it & 1;
                if (warp == 0) {
                    mbar_arrive(&bar[1]);
                    if (!mbar_wait(&bar[2], ph)) break;
                } else {
                    if (!mbar_wait(&bar[1], ph)) break;
                    mbar_arrive(&bar[2]);
                }
            }
            dt = clock64() - t0;
        }
    }
    sink[blockIdx.x * 512 + tid] = x;
    if (tid == 0) cyc[blockIdx.x] = dt;
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tm) : "memory");
}

// ------------------------------------------------ TMA reads (L2 and HBM)
// One thread a CTA keeps kTmaStages bulk copies of 16 KB in flight; CTA b reads
// the chunks b, b + gridDim.x, ... of the buffer, wrapping at `span` bytes.
constexpr int kTmaStages = 8;
constexpr int kTmaChunk = 16384;
__global__ void __launch_bounds__(32, 1) k_tma(const uint8_t *src, long long span, int iters,
                                               long long *cyc) {
    extern __shared__ __align__(1024) uint8_t tsm[];
    __shared__ __align__(8) uint64_t bars[kTmaStages];
    if (threadIdx.x != 0) return;
    for (int s = 0; s < kTmaStages; ++s) mbar_init(&bars[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const long long nchunks = span / kTmaChunk;
    long long c = blockIdx.x;
    auto issue = [&](int s) {
        const uint8_t *g = src + (c % nchunks) * kTmaChunk;
        c += gridDim.x;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(&bars[s])),
                     "r"(kTmaChunk)
                     : "memory");
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                su32(tsm + s * kTmaChunk)),
            "l"(g), "r"(kTmaChunk), "r"(su32(&bars[s]))
            : "memory");
    };
    const long long t0 = clock64();
    for (int s = 0; s < kTmaStages; ++s) issue(s);
    for (int i = 0; i < iters; ++i)
        for (int s = 0; s < kTmaStages; ++s) {
            if (!mbar_wait(&bars[s], i & 1)) {
                // gave up (g_err is set): wait, bounded, for the copies still in flight
                for (int r = s; r < kTmaStages; ++r) mbar_wait(&bars[r], i & 1);
                for (int r = 0; r < s && i + 1 < iters; ++r) mbar_wait(&bars[r], (i + 1) & 1);
                return;
            }
            if (i + 1 < iters) issue(s);
        }
    cyc[blockIdx.x] = clock64() - t0;
}

// ---------------------------------------- launch floor of the pp512 quantizer sizes
__global__ void k_empty() {}

// the activation quantizer's access pattern without its arithmetic: a warp takes
// 4 rows x 8 blocks of 32 bf16 values, a thread loads its block (64 bytes) and
// stores 32 code bytes and one scale (block-major)
__global__ void __launch_bounds__(256) k_copy(const uint16_t *x, int M, int K, uint8_t *xw,
                                              float *xdt, int ldxd) {
    const int nb = K / 32, tiles_b = (nb + 7) / 8, ntiles = ((M + 3) / 4) * tiles_b;
    const int lane = threadIdx.x & 31, nwarps = gridDim.x * (blockDim.x >> 5);
    for (int wt = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); wt < ntiles; wt += nwarps) {
        const int tr = wt / tiles_b, tb = wt - tr * tiles_b;
        const int row = tr * 4 + (lane >> 3), b = tb * 8 + (lane & 7);
        if (row >= M || b >= nb) continue;
        const uint4 *p = reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(row) * K + 32 * b);
        const uint4 a = __ldg(p), c = __ldg(p + 1), d = __ldg(p + 2), e = __ldg(p + 3);
        uint4 *o = reinterpret_cast<uint4 *>(xw + static_cast<int64_t>(row) * K + 32 * b);
        o[0] = make_uint4(a.x ^ c.x, a.y ^ c.y, a.z ^ c.z, a.w ^ c.w);
        o[1] = make_uint4(d.x ^ e.x, d.y ^ e.y, d.z ^ e.z, d.w ^ e.w);
        xdt[static_cast<int64_t>(b) * ldxd + row] = __uint_as_float(a.x);
    }
}

static double mean_cycles(const long long *d, int n) {
    long long h[2048];
    CK(cudaMemcpy(h, d, n * sizeof(long long), cudaMemcpyDeviceToHost));
    double s = 0;
    for (int i = 0; i < n; ++i) s += static_cast<double>(h[i]);
    return s / n;
}

template <int MODE, int N>
static double run_sm(int sms, int threads, int iters, long long *cyc, uint32_t *sink) {
    // more than half of the shared memory of an SM: one CTA (one TMEM allocation) per SM
    const int smem = 120 * 1024;
    CK(cudaFuncSetAttribute(k_sm<MODE, N>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    for (int rep = 0; rep < 2; ++rep) {
        k_sm<MODE, N><<<sms, threads, smem>>>(iters, cyc, sink);
        CK(cudaGetLastError());
        CK(cudaDeviceSynchronize());
    }
    return mean_cycles(cyc, sms);
}

int main() {
    int dev = 0, sms = 0, clk = 0;
    CK(cudaGetDevice(&dev));
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    CK(cudaDeviceGetAttribute(&clk, cudaDevAttrClockRate, dev));
    float *fout;
    int *iout;
    long long *cyc;
    uint32_t *sink;
    // sized for the largest grid of each buffer's kernels: fp32 2 CTAs per SM x 512
    // threads, mma.sync 4 CTAs per SM x 256 threads, the others 1 CTA per SM x 512
    CK(cudaMalloc(&fout, sms * 2 * 512 * sizeof(float)));
    CK(cudaMalloc(&iout, sms * 4 * 256 * sizeof(int)));
    CK(cudaMalloc(&cyc, sms * 4 * sizeof(long long)));
    CK(cudaMalloc(&sink, sms * 512 * sizeof(uint32_t)));
    if (sms > 1024) {
        printf("{\"error\": \"more than 1024 SMs: host buffers too small\"}\n");
        return 1;
    }
    printf("{\"probe\": \"device\", \"sm_count\": %d, \"max_sm_clock_mhz\": %.0f}\n", sms, clk / 1e3);

    // fp32: two 512-thread CTAs per SM run at once
    const int it = 20000;
    const char *fp_names[3] = {"fma.rn.f32", "fma.rn.f32x2", "mul.rn.f32x2 + fma.rn.f32x2"};
    const double fp_ops[3] = {16, 16, 32};   // lane operations per thread per iteration
    for (int m = 0; m < 3; ++m) {
        for (int rep = 0; rep < 2; ++rep) {
            if (m == 0) k_fp32<0><<<sms * 2, 512>>>(it, fout, cyc);
            if (m == 1) k_fp32<1><<<sms * 2, 512>>>(it, fout, cyc);
            if (m == 2) k_fp32<2><<<sms * 2, 512>>>(it, fout, cyc);
            CK(cudaGetLastError());
            CK(cudaDeviceSynchronize());
        }
        const double c = mean_cycles(cyc, sms * 2);
        printf("{\"probe\": \"fp32\", \"instructions\": \"%s\", \"lane_ops_per_clock_per_sm\": %.1f}\n",
               fp_names[m], 2 * 512 * fp_ops[m] * it / c);
    }
    // mma.sync s8: four 256-thread CTAs per SM
    {
        const int iters = 4000;
        for (int rep = 0; rep < 2; ++rep) {
            k_mma_sync<<<sms * 4, 256>>>(iters, iout, cyc);
            CK(cudaGetLastError());
            CK(cudaDeviceSynchronize());
        }
        double hc = 0;
        long long h[4096];
        CK(cudaMemcpy(h, cyc, sms * 4 * sizeof(long long), cudaMemcpyDeviceToHost));
        for (int i = 0; i < sms * 4; ++i) hc += static_cast<double>(h[i]);
        hc /= sms * 4;
        // 8 warps x 4 MMAs of 16 x 8 x 32 MACs per iteration and CTA, 4 CTAs per SM
        printf("{\"probe\": \"mma_sync\", \"instructions\": \"mma.sync.m16n8k32 s8\", "
               "\"macs_per_clock_per_sm\": %.1f}\n",
               4.0 * 8 * 4 * 16 * 8 * 32 * iters / hc);
    }
    {
        const int iters = 200;
        const double c128 = run_sm<0, 128>(sms, 64, iters, cyc, sink) / (iters * 32.0);
        const double c256 = run_sm<0, 256>(sms, 64, iters, cyc, sink) / (iters * 32.0);
        const double lat = run_sm<1, 128>(sms, 64, 2000, cyc, sink) / 2000.0;
        printf("{\"probe\": \"tcgen05\", \"instructions\": \"tcgen05.mma kind::f8f6f4 e4m3\", "
               "\"macs_per_clock_per_sm_n128\": %.0f, \"macs_per_clock_per_sm_n256\": %.0f, "
               "\"clocks_per_mma_128x128x32\": %.1f, \"issue_to_commit_clocks\": %.0f}\n",
               128.0 * 128 * 32 / c128, 128.0 * 256 * 32 / c256, c128, lat);
    }
    {
        const int iters = 4000;
        const double c = run_sm<2, 128>(sms, 512, iters, cyc, sink) / iters;   // per 64 KB
        printf("{\"probe\": \"tmem\", \"instructions\": \"tcgen05.ld 32x32b.x16, 16 warps\", "
               "\"bytes_per_clock_per_sm\": %.0f, \"clocks_per_128x128_fp32_block\": %.1f}\n",
               65536.0 / c, c);
        const double l = run_sm<3, 128>(sms, 512, iters, cyc, sink) / iters;   // per 128 loads
        printf("{\"probe\": \"lds\", \"instructions\": \"ld.shared.v4 broadcast, 16 warps\", "
               "\"clocks_per_instruction_per_sm\": %.2f}\n", l / 128.0);
        const double b = run_sm<4, 128>(sms, 64, 20000, cyc, sink) / 20000.0;
        printf("{\"probe\": \"mbarrier\", \"clocks_per_hop\": %.0f}\n", b / 2.0);
    }
    // TMA reads: a 32 MB buffer (L2-resident after the first pass) and a 2 GB one
    {
        uint8_t *buf;
        const long long big = 2ll << 30, small = 32ll << 20;
        CK(cudaMalloc(&buf, big));
        CK(cudaMemset(buf, 1, big));
        CK(cudaFuncSetAttribute(k_tma, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kTmaStages * kTmaChunk));
        cudaEvent_t e0, e1;
        CK(cudaEventCreate(&e0));
        CK(cudaEventCreate(&e1));
        const long long spans[2] = {small, big};
        const char *names[2] = {"l2_32MB", "hbm_2GB"};
        for (int m = 0; m < 2; ++m) {
            // HBM: each CTA streams its share of the 2 GB once
            const int iters = m == 0 ? 400 : static_cast<int>(big / kTmaChunk / sms / kTmaStages);
            float ms = 0;
            for (int rep = 0; rep < 2; ++rep) {
                CK(cudaEventRecord(e0));
                k_tma<<<sms, 32, kTmaStages * kTmaChunk>>>(buf, spans[m], iters, cyc);
                CK(cudaGetLastError());
                CK(cudaEventRecord(e1));
                CK(cudaEventSynchronize(e1));
                CK(cudaEventElapsedTime(&ms, e0, e1));
            }
            const double bytes = static_cast<double>(sms) * iters * kTmaStages * kTmaChunk;
            const double c = mean_cycles(cyc, sms);
            printf("{\"probe\": \"tma_read\", \"source\": \"%s\", \"bytes_per_clock_per_sm\": %.1f, "
                   "\"aggregate_GBps\": %.0f}\n",
                   names[m], bytes / sms / c, bytes / (ms * 1e-3) / 1e9);
        }
        CK(cudaFree(buf));
    }
    // the quantizer's launch floor at the pp512 sizes: median of 25 launches, each
    // after a 256 MB write that flushes L2, on the grid the quantizer uses
    {
        uint8_t *flush;
        CK(cudaMalloc(&flush, 256u << 20));
        cudaEvent_t e0, e1;
        CK(cudaEventCreate(&e0));
        CK(cudaEventCreate(&e1));
        const int M = 512;
        const int Ks[2] = {5120, 17408};
        for (int ki = 0; ki < 2; ++ki) {
            const int K = Ks[ki], nb = K / 32;
            uint16_t *x;
            uint8_t *xw;
            float *xdt;
            CK(cudaMalloc(&x, static_cast<size_t>(M) * K * 2));
            CK(cudaMemset(x, 0x3c, static_cast<size_t>(M) * K * 2));
            CK(cudaMalloc(&xw, static_cast<size_t>(M) * K));
            CK(cudaMalloc(&xdt, static_cast<size_t>(nb) * M * 4));
            const int want = (M * nb + 255) / 256, grid = want < sms * 8 ? want : sms * 8;
            double med[2];
            for (int mode = 0; mode < 2; ++mode) {
                float t[25];
                for (int r = 0; r < 27; ++r) {
                    CK(cudaMemsetAsync(flush, r, 256u << 20));
                    CK(cudaEventRecord(e0));
                    if (mode == 0) k_empty<<<grid, 256>>>();
                    else k_copy<<<grid, 256>>>(x, M, K, xw, xdt, M);
                    CK(cudaGetLastError());
                    CK(cudaEventRecord(e1));
                    CK(cudaEventSynchronize(e1));
                    float ms;
                    CK(cudaEventElapsedTime(&ms, e0, e1));
                    if (r >= 2) t[r - 2] = ms;
                }
                for (int i = 1; i < 25; ++i)   // insertion sort of 25 values
                    for (int j = i; j > 0 && t[j] < t[j - 1]; --j) {
                        const float tmp = t[j];
                        t[j] = t[j - 1];
                        t[j - 1] = tmp;
                    }
                med[mode] = t[12] * 1e3;
            }
            printf("{\"probe\": \"quantizer_launch_floor\", \"shape\": \"512x%d bf16\", \"grid\": %d, "
                   "\"empty_kernel_us\": %.2f, \"same_pattern_copy_us\": %.2f}\n",
                   K, grid, med[0], med[1]);
            CK(cudaFree(x));
            CK(cudaFree(xw));
            CK(cudaFree(xdt));
        }
        CK(cudaFree(flush));
    }
    int err = 0;
    CK(cudaMemcpyFromSymbol(&err, g_err, sizeof(int)));
    printf("{\"probe\": \"status\", \"bounded_wait_gave_up\": %d}\n", err);
    CK(cudaFree(fout));
    CK(cudaFree(iout));
    CK(cudaFree(cyc));
    CK(cudaFree(sink));
    return err;
}
