// W4A4 GEMM on tensor-core-form operands (sm_103a): q4_0_x_q4_gemm_tc.
//
// Same product as q4_0_x_q4_gemm ("509 tokens a second of prompt: the
// Hadamard route ships", sections "Why prompts are a matrix-unit problem" and
// "The rotation"): per 32-block the exact integer dot product S of 4-bit
// activation codes and Q4_0 weight codes, scaled by both scales and
// accumulated in block order, acc = fma(fp32(d_w * d_x), S, acc), bit for bit.
//
// Here both operands arrive already in the byte form the FP8 tensor cores
// consume (each code v as the e4m3 byte of the integer v, exact for |v| <= 8):
// the weights repacked once offline, the activations written so by their
// quantizer.  One K = 32 MMA yields the block sum S itself, exact in fp32 (an
// integer of magnitude <= 2048), so the epilogue is the definition as written
// for every finite scale, subnormal products included.  The kernel is
// therefore a plain warp-specialised pipeline with no widening step:
//   warp 0      TMA producer: per 128-element K stage, a 128-row weight tile
//               and a token tile (128-byte rows, 128B-swizzled, consumed by
//               tcgen05.mma straight from shared memory), the weight scales
//               (128 rows x 4 blocks) and the token scales (4 blocks x tokens)
//   warp 1      TMEM allocator and MMA issuer: one K=32 MMA per block into one
//               of four 128-column TMEM slots; a commit per two blocks
//   warps 2..   epilogue (16 warps, four per TMEM lane quarter, each a
//               quarter of the tile's columns): tcgen05.ld each block's S, fold
//               the scales in with packed fp32 operations, store rows of y
// The MMA and the epilogue hand off two blocks per synchronization; measured
// on GB300, one block per hand-off (four buffers) is slower, as every hand-off
// puts all epilogue warps in step.  Every wait is bounded.

// epilogue warps per TMEM lane quarter
#ifndef H32_TC_EPI_PER_QUAD
#define H32_TC_EPI_PER_QUAD 4
#endif
// poll without sleeping: the waits here are short and on the critical path
#ifndef H32_WAIT_SLEEP
#define H32_WAIT_SLEEP 0
#endif

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "h32_common.cuh"
#include "h32_epilogue.cuh"

namespace h32 {
namespace {

__device__ uint32_t g_tc_status;

constexpr int kBM = 128;             // weight rows per tile (MMA M, TMEM lanes)
constexpr int kBNMax = 128;          // tokens per tile (MMA N)
constexpr int kStages = 5;           // 128-element K stages in flight
constexpr int kTileBytes = 16384;    // 128 rows x 128 bytes
constexpr int kScaleBytes = 2048;    // 4 blocks x 128 fp32
#ifndef H32_TC_GROUP
#define H32_TC_GROUP 2
#endif
constexpr int kGroup = H32_TC_GROUP;       // blocks per MMA -> epilogue hand-off
constexpr int kBufs = 4 / kGroup;          // hand-off buffers in TMEM (4 blocks of 128 columns)
constexpr int kTmemCols = 512;       // kBufs hand-off buffers x kGroup blocks x 128 columns
constexpr uint64_t kDrainPolls = 1ull << 22;

template <int EPQ>
struct TcCfg {
    static constexpr int kEpiWarps = 4 * EPQ;
    static constexpr int kThreads = (2 + kEpiWarps) * 32;
    static constexpr int kMaxChunks = (8 + EPQ - 1) / EPQ;  // 16-column chunks per warp
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kTileBytes;
    static constexpr int kOffSA = kOffB + kStages * kTileBytes;
    static constexpr int kOffSB = kOffSA + kStages * kScaleBytes;
    static constexpr int kOffBar = kOffSB + kStages * kScaleBytes;
    static constexpr int kOffMisc = kOffBar + 32 * 8;
    static constexpr int kBytes = kOffMisc + 16 * 4;
    static constexpr int kSmem = kBytes + 1024;
};

enum {
    kBarFull = 0,
    kBarEmpty = kBarFull + kStages,
    kBarSFull = kBarEmpty + kStages,
    kBarSEmpty = kBarSFull + kBufs,
    kBarDrain = kBarSEmpty + kBufs
};
enum { kMiscTmem = 0, kMiscAbort = 1 };

struct TcArgs {
    float *y;
    int32_t *bsum;
    int64_t ldy;
    int32_t M, N, nb, bn, chunks, total;
    uint64_t wait_limit;
};

__device__ __forceinline__ void record(uint32_t bits) { atomicOr(&g_tc_status, bits); }

__device__ __forceinline__ void set_abort(volatile int *misc) {
    misc[kMiscAbort] = 1;
    record(kStatusTimeout);
}

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t limit,
                                          volatile int *abort) {
    const bool ok = mbar_wait_bounded(bar, parity, limit, abort);
    return __all_sync(0xFFFFFFFFu, ok);
}

// K-major operand in 128B-swizzled 8-row x 128-byte atoms, as TMA writes it
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;            // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;    // 8-row group stride: 1024 bytes
    d |= static_cast<uint64_t>(1) << 46;            // descriptor version
    d |= static_cast<uint64_t>(2) << 61;            // swizzle: 128 bytes
    return d;
}

// one elected lane of the (converged) warp arrives on `bar`; no branch
__device__ __forceinline__ void elect_arrive(uint64_t *bar) {
    asm volatile(
        "{\n.reg .pred p;\n.reg .b64 st;\nelect.sync _|p, 0xffffffff;\n"
        "@p mbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(smem_u32(bar))
        : "memory");
}

struct TcTile {
    int n0, g0, rows, ncols;
};

__device__ __forceinline__ TcTile tc_tile(int t, const TcArgs &a) {
    TcTile ti;
    const int nt = t / a.chunks, ch = t - nt * a.chunks;
    ti.n0 = nt * kBM;
    ti.g0 = ch * a.bn;
    ti.rows = min(a.bn, a.M - ti.g0);
    ti.ncols = (ti.rows + 15) & ~15;
    return ti;
}

// The epilogue of one warp over all of its tiles, without block sums: ring
// positions of the shared-memory stages and TMEM buffers are carried as
// counters and phase bits, arrivals come from one elected lane.  Returns false
// when a wait gave up.
template <int EPQ>
__device__ __forceinline__ bool epilogue_tiles(const TcArgs &a, uint64_t *bars, const float *s_sa,
                                               const float *s_sb, uint32_t tmem, int warp, int lane,
                                               volatile int *abort_flag) {
    using C = TcCfg<EPQ>;
    const int ew = warp - 2;
    const int quad = warp & 3;                 // TMEM lanes 32 quad .. 32 quad + 31
    const int part = ew >> 2;                  // share of the columns
    const int row = quad * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const int nst = a.nb / 4;
    const uint64_t lim = a.wait_limit;
    uint32_t s = 0, sph = 0, gb = 0, gph = 0;
    for (int t = blockIdx.x; t < a.total; t += gridDim.x) {
        const TcTile ti = tc_tile(t, a);
        const int n16 = ti.ncols >> 4;
        const int base = n16 / EPQ, rem = n16 % EPQ;
        const int nch = base + (part < rem ? 1 : 0);
        const int c0 = 16 * (part * base + min(part, rem));
        const uint32_t tcol_base = tmem + lane_addr + c0;
        uint64_t acc[8 * C::kMaxChunks];
#pragma unroll
        for (int i = 0; i < 8 * C::kMaxChunks; ++i) acc[i] = 0ull;
        for (int st = 0; st < nst; ++st) {
            if (!warp_wait(&bars[kBarFull + s], sph, lim, abort_flag)) return false;
            const float4 dw4 = *reinterpret_cast<const float4 *>(s_sa + s * (kScaleBytes / 4) + 4 * row);
            const float dws[4] = {dw4.x, dw4.y, dw4.z, dw4.w};
            const float *sb = s_sb + s * (kScaleBytes / 4) + c0;   // [4 blocks][bn tokens]
#pragma unroll
            for (int j0 = 0; j0 < 4; j0 += kGroup) {
                if (!warp_wait(&bars[kBarSFull + gb], gph, lim, abort_flag)) return false;
                tc_fence_after();
                const uint32_t tcol0 = tcol_base + gb * (kGroup * 128);
                // each chunk of every block of the group under one TMEM wait;
                // every accumulator still takes the blocks in order
#pragma unroll
                for (int c = 0; c < C::kMaxChunks; ++c) {
                    if (c < nch) {
                        uint32_t v[kGroup][16];
#pragma unroll
                        for (int i = 0; i < kGroup; ++i) tmem_ld_x16(tcol0 + i * 128 + c * 16, v[i]);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < kGroup; ++i)
                            fold16(acc + 8 * c, dws[j0 + i], sb + (j0 + i) * a.bn + 16 * c, v[i]);
                    }
                }
                // the warp-wide wait above: every lane's TMEM reads of the buffer are done
                tc_fence_before();
                elect_arrive(&bars[kBarSEmpty + gb]);
                if (++gb == kBufs) {
                    gb = 0;
                    gph ^= 1;
                }
            }
            __syncwarp();
            elect_arrive(&bars[kBarEmpty + s]);
            if (++s == kStages) {
                s = 0;
                sph ^= 1;
            }
        }
        const int64_t n = ti.n0 + row;
        if (n < a.N) {
#pragma unroll
            for (int c = 0; c < C::kMaxChunks; ++c) {
                if (c < nch) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int col = c0 + c * 16 + 2 * q;
                        const uint64_t pr = acc[8 * c + q];
                        if (col < ti.rows)
                            a.y[(ti.g0 + col) * a.ldy + n] = __uint_as_float(static_cast<uint32_t>(pr));
                        if (col + 1 < ti.rows)
                            a.y[(ti.g0 + col + 1) * a.ldy + n] =
                                __uint_as_float(static_cast<uint32_t>(pr >> 32));
                    }
                }
            }
        }
    }
    return true;
}

template <int EPQ, bool kSums>
__global__ void __launch_bounds__(TcCfg<EPQ>::kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_sa,
                   const __grid_constant__ CUtensorMap map_sb, const TcArgs a) {
    using C = TcCfg<EPQ>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *s_a = smem + C::kOffA;
    uint8_t *s_b = smem + C::kOffB;
    float *s_sa = reinterpret_cast<float *>(smem + C::kOffSA);
    float *s_sb = reinterpret_cast<float *>(smem + C::kOffSB);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    volatile int *misc = reinterpret_cast<volatile int *>(smem + C::kOffMisc);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nst = a.nb / 4;
    const uint64_t lim = a.wait_limit;
    const uint32_t stage_tx = kTileBytes + a.bn * 128 + kScaleBytes + a.bn * 16;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&bars[kBarFull + i], 1);
            mbar_init(&bars[kBarEmpty + i], 1 + C::kEpiWarps);
        }
        for (int i = 0; i < kBufs; ++i) {
            mbar_init(&bars[kBarSFull + i], 1);
            mbar_init(&bars[kBarSEmpty + i], C::kEpiWarps);
        }
        mbar_init(&bars[kBarDrain], 1);
        misc[kMiscAbort] = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        __syncwarp();
        tmem_alloc(reinterpret_cast<uint32_t *>(const_cast<int *>(&misc[kMiscTmem])), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = static_cast<uint32_t>(misc[kMiscTmem]);
    volatile int *abort_flag = &misc[kMiscAbort];

    if (warp == 0) {
        // ------------------------------------------------------------ TMA
        if (lane == 0) {
            prefetch_tmap(&map_a);
            prefetch_tmap(&map_b);
            prefetch_tmap(&map_sa);
            prefetch_tmap(&map_sb);
            uint32_t ks = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < a.total && ok; t += gridDim.x) {
                const TcTile ti = tc_tile(t, a);
                for (int st = 0; st < nst; ++st, ++ks) {
                    const int s = ks % kStages;
                    if (!mbar_wait_bounded(&bars[kBarEmpty + s], ((ks / kStages) & 1) ^ 1, lim,
                                           abort_flag)) {
                        set_abort(misc);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars[kBarFull + s], stage_tx);
                    tma_load_2d(s_a + s * kTileBytes, &map_a, &bars[kBarFull + s], st * 128, ti.n0);
                    tma_load_2d(s_b + s * kTileBytes, &map_b, &bars[kBarFull + s], st * 128, ti.g0);
                    tma_load_2d(s_sa + s * (kScaleBytes / 4), &map_sa, &bars[kBarFull + s], st * 4,
                                ti.n0);
                    tma_load_2d(s_sb + s * (kScaleBytes / 4), &map_sb, &bars[kBarFull + s], ti.g0,
                                st * 4);
                }
            }
            if (!ok) {
                for (uint32_t k = (ks > kStages ? ks - kStages : 0); k < ks; ++k)
                    mbar_wait_bounded(&bars[kBarFull + k % kStages], (k / kStages) & 1, kDrainPolls,
                                      nullptr);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            uint32_t ks = 0, kg = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < a.total && ok; t += gridDim.x) {
                const TcTile ti = tc_tile(t, a);
                const uint32_t idesc = idesc_e4m3_f32(kBM, ti.ncols);
                for (int st = 0; st < nst && ok; ++st, ++ks) {
                    const int s = ks % kStages;
                    if (!mbar_wait_bounded(&bars[kBarFull + s], (ks / kStages) & 1, lim, abort_flag)) {
                        set_abort(misc);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t da = smem_desc_sw128(smem_u32(s_a + s * kTileBytes));
                    const uint64_t db = smem_desc_sw128(smem_u32(s_b + s * kTileBytes));
                    for (int j0 = 0; j0 < 4; j0 += kGroup, ++kg) {
                        const int gb = kg % kBufs;
                        if (!mbar_wait_bounded(&bars[kBarSEmpty + gb], ((kg / kBufs) & 1) ^ 1, lim,
                                               abort_flag)) {
                            set_abort(misc);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int i = 0; i < kGroup; ++i) {
                            // block j's 32 bytes start 32 j bytes into each 128-byte row
                            const uint64_t koff = (32 * (j0 + i)) >> 4;
                            mma_f8f6f4(tmem + (gb * kGroup + i) * 128, da + koff, db + koff, idesc,
                                       0);
                        }
                        mma_commit(&bars[kBarSFull + gb]);
                    }
                    if (!ok) break;
                    mma_commit(&bars[kBarEmpty + s]);
                }
            }
            mma_commit(&bars[kBarDrain]);
            mbar_wait_bounded(&bars[kBarDrain], 0, kDrainPolls, nullptr);
        }
    } else if constexpr (!kSums) {
        // ------------------------------------------------------- epilogue
        if (!epilogue_tiles<EPQ>(a, bars, s_sa, s_sb, tmem, warp, lane, abort_flag)) set_abort(misc);
    } else {
        // ------------------------------------ epilogue with block sums
        const int ew = warp - 2;
        const int quad = warp & 3;                 // TMEM lanes 32*quad .. +31
        const int part = ew >> 2;                  // share of the columns
        const int row = quad * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        uint32_t ks = 0, kg = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < a.total && ok; t += gridDim.x) {
            const TcTile ti = tc_tile(t, a);
            const int n16 = ti.ncols >> 4;
            const int base = n16 / EPQ, rem = n16 % EPQ;
            const int nch = base + (part < rem ? 1 : 0);
            const int c0 = 16 * (part * base + min(part, rem));
            uint64_t acc[8 * C::kMaxChunks];
#pragma unroll
            for (int i = 0; i < 8 * C::kMaxChunks; ++i) acc[i] = 0ull;
            for (int st = 0; st < nst && ok; ++st, ++ks) {
                const int s = ks % kStages;
                if (!warp_wait(&bars[kBarFull + s], (ks / kStages) & 1, lim, abort_flag)) {
                    set_abort(misc);
                    ok = false;
                    break;
                }
                const float *sa = s_sa + s * (kScaleBytes / 4);   // [128 rows][4 blocks]
                const float *sb = s_sb + s * (kScaleBytes / 4);   // [4 blocks][bn tokens]
                const float4 dw4 = *reinterpret_cast<const float4 *>(sa + 4 * row);
                const float dws[4] = {dw4.x, dw4.y, dw4.z, dw4.w};
#pragma unroll
                for (int j0 = 0; j0 < 4; j0 += kGroup, ++kg) {
                    const int gb = kg % kBufs;
                    if (!warp_wait(&bars[kBarSFull + gb], (kg / kBufs) & 1, lim, abort_flag)) {
                        set_abort(misc);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t tcol0 = tmem + lane_addr + gb * kGroup * 128 + c0;
#pragma unroll
                    for (int i = 0; i < kGroup; ++i) {
                        const int j = j0 + i;
                        const float dw = dws[j];
                        const float *dxj = sb + j * a.bn + c0;
                        const uint32_t tcol = tcol0 + i * 128;
#pragma unroll
                        for (int c = 0; c < C::kMaxChunks; ++c) {
                            if (c < nch) {
                                uint32_t v[16];
                                tmem_ld_x16(tcol + c * 16, v);
                                tmem_ld_wait();
                                fold16(acc + 8 * c, dw, dxj + 16 * c, v);
                                if constexpr (kSums) {
                                    const int n = ti.n0 + row;
                                    const int col0 = c0 + c * 16;
                                    const int64_t step = static_cast<int64_t>(a.N) * a.nb;
                                    int32_t *bp = a.bsum + (ti.g0 + col0) * step +
                                                  static_cast<int64_t>(n) * a.nb + st * 4 + j;
                                    const int lim_q = min(16, ti.rows - col0);
                                    if (n < a.N) {
#pragma unroll
                                        for (int q = 0; q < 16; ++q)
                                            if (q < lim_q)
                                                bp[q * step] =
                                                    __float2int_rn(__uint_as_float(v[q]));
                                    }
                                }
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[kBarSEmpty + gb]);
                }
                if (!ok) break;
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kBarEmpty + s]);
            }
            if (!ok) break;
            const int64_t n = ti.n0 + row;
            if (n < a.N) {
#pragma unroll
                for (int c = 0; c < C::kMaxChunks; ++c) {
                    if (c < nch) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const int col = c0 + c * 16 + 2 * q;
                            const uint64_t pr = acc[8 * c + q];
                            if (col < ti.rows)
                                a.y[(ti.g0 + col) * a.ldy + n] =
                                    __uint_as_float(static_cast<uint32_t>(pr));
                            if (col + 1 < ti.rows)
                                a.y[(ti.g0 + col + 1) * a.ldy + n] =
                                    __uint_as_float(static_cast<uint32_t>(pr >> 32));
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

h32_status make_map(CUtensorMap *map, CUtensorMapDataType type, int esize, const void *base,
                    uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                    uint32_t box_outer, bool swizzle) {
    auto enc = encoder();
    if (!enc) {
        note_error("cuTensorMapEncodeTiled is not available from the driver");
        return H32_ERR_CUDA;
    }
    (void)esize;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r =
        enc(map, type, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        note_error("cuTensorMapEncodeTiled rejected a tensor map of the tc GEMM");
        return H32_ERR_CUDA;
    }
    return H32_OK;
}

// tokens per tile: simulate the static round-robin schedule (as the Q4_0 GEMM)
int choose_bn_tc(int64_t M, int64_t N, int sms) {
    const int64_t nt = (N + kBM - 1) / kBM;
    int best = kBNMax;
    double best_cost = 1e300;
    for (int bn = kBNMax; bn >= 32; bn -= 16) {
        const int64_t chunks = (M + bn - 1) / bn;
        const int64_t tiles = nt * chunks;
        const int64_t grid = tiles < sms ? tiles : sms;
        double worst = 0.0;
        for (int64_t c = 0; c < grid; ++c) {
            double cost = 0.0;
            for (int64_t t = c; t < tiles; t += grid) {
                const int64_t ch = t % chunks;
                const int64_t rows = (ch == chunks - 1) ? M - ch * bn : bn;
                cost += ((rows + 15) / 16) * 16 + 24;
            }
            if (cost > worst) worst = cost;
        }
        if (worst < best_cost - 1e-9) {
            best_cost = worst;
            best = bn;
        }
    }
    return best;
}

template <int EPQ, bool kSums>
h32_status launch_tc(const CUtensorMap *maps, const TcArgs &a, int grid, cudaStream_t s) {
    using C = TcCfg<EPQ>;
    const cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<EPQ, kSums>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return launch_status(e);
    gemm_tc_kernel<EPQ, kSums><<<grid, C::kThreads, C::kSmem, s>>>(maps[0], maps[1], maps[2], maps[3],
                                                                     a);
    return launch_status(cudaGetLastError());
}

}  // namespace

h32_status tc_read_and_clear_status(cudaStream_t s) {
    uint32_t v = 0;
    const uint32_t z = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_tc_status, 4, 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return H32_ERR_CUDA;
    if (cudaMemcpyToSymbolAsync(g_tc_status, &z, 4, 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return H32_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return H32_ERR_CUDA;
    if (v & kStatusTimeout) return H32_ERR_TIMEOUT;
    if (v & kStatusGuard) return H32_ERR_DEVICE_GUARD;
    return H32_OK;
}

}  // namespace h32

extern "C" h32_status q4_0_x_q4_gemm_tc(const uint8_t *wp, const float *wsc, int64_t ldws,
                                        const uint8_t *xw, const float *xdt, int64_t ldxd,
                                        int64_t M, int64_t N, int64_t K, float *y, int64_t ldy,
                                        int32_t *block_sums, void *stream) {
    using namespace h32;
    if (M < 0 || N <= 0 || K <= 0 || (K % 128) != 0 || (N % 16) != 0 || ldy < N ||
        ldws < K / 32 || (ldws % 4) != 0 || ldxd < M || (ldxd % 4) != 0)
        return H32_ERR_INVALID_ARG;
    if (M == 0) return H32_OK;
    if (!wp || !wsc || !xw || !xdt || !y) return H32_ERR_INVALID_ARG;
    if (!aligned16(wp) || !aligned16(wsc) || !aligned16(xw) || !aligned16(xdt) || !aligned16(y) ||
        (block_sums && !aligned16(block_sums)) || (ldy % 4) != 0)
        return H32_ERR_ALIGNMENT;
    if (M > 0x7FFFFFFFll || N > 0x7FFFFFFFll || K > 0x7FFFFFFFll) return H32_ERR_INVALID_ARG;
    int sms = 0;
    H32_TRY(check_device(&sms));
    const int bn = choose_bn_tc(M, N, sms);
    CUtensorMap maps[4];
    H32_TRY(make_map(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, wp, K, N, K, 128, kBM, true));
    H32_TRY(make_map(&maps[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, xw, K, M, K, 128, bn, true));
    H32_TRY(make_map(&maps[2], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, wsc, ldws, N, ldws * 4, 4, kBM,
                     false));
    H32_TRY(make_map(&maps[3], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, xdt, ldxd, K / 32, ldxd * 4, bn, 4,
                     false));
    TcArgs a{};
    a.y = y;
    a.bsum = block_sums;
    a.ldy = ldy;
    a.M = static_cast<int32_t>(M);
    a.N = static_cast<int32_t>(N);
    a.nb = static_cast<int32_t>(K / 32);
    a.bn = bn;
    a.chunks = static_cast<int32_t>((M + bn - 1) / bn);
    const int64_t total = ((N + kBM - 1) / kBM) * a.chunks;
    if (total > 0x7FFFFFFFll) return H32_ERR_INVALID_ARG;
    a.total = static_cast<int32_t>(total);
    a.wait_limit = wait_limit();
    const int grid = static_cast<int>(total < sms ? total : sms);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return block_sums ? launch_tc<H32_TC_EPI_PER_QUAD, true>(maps, a, grid, s)
                      : launch_tc<H32_TC_EPI_PER_QUAD, false>(maps, a, grid, s);
}
