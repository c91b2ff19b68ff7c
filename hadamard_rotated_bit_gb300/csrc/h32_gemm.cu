// Block-scaled integer GEMM of Q4_0 weights against 4-bit (or 8-bit)
// activation codes on the 5th-generation tensor cores (sm_103a).
//
// What it computes ("509 tokens a second of prompt: the Hadamard route
// ships", sections "Why prompts are a matrix-unit problem" and "The
// rotation"): for every output y[m][n] and every 32-block b along K, the
// exact integer dot product S = sum_j x_code * (w_code - 8) of the block's
// codes, scaled by both blocks' scales and accumulated in block order:
//     acc = fma(fp32(d_w * d_x), S, acc),  acc starting at +0.
// The result is bit-identical to that sequential fp32 evaluation.
//
// How it maps to GB300.  sm_103a has no integer tcgen05 MMA, so the exact
// integer products run on the FP8 path (tcgen05.mma kind::f8f6f4, fp32
// accumulators in tensor memory): every 4-bit code v in [-8, 8] is widened in
// shared memory to the e4m3 byte that encodes v * 2^-9 exactly (sign bit plus
// the magnitude in the low bits; 0..7 are subnormals, 8 is the smallest
// normal).  One MMA with K = 32 then produces S * 2^-18 exactly in fp32 (the
// products are small integers times 2^-18 and their sum stays far inside the
// accumulator's precision; checked bit-for-bit against integer sums).  The
// 2^18 is folded into the weight scale, so the epilogue still performs the
// same two roundings as the sequential definition.
//
// One CTA per SM, persistent over a static list of output tiles of 128 weight
// rows (the MMA's M side, TMEM lanes) x up to 128 tokens (the MMA's N side, a
// multiple of 16, so ragged expert groups only shrink N).  Warp roles:
//   warp 0      TMA producer: 128 x 64-byte tiles of weight nibbles
//   warp 1      TMEM allocator and MMA issuer (one thread)
//   warps 2-5   converters: widen weight nibbles (from TMA) and activation
//               codes (gathered from global by row index) to e4m3 operand
//               tiles in the canonical no-swizzle K-major layout; stage the
//               per-block scales
//   warps 6-13  epilogue: tcgen05.ld each block's S from TMEM, apply the
//               scales, accumulate in registers, store y with coalesced rows
// Every wait is bounded; a wait that gives up records a status bit, makes the
// other roles leave their loops, drains the CTA's own TMA copies and MMAs,
// frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <map>
#include <mutex>
#include <tuple>

#include "h32_common.cuh"
#include "h32_epilogue.cuh"

namespace h32 {
namespace {

__device__ uint32_t g_gemm_status;

constexpr int kBM = 128;                  // weight rows per tile
constexpr int kBNMax = 128;               // tokens per tile
constexpr int kStageBlocks = 4;           // 32-blocks per pipeline stage
constexpr int kNibStages = 4;             // TMA stages of weight nibbles
constexpr int kConvStages = 3;            // widened operand stages
constexpr int kMaxExperts = 1024;
constexpr int kTmemCols = 512;
constexpr uint64_t kDrainPolls = 1ull << 22;

// tuning constants (measured on GB300; see the design notes)
#ifndef H32_Q4_GROUP
#define H32_Q4_GROUP 1
#endif
#ifndef H32_Q4_EPI_PER_QUAD
#define H32_Q4_EPI_PER_QUAD 2
#endif
#ifndef H32_PIPE_TMEM_LOADS
#define H32_PIPE_TMEM_LOADS 0
#endif

constexpr int kWarpTma = 0, kWarpMma = 1, kWarpConv0 = 2, kNumConv = 4, kWarpEpi0 = 6;
constexpr int kConvThreads = kNumConv * 32;  // 128

constexpr int kNibBytes = kBM * 64;          // one stage of weight nibbles (8 KB)
// one widened operand stage: 16 row groups of 8 K-chunks of 16-byte core-matrix rows
constexpr int kOpBytes = (kBNMax / 8) * 1152;  // 18 KB
constexpr int kScaleBytes = kStageBlocks * kBNMax * 4;  // 2 KB

// The MMA's view of a widened operand tile: core matrix (row group g, K chunk
// c) at g * 1152 + c * 144.  The K-direction stride of 144 bytes (not 128)
// staggers the chunks by four banks, so the converters' 16-byte stores of
// eight rows x four blocks per warp phase hit 32 distinct banks.
constexpr uint32_t kLBO = 144, kSBO = 1152;
__device__ __forceinline__ uint32_t op_offset(int r, int chunk) {
    return (r >> 3) * kSBO + chunk * kLBO + (r & 7) * 16;
}

template <int XB>
struct Cfg {
    static constexpr int kBOps = (XB == 4) ? 1 : 2;      // B operands per stage (q8: hi, lo)
    static constexpr int kSCols = (XB == 4) ? 128 : 256; // TMEM columns per block
    // blocks handed from the MMA to the epilogue per synchronization, and the
    // number of such groups in flight in TMEM (512 columns in all)
    static constexpr int kGroup = (XB == 4) ? H32_Q4_GROUP : 1;
    static constexpr int kGroupBufs = kTmemCols / (kGroup * kSCols);
    static constexpr bool kPipeLoads = H32_PIPE_TMEM_LOADS;
    // epilogue warps per TMEM lane quadrant (each takes an even share of the
    // tile's 16-column chunks)
    static constexpr int kEpiPerQuad = (XB == 4) ? H32_Q4_EPI_PER_QUAD : 2;
    static constexpr int kEpiWarps = 4 * kEpiPerQuad;
    static constexpr int kMaxChunks = (8 + kEpiPerQuad - 1) / kEpiPerQuad;  // 16-column chunks
    static constexpr int kThreads = (kWarpEpi0 + kEpiWarps) * 32;
    // shared memory map (offsets from a 1024-aligned base)
    static constexpr int kOffNib = 0;
    static constexpr int kOffA = kOffNib + kNibStages * kNibBytes;
    static constexpr int kOffB = kOffA + kConvStages * kOpBytes;
    static constexpr int kOffDw = kOffB + kConvStages * kBOps * kOpBytes;
    static constexpr int kOffDx = kOffDw + kConvStages * kScaleBytes;
    static constexpr int kOffBar = kOffDx + kConvStages * kScaleBytes;
    static constexpr int kOffMisc = kOffBar + 32 * 8;
    static constexpr int kOffGrp = kOffMisc + 64 * 4;
    static constexpr int kBytes = kOffGrp + 2 * (kMaxExperts + 1) * 4;
    static constexpr int kSmem = kBytes + 1024;  // alignment slack
};

struct GemmArgs {
    const uint16_t *wd;         // [E*N][nb] fp16 bits
    const uint8_t *xq;          // [T][row bytes]
    const float *xd;            // [T][nb]
    const int32_t *row_idx;     // [R] or null
    const int32_t *expert_off;  // [E+1] or null (one group of R rows)
    float *y;                   // [R][ldy]
    int32_t *bsum;              // [R][N][nb] or null
    int64_t ldy;
    int64_t R, T;
    int32_t E, N, K, nb;
    int32_t bn;                 // tokens per tile (multiple of 16, <= 128)
    uint64_t wait_limit;
};

struct Tile {
    int e, n0, g0, rows, ncols;
};

// barrier slots
enum {
    kBarNibFull = 0,
    kBarNibEmpty = kBarNibFull + kNibStages,
    kBarConvFull = kBarNibEmpty + kNibStages,
    kBarConvEmpty = kBarConvFull + kConvStages,
    kBarSFull = kBarConvEmpty + kConvStages,
    kBarSEmpty = kBarSFull + 4,
    kBarDrain = kBarSEmpty + 4,
    kNumBars = kBarDrain + 1
};
// misc words
enum { kMiscTmem = 0, kMiscAbort = 1, kMiscTotal = 2, kMiscBad = 3, kMiscSlow = 8 };

__device__ __forceinline__ void record(uint32_t bits) { atomicOr(&g_gemm_status, bits); }

__device__ __forceinline__ void set_abort(volatile int *misc) {
    misc[kMiscAbort] = 1;
    record(kStatusTimeout);
}

__device__ __forceinline__ Tile decode_tile(int t, int E, const int *s_off, const int *s_tpre,
                                            int bn) {
    int lo = 0, hi = E;  // invariant: s_tpre[lo] <= t < s_tpre[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_tpre[mid] <= t) lo = mid;
        else hi = mid;
    }
    Tile ti;
    ti.e = lo;
    const int local = t - s_tpre[lo];
    const int cnt = s_off[lo + 1] - s_off[lo];
    const int chunks = (cnt + bn - 1) / bn;
    const int nt = local / chunks, ch = local - nt * chunks;
    ti.n0 = nt * kBM;
    ti.g0 = s_off[lo] + ch * bn;
    ti.rows = min(bn, cnt - ch * bn);
    ti.ncols = (ti.rows + 15) & ~15;
    return ti;
}

// prmt with sign replication: 0xFF in every byte whose top bit is set
__device__ __forceinline__ uint32_t byte_sign_mask(uint32_t x) {
    uint32_t r;
    asm("prmt.b32 %0, %1, 0, 0xBA98;" : "=r"(r) : "r"(x));
    return r;
}

// Four two's-complement nibble codes (one per byte, low nibble) -> four e4m3
// bytes of v * 2^-9 (sign-magnitude).  `m` marks the negative bytes.
__device__ __forceinline__ uint32_t smag4(uint32_t x, uint32_t m) {
    return (x & ~m) | ((0x90909090u - x) & m);
}

// 8 two's-complement nibbles -> lo (low nibbles) and hi (high nibbles) e4m3 words
__device__ __forceinline__ void widen8(uint32_t w, uint32_t &lo, uint32_t &hi) {
    lo = smag4(w & 0x0F0F0F0Fu, byte_sign_mask(w << 4));
    hi = smag4((w >> 4) & 0x0F0F0F0Fu, byte_sign_mask(w));
}

// four int8 codes q in [-127, 127] -> e4m3 words of h and l, q = 16 h + l,
// l in [-8, 7], h in [-8, 8] (both as v * 2^-9)
__device__ __forceinline__ void split_q8(uint32_t w, uint32_t &h, uint32_t &l) {
    l = smag4(w & 0x0F0F0F0Fu, byte_sign_mask(w << 4));
    const uint32_t h8 = (((w >> 4) & 0x0F0F0F0Fu) ^ 0x08080808u) + ((w >> 3) & 0x01010101u);
    const uint32_t t = h8 + 0x78787878u;  // top bit set where h >= 0
    const uint32_t m = byte_sign_mask(t);
    h = ((t ^ 0x80808080u) & m) | ((0x88888888u - h8) & ~m);
}

// the exact block sums of 16 columns (debug output)
__device__ __forceinline__ void store_sums(const GemmArgs &a, const Tile &ti, int row, int col0,
                                           int b, const uint32_t (&v)[16]) {
    const int64_t n = ti.n0 + row;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int col = col0 + i;
        if (col < ti.rows && n < a.N)
            a.bsum[((ti.g0 + col) * static_cast<int64_t>(a.N) + n) * a.nb + b] =
                __float2int_rn(__uint_as_float(v[i]) * 262144.0f);
    }
}

// activation items and weight-scale items of one stage, held in registers
// between their global loads and their use
template <int XB>
struct StageRegs {
    uint4 q[4][XB == 4 ? 1 : 2];
    float dx[4];
    uint32_t wd[4];
};

// Predicated global loads into registers the caller zeroed: a load that is
// switched off leaves the zero, and no instruction consumes the loaded value
// until it is used, so the loads of the next stage stay in flight.
__device__ __forceinline__ void ldg_pred(uint4 &v, const void *p, bool on) {
    asm volatile(
        "{\n.reg .pred q;\nsetp.ne.b32 q, %5, 0;\n"
        "@q ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];\n}\n"
        : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
        : "l"(p), "r"(static_cast<int>(on)));
}
__device__ __forceinline__ void ldg_pred(float &v, const float *p, bool on) {
    asm volatile(
        "{\n.reg .pred q;\nsetp.ne.b32 q, %2, 0;\n@q ld.global.nc.f32 %0, [%1];\n}\n"
        : "+f"(v)
        : "l"(p), "r"(static_cast<int>(on)));
}
__device__ __forceinline__ void ldg_pred_u16(uint32_t &v, const uint16_t *p, bool on) {
    asm volatile(
        "{\n.reg .pred q;\nsetp.ne.b32 q, %2, 0;\n@q ld.global.nc.u16 %0, [%1];\n}\n"
        : "+r"(v)
        : "l"(p), "r"(static_cast<int>(on)));
}

template <int XB>
__device__ __forceinline__ void load_stage(const GemmArgs &a, const Tile &ti, int st, int ct,
                                           StageRegs<XB> &R) {
    const int64_t xrow_bytes = (XB == 4) ? a.K / 2 : a.K;
    const int nb = a.nb;
    const int kb0 = st * kStageBlocks;
    const int nblk = min(kStageBlocks, nb - kb0);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = ct + k * kConvThreads;
        const int m = i >> 2, j = i & 3;
        bool valid = (m < ti.rows) && (j < nblk);
        int64_t tok = 0;
        if (valid) {
            const int64_t r = ti.g0 + m;
            tok = a.row_idx ? a.row_idx[r] : r;
            if (tok < 0 || tok >= a.T) {
                record(kStatusGuard);
                valid = false;
            }
        }
#pragma unroll
        for (int h = 0; h < (XB == 4 ? 1 : 2); ++h) R.q[k][h] = make_uint4(0, 0, 0, 0);
        R.dx[k] = 0.0f;
        const uint8_t *src = a.xq + tok * xrow_bytes + (kb0 + j) * (XB == 4 ? 16 : 32);
#pragma unroll
        for (int h = 0; h < (XB == 4 ? 1 : 2); ++h) ldg_pred(R.q[k][h], src + 16 * h, valid);
        ldg_pred(R.dx[k], a.xd + tok * nb + kb0 + j, valid);
    }
    const int wrow0 = ti.e * a.N + ti.n0;
    const int nvalid_w = min(kBM, a.N - ti.n0);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = ct + k * kConvThreads;
        const int r = i >> 2, j = i & 3;
        R.wd[k] = 0u;
        ldg_pred_u16(R.wd[k], a.wd + static_cast<int64_t>(wrow0 + r) * nb + kb0 + j,
                     r < nvalid_w && j < nblk);
    }
}

// Widen one stage: activation items from registers, weight nibbles from the
// TMA tile; stage the scales.  Returns false when a wait gave up.
template <int XB>
__device__ __forceinline__ bool convert_stage(const GemmArgs &a, const Tile &ti, int st, uint32_t ks,
                                              int ct, int lane, int cw, const StageRegs<XB> &R,
                                              uint8_t *s_nib, uint8_t *s_a, uint8_t *s_b,
                                              float *s_dw, float *s_dx, uint64_t *bars,
                                              volatile int *misc, uint64_t lim,
                                              volatile int *abort_flag) {
    constexpr int kBOps = Cfg<XB>::kBOps;
    const int cs = ks % kConvStages, ns = ks % kNibStages;
    const int kb0 = st * kStageBlocks;
    const int nblk = min(kStageBlocks, a.nb - kb0);
    if (!warp_wait(&bars[kBarConvEmpty + cs], ((ks / kConvStages) & 1) ^ 1, lim, abort_flag)) {
        set_abort(misc);
        return false;
    }
    uint8_t *bdst = s_b + cs * kBOps * kOpBytes;
    float *dx_dst = s_dx + cs * (kStageBlocks * kBNMax);
    bool slow = false;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = ct + k * kConvThreads;
        const int m = i >> 2, j = i & 3;
        if (m < ti.ncols) {
            if constexpr (XB == 4) {
                const uint4 q = R.q[k][0];
                uint32_t lo[4], hi[4];
                widen8(q.x, lo[0], hi[0]);
                widen8(q.y, lo[1], hi[1]);
                widen8(q.z, lo[2], hi[2]);
                widen8(q.w, lo[3], hi[3]);
                *reinterpret_cast<uint4 *>(bdst + op_offset(m, 2 * j)) =
                    make_uint4(lo[0], lo[1], lo[2], lo[3]);
                *reinterpret_cast<uint4 *>(bdst + op_offset(m, 2 * j + 1)) =
                    make_uint4(hi[0], hi[1], hi[2], hi[3]);
            } else {
                const uint4 q0 = R.q[k][0], q1 = R.q[k][1];
                const uint32_t w8[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                uint32_t h[8], l[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) split_q8(w8[u], h[u], l[u]);
                // elements 0..15 -> chunk 2j, 16..31 -> chunk 2j + 1
                *reinterpret_cast<uint4 *>(bdst + op_offset(m, 2 * j)) =
                    make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4 *>(bdst + op_offset(m, 2 * j + 1)) =
                    make_uint4(h[4], h[5], h[6], h[7]);
                *reinterpret_cast<uint4 *>(bdst + kOpBytes + op_offset(m, 2 * j)) =
                    make_uint4(l[0], l[1], l[2], l[3]);
                *reinterpret_cast<uint4 *>(bdst + kOpBytes + op_offset(m, 2 * j + 1)) =
                    make_uint4(l[4], l[5], l[6], l[7]);
            }
            const float dx = R.dx[k];
            const float adx = fabsf(dx);
            if (dx != 0.0f && !(adx >= 0x1p-100f && adx <= 0x1p90f)) slow = true;
            dx_dst[j * kBNMax + m] = dx;
        }
    }
    // weights (TMA tile): item -> row r = i / 4, block j = i % 4
    if (!warp_wait(&bars[kBarNibFull + ns], (ks / kNibStages) & 1, lim, abort_flag)) {
        set_abort(misc);
        return false;
    }
    uint8_t *adst = s_a + cs * kOpBytes;
    float *dw_dst = s_dw + cs * (kStageBlocks * kBNMax);
    const uint8_t *nib = s_nib + ns * kNibBytes;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = ct + k * kConvThreads;
        const int r = i >> 2, j = i & 3;
        const uint4 q = *reinterpret_cast<const uint4 *>(nib + r * 64 + j * 16);
        // Q4_0 code c means c - 8: flipping the top bit of each nibble gives
        // that value in two's complement
        uint32_t lo[4], hi[4];
        widen8(q.x ^ 0x88888888u, lo[0], hi[0]);
        widen8(q.y ^ 0x88888888u, lo[1], hi[1]);
        widen8(q.z ^ 0x88888888u, lo[2], hi[2]);
        widen8(q.w ^ 0x88888888u, lo[3], hi[3]);
        *reinterpret_cast<uint4 *>(adst + op_offset(r, 2 * j)) =
            make_uint4(lo[0], lo[1], lo[2], lo[3]);
        *reinterpret_cast<uint4 *>(adst + op_offset(r, 2 * j + 1)) =
            make_uint4(hi[0], hi[1], hi[2], hi[3]);
        const float dw = __half2float(__ushort_as_half(static_cast<unsigned short>(R.wd[k])));
        // fold in the 2^18 of the MMA's operand encoding (exact)
        dw_dst[j * kBNMax + r] = dw * 262144.0f;
    }
    // one arrival per warp: every lane's shared-memory reads and writes of
    // this stage are ordered before it by __syncwarp
    const unsigned any_slow = __any_sync(0xFFFFFFFFu, slow);
    fence_proxy_async_smem();  // this thread's operand writes -> tensor-core reads
    __syncwarp();
    if (lane == 0) {
        misc[kMiscSlow + cs * kNumConv + cw] = any_slow ? 1 : 0;
        mbar_arrive(&bars[kBarNibEmpty + ns]);
        mbar_arrive(&bars[kBarConvFull + cs]);
    }
    return true;
}

template <int XB, bool kSums>
__global__ void __launch_bounds__(Cfg<XB>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_w, const GemmArgs a) {
    using C = Cfg<XB>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // align by offsetting the __shared__ pointer itself (a round trip through
    // an integer would turn every shared access into a generic one)
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *s_nib = smem + C::kOffNib;
    uint8_t *s_a = smem + C::kOffA;
    uint8_t *s_b = smem + C::kOffB;
    float *s_dw = reinterpret_cast<float *>(smem + C::kOffDw);
    float *s_dx = reinterpret_cast<float *>(smem + C::kOffDx);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    volatile int *misc = reinterpret_cast<volatile int *>(smem + C::kOffMisc);
    int *s_off = reinterpret_cast<int *>(smem + C::kOffGrp);
    int *s_tpre = s_off + kMaxExperts + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool dense = (a.expert_off == nullptr);
    const int E = dense ? 1 : a.E;
    const int nt = (a.N + kBM - 1) / kBM;
    const int nb = a.nb;
    const int nst = (nb + kStageBlocks - 1) / kStageBlocks;
    const uint64_t lim = a.wait_limit;

    // ---------------------------------------------------------------- setup
    if (tid == 0) {
        for (int i = 0; i < kNibStages; ++i) {
            mbar_init(&bars[kBarNibFull + i], 1);
            mbar_init(&bars[kBarNibEmpty + i], kNumConv);
        }
        for (int i = 0; i < kConvStages; ++i) {
            mbar_init(&bars[kBarConvFull + i], kNumConv);
            mbar_init(&bars[kBarConvEmpty + i], 1 + C::kEpiWarps);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&bars[kBarSFull + i], 1);
            mbar_init(&bars[kBarSEmpty + i], C::kEpiWarps);
        }
        mbar_init(&bars[kBarDrain], 1);
        misc[kMiscAbort] = 0;
        misc[kMiscBad] = 0;
        fence_barrier_init();
    }
    if (dense) {
        if (tid == 0) {
            s_off[0] = 0;
            s_off[1] = static_cast<int>(a.R);
        }
    } else {
        for (int i = tid; i <= E; i += C::kThreads) s_off[i] = a.expert_off[i];
    }
    __syncthreads();
    if (!dense) {
        for (int i = tid; i <= E; i += C::kThreads) {
            const int v = s_off[i];
            bool bad = (i == 0 && v != 0) || (i == E && static_cast<int64_t>(v) != a.R) ||
                       (i < E && s_off[i + 1] < v);
            if (bad) misc[kMiscBad] = 1;
        }
    }
    // tiles per group, exclusive prefix (warp 0)
    if (warp == 0) {
        const int per = (E + 31) / 32;
        const int b0 = lane * per;
        int sum = 0;
        for (int i = 0; i < per; ++i) {
            const int e = b0 + i;
            if (e < E) {
                const int cnt = max(0, s_off[e + 1] - s_off[e]);
                sum += nt * ((cnt + a.bn - 1) / a.bn);
            }
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - sum;
        for (int i = 0; i < per; ++i) {
            const int e = b0 + i;
            if (e < E) {
                s_tpre[e] = run;
                const int cnt = max(0, s_off[e + 1] - s_off[e]);
                run += nt * ((cnt + a.bn - 1) / a.bn);
            }
        }
        if (lane == 31) {
            s_tpre[E] = incl;
            misc[kMiscTotal] = incl;
        }
    }
    __syncthreads();
    if (misc[kMiscBad]) {
        if (tid == 0 && blockIdx.x == 0) record(kStatusGuard);
        return;
    }
    const int total = misc[kMiscTotal];
    if (static_cast<int>(blockIdx.x) >= total) return;

    if (warp == kWarpMma) {
        __syncwarp();
        tmem_alloc(reinterpret_cast<uint32_t *>(const_cast<int *>(&misc[kMiscTmem])), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = static_cast<uint32_t>(misc[kMiscTmem]);
    volatile int *abort_flag = &misc[kMiscAbort];

    // ---------------------------------------------------------------- roles
    if (warp == kWarpTma) {
        if (lane == 0) {
            prefetch_tmap(&tmap_w);
            uint32_t ks = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile ti = decode_tile(t, E, s_off, s_tpre, a.bn);
                const int wrow0 = ti.e * a.N + ti.n0;
                for (int st = 0; st < nst; ++st, ++ks) {
                    const int slot = ks % kNibStages;
                    if (!mbar_wait_bounded(&bars[kBarNibEmpty + slot], ((ks / kNibStages) & 1) ^ 1,
                                           lim, abort_flag)) {
                        set_abort(misc);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars[kBarNibFull + slot], kNibBytes);
                    tma_load_2d(s_nib + slot * kNibBytes, &tmap_w, &bars[kBarNibFull + slot],
                                st * 64, wrow0);
                }
            }
            if (!ok) {  // drain this role's own copies before the CTA exits
                for (uint32_t k = (ks > kNibStages ? ks - kNibStages : 0); k < ks; ++k)
                    mbar_wait_bounded(&bars[kBarNibFull + k % kNibStages], (k / kNibStages) & 1,
                                      kDrainPolls, nullptr);
            }
        }
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            uint32_t ks = 0, kg = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const Tile ti = decode_tile(t, E, s_off, s_tpre, a.bn);
                const uint32_t idesc = idesc_e4m3_f32(kBM, ti.ncols);
                for (int st = 0; st < nst && ok; ++st, ++ks) {
                    const int cs = ks % kConvStages;
                    if (!mbar_wait_bounded(&bars[kBarConvFull + cs], (ks / kConvStages) & 1, lim,
                                           abort_flag)) {
                        set_abort(misc);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int nblk = min(kStageBlocks, nb - st * kStageBlocks);
                    const uint64_t a_desc0 =
                        smem_desc_noswizzle(smem_u32(s_a + cs * kOpBytes), kLBO, kSBO);
                    const uint64_t b_desc0 =
                        smem_desc_noswizzle(smem_u32(s_b + cs * C::kBOps * kOpBytes), kLBO, kSBO);
                    for (int j0 = 0; j0 < nblk; j0 += C::kGroup, ++kg) {
                        const int gb = kg % C::kGroupBufs;
                        if (!mbar_wait_bounded(&bars[kBarSEmpty + gb], ((kg / C::kGroupBufs) & 1) ^ 1, lim,
                                               abort_flag)) {
                            set_abort(misc);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
#pragma unroll
                        for (int i = 0; i < C::kGroup; ++i) {
                            const int j = j0 + i;
                            if (j < nblk) {
                                // block j's operands start 2 * j K-chunks into the tile
                                // (descriptor addresses are in 16-byte units)
                                const uint64_t koff = (2 * j * kLBO) >> 4;
                                const uint32_t d = tmem + (gb * C::kGroup + i) * C::kSCols;
                                mma_f8f6f4(d, a_desc0 + koff, b_desc0 + koff, idesc, 0);
                                if constexpr (XB == 8)
                                    mma_f8f6f4(d + 128, a_desc0 + koff,
                                               b_desc0 + koff + (kOpBytes >> 4), idesc, 0);
                            }
                        }
                        mma_commit(&bars[kBarSFull + gb]);
                    }
                    if (!ok) break;
                    mma_commit(&bars[kBarConvEmpty + cs]);
                }
            }
            // all MMAs of this CTA complete before tensor memory is released
            mma_commit(&bars[kBarDrain]);
            mbar_wait_bounded(&bars[kBarDrain], 0, kDrainPolls, nullptr);
        }
    } else if (warp < kWarpEpi0) {
        // ------------------------------------------------------ converters
        // Each thread owns four activation items (token m, block j) and four
        // weight items (row r, block j) per stage; the global loads of the
        // next stage are issued before the current stage is widened, so their
        // latency hides behind the widening work.
        const int ct = tid - kWarpConv0 * 32;  // 0..127
        const int cw = warp - kWarpConv0;
        uint32_t ks = 0;
        bool ok = true;
        int t = blockIdx.x, st = 0;
        Tile ti = decode_tile(t, E, s_off, s_tpre, a.bn);
        StageRegs<XB> R0, R1;
        load_stage<XB>(a, ti, st, ct, R0);
        auto step = [&](StageRegs<XB> &cur, StageRegs<XB> &nxt) {
            // where the next stage is
            int t2 = t, st2 = st + 1;
            Tile ti2 = ti;
            if (st2 == nst) {
                st2 = 0;
                t2 += gridDim.x;
                if (t2 < total) ti2 = decode_tile(t2, E, s_off, s_tpre, a.bn);
            }
            if (t2 < total) load_stage<XB>(a, ti2, st2, ct, nxt);
            ok = convert_stage<XB>(a, ti, st, ks, ct, lane, cw, cur, s_nib, s_a, s_b, s_dw, s_dx,
                                   bars, misc, lim, abort_flag);
            ++ks;
            t = t2;
            st = st2;
            ti = ti2;
        };
        while (t < total && ok) {
            step(R0, R1);
            if (t >= total || !ok) break;
            step(R1, R0);
        }
    } else {
        // -------------------------------------------------------- epilogue
        const int quad = warp & 3;                  // TMEM lanes 32*quad .. 32*quad+31
        const int part = (warp - kWarpEpi0) >> 2;   // which share of the columns
        const int row = quad * 32 + lane;           // weight row within the tile
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        uint32_t ks = 0, kg = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const Tile ti = decode_tile(t, E, s_off, s_tpre, a.bn);
            // the tile's 16-column chunks, split as evenly as possible
            const int n16 = ti.ncols >> 4;
            const int base = n16 / C::kEpiPerQuad, rem = n16 % C::kEpiPerQuad;
            const int nch = base + (part < rem ? 1 : 0);  // <= kMaxChunks
            const int c0 = 16 * (part * base + min(part, rem));
            uint64_t acc[8 * C::kMaxChunks];              // column pairs (fp32 x 2)
#pragma unroll
            for (int i = 0; i < 8 * C::kMaxChunks; ++i) acc[i] = 0ull;
            for (int st = 0; st < nst && ok; ++st, ++ks) {
                const int cs = ks % kConvStages;
                const int kb0 = st * kStageBlocks;
                const int nblk = min(kStageBlocks, nb - kb0);
                if (!warp_wait(&bars[kBarConvFull + cs], (ks / kConvStages) & 1, lim, abort_flag)) {
                    set_abort(misc);
                    ok = false;
                    break;
                }
                const bool slow = misc[kMiscSlow + cs * kNumConv + 0] |
                                  misc[kMiscSlow + cs * kNumConv + 1] |
                                  misc[kMiscSlow + cs * kNumConv + 2] |
                                  misc[kMiscSlow + cs * kNumConv + 3];
                const float *dxs = s_dx + cs * (kStageBlocks * kBNMax);
                const float *dws = s_dw + cs * (kStageBlocks * kBNMax);
                for (int j0 = 0; j0 < nblk; j0 += C::kGroup, ++kg) {
                    const int gb = kg % C::kGroupBufs;
                    if (!warp_wait(&bars[kBarSFull + gb], (kg / C::kGroupBufs) & 1, lim, abort_flag)) {
                        set_abort(misc);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int i = 0; i < C::kGroup; ++i) {
                        const int j = j0 + i;
                        if (j >= nblk) break;
                        const float dw = dws[j * kBNMax + row];
                        const float *dxj = dxs + j * kBNMax + c0;
                        const uint32_t tcol =
                            tmem + lane_addr + (gb * C::kGroup + i) * C::kSCols + c0;
                        if constexpr (XB == 4 && C::kPipeLoads) {
                            // software pipeline: the load of chunk c + 1 is in flight
                            // while chunk c is folded
                            uint32_t v0[16], v1[16];
                            if (nch > 0) tmem_ld_x16(tcol, v0);
#pragma unroll
                            for (int c = 0; c < C::kMaxChunks; ++c) {
                                if (c < nch) {
                                    tmem_ld_wait();
                                    uint32_t(&cur)[16] = (c & 1) ? v1 : v0;
                                    uint32_t(&nxt)[16] = (c & 1) ? v0 : v1;
                                    if (c + 1 < nch) tmem_ld_x16(tcol + (c + 1) * 16, nxt);
                                    if (!slow) fold16(acc + 8 * c, dw, dxj + 16 * c, cur);
                                    else fold16_exact(acc + 8 * c, dw, dxj + 16 * c, cur);
                                    if constexpr (kSums)
                                        store_sums(a, ti, row, c0 + c * 16, st * kStageBlocks + j, cur);
                                }
                            }
                        } else if constexpr (XB == 4) {
#pragma unroll
                            for (int c = 0; c < C::kMaxChunks; ++c) {
                                if (c < nch) {
                                    uint32_t v[16];
                                    tmem_ld_x16(tcol + c * 16, v);
                                    tmem_ld_wait();
                                    if (!slow) fold16(acc + 8 * c, dw, dxj + 16 * c, v);
                                    else fold16_exact(acc + 8 * c, dw, dxj + 16 * c, v);
                                    if constexpr (kSums)
                                        store_sums(a, ti, row, c0 + c * 16, st * kStageBlocks + j, v);
                                }
                            }
                        } else {
#pragma unroll
                            for (int c = 0; c < C::kMaxChunks; ++c) {
                                if (c < nch) {
                                    uint32_t v[16], u[16];
                                    tmem_ld_x16(tcol + c * 16, v);
                                    tmem_ld_x16(tcol + 128 + c * 16, u);
                                    tmem_ld_wait();
                                    // S = 16 S_h + S_l, exact in fp32
#pragma unroll
                                    for (int q = 0; q < 16; ++q)
                                        v[q] = __float_as_uint(__fmaf_rn(
                                            16.0f, __uint_as_float(v[q]), __uint_as_float(u[q])));
                                    if (!slow) fold16(acc + 8 * c, dw, dxj + 16 * c, v);
                                    else fold16_exact(acc + 8 * c, dw, dxj + 16 * c, v);
                                    if constexpr (kSums)
                                        store_sums(a, ti, row, c0 + c * 16, st * kStageBlocks + j, v);
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
                if (lane == 0) mbar_arrive(&bars[kBarConvEmpty + cs]);
            }
            if (!ok) break;
            // store: lanes hold 32 consecutive weight rows of one token column
            const int64_t n = ti.n0 + row;
            if (n < a.N) {
#pragma unroll
                for (int c = 0; c < C::kMaxChunks; ++c) {
                    if (c < nch) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int col = c0 + c * 16 + 2 * i;
                            const uint64_t pr = acc[8 * c + i];
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

    // ------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kWarpMma) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// 128 rows x 64 bytes boxes over the weight nibbles viewed as [rows][K/2] bytes
h32_status make_weight_map(CUtensorMap *map, const uint8_t *wq, int64_t rows, int64_t K) {
    auto enc = tensor_map_encoder();
    if (!enc) {
        note_error("cuTensorMapEncodeTiled is not available from the driver");
        return H32_ERR_CUDA;
    }
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
    const cuuint32_t box[2] = {64, kBM};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(wq), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        note_error("cuTensorMapEncodeTiled rejected the weight tensor map");
        return H32_ERR_CUDA;
    }
    return H32_OK;
}

// Tokens per tile for a dense product: simulate the static round-robin
// assignment of tiles to SMs and keep the width with the shortest makespan
// (a tile costs its 16-rounded width plus a fixed share for widening its
// weight tile).
int choose_bn_uncached(int64_t M, int64_t N, int sms) {
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
                cost += ((rows + 15) / 16) * 16 + 40;
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

// the simulation costs O(tiles) host time: remember each shape's width (a
// bounded table, emptied when full)
int choose_bn(int64_t M, int64_t N, int sms) {
    static std::mutex mu;
    static std::map<std::tuple<int64_t, int64_t, int>, int> widths;
    const auto key = std::make_tuple(M, N, sms);
    {
        std::lock_guard<std::mutex> lock(mu);
        const auto it = widths.find(key);
        if (it != widths.end()) return it->second;
    }
    const int bn = choose_bn_uncached(M, N, sms);
    std::lock_guard<std::mutex> lock(mu);
    if (widths.size() >= 4096) widths.clear();
    widths.emplace(key, bn);
    return bn;
}

template <int XB, bool kSums>
h32_status launch_variant(const CUtensorMap &map, const GemmArgs &a, int grid, cudaStream_t s) {
    using C = Cfg<XB>;
    const cudaError_t e = cudaFuncSetAttribute(
        gemm_kernel<XB, kSums>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return launch_status(e);
    gemm_kernel<XB, kSums><<<grid, C::kThreads, C::kSmem, s>>>(map, a);
    return launch_status(cudaGetLastError());
}

// the block-sum debug output is a separate compiled variant, so the product
// path carries no per-element check for it
template <int XB>
h32_status launch(const CUtensorMap &map, const GemmArgs &a, int grid, cudaStream_t s) {
    return a.bsum ? launch_variant<XB, true>(map, a, grid, s)
                  : launch_variant<XB, false>(map, a, grid, s);
}

template <int XB>
h32_status gemm_dense(const uint8_t *wq, const uint16_t *wd, const void *xq, const float *xd,
                      int64_t M, int64_t N, int64_t K, float *y, int64_t ldy, int32_t *bsum,
                      void *stream) {
    if (M < 0 || N <= 0 || K <= 0 || (K % 32) != 0 || (N % 16) != 0 || ldy < N)
        return H32_ERR_INVALID_ARG;
    if (M == 0) return H32_OK;
    if (!wq || !wd || !xq || !xd || !y) return H32_ERR_INVALID_ARG;
    if (!aligned16(wq) || !aligned16(wd) || !aligned16(xq) || !aligned16(xd) || !aligned16(y) ||
        (bsum && !aligned16(bsum)) || (ldy % 4) != 0)
        return H32_ERR_ALIGNMENT;
    if (M > 0x7FFFFFFFll || N > 0x7FFFFFFFll || K > 0x7FFFFFFFll) return H32_ERR_INVALID_ARG;
    int sms = 0;
    H32_TRY(check_device(&sms));
    CUtensorMap map;
    H32_TRY(make_weight_map(&map, wq, N, K));
    GemmArgs a{};
    a.wd = wd;
    a.xq = reinterpret_cast<const uint8_t *>(xq);
    a.xd = xd;
    a.row_idx = nullptr;
    a.expert_off = nullptr;
    a.y = y;
    a.bsum = bsum;
    a.ldy = ldy;
    a.R = M;
    a.T = M;
    a.E = 1;
    a.N = static_cast<int32_t>(N);
    a.K = static_cast<int32_t>(K);
    a.nb = static_cast<int32_t>(K / 32);
    a.bn = choose_bn(M, N, sms);
    a.wait_limit = wait_limit();
    const int64_t tiles = ((N + kBM - 1) / kBM) * ((M + a.bn - 1) / a.bn);
    if (tiles > 0x7FFFFFFFll) return H32_ERR_INVALID_ARG;
    const int grid = static_cast<int>(tiles < sms ? tiles : sms);
    return launch<XB>(map, a, grid, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

__device__ uint32_t g_gemm_status_taken;
__global__ void take_g_gemm_status() { g_gemm_status_taken = atomicExch(&g_gemm_status, 0u); }

h32_status gemm_read_and_clear_status(cudaStream_t s) {
    bool ok = false;
    const uint32_t v = take_status(take_g_gemm_status, g_gemm_status_taken, s, &ok);
    if (!ok) return H32_ERR_CUDA;
    if (v & kStatusTimeout) return H32_ERR_TIMEOUT;
    if (v & kStatusGuard) return H32_ERR_DEVICE_GUARD;
    return H32_OK;
}

}  // namespace h32

extern "C" h32_status q4_0_x_q4_gemm(const uint8_t *wq, const uint16_t *wd, const uint8_t *xq,
                                     const float *xd, int64_t M, int64_t N, int64_t K, float *y,
                                     int64_t ldy, int32_t *block_sums, void *stream) {
    return h32::gemm_dense<4>(wq, wd, xq, xd, M, N, K, y, ldy, block_sums, stream);
}

extern "C" h32_status q4_0_x_q8_gemm(const uint8_t *wq, const uint16_t *wd, const int8_t *xq,
                                     const float *xd, int64_t M, int64_t N, int64_t K, float *y,
                                     int64_t ldy, int32_t *block_sums, void *stream) {
    return h32::gemm_dense<8>(wq, wd, xq, xd, M, N, K, y, ldy, block_sums, stream);
}

extern "C" h32_status q4_0_x_q4_gemm_experts(const uint8_t *wq, const uint16_t *wd, int32_t E,
                                             const uint8_t *xq, const float *xd,
                                             const int32_t *row_idx, int64_t T,
                                             const int32_t *expert_off, int64_t R, int64_t N,
                                             int64_t K, float *y, int64_t ldy, int32_t *block_sums,
                                             void *stream) {
    using namespace h32;
    if (E < 1 || E > kMaxExperts || R < 0 || N <= 0 || K <= 0 || (K % 32) != 0 ||
        (N % 16) != 0 || ldy < N || T < 0)
        return H32_ERR_INVALID_ARG;
    if (!expert_off) return H32_ERR_INVALID_ARG;
    if (R == 0) return H32_OK;
    if (!wq || !wd || !xq || !xd || !y || T == 0) return H32_ERR_INVALID_ARG;
    if (!row_idx && T < R) return H32_ERR_INVALID_ARG;
    if (!aligned16(wq) || !aligned16(wd) || !aligned16(xq) || !aligned16(xd) || !aligned16(y) ||
        !aligned16(expert_off) || (row_idx && !aligned16(row_idx)) ||
        (block_sums && !aligned16(block_sums)) || (ldy % 4) != 0)
        return H32_ERR_ALIGNMENT;
    if (R > 0x7FFFFFFFll || static_cast<int64_t>(E) * N > 0x7FFFFFFFll || K > 0x7FFFFFFFll)
        return H32_ERR_INVALID_ARG;
    int sms = 0;
    H32_TRY(check_device(&sms));
    CUtensorMap map;
    H32_TRY(make_weight_map(&map, wq, static_cast<int64_t>(E) * N, K));
    GemmArgs a{};
    a.wd = wd;
    a.xq = xq;
    a.xd = xd;
    a.row_idx = row_idx;
    a.expert_off = expert_off;
    a.y = y;
    a.bsum = block_sums;
    a.ldy = ldy;
    a.R = R;
    a.T = T;
    a.E = E;
    a.N = static_cast<int32_t>(N);
    a.K = static_cast<int32_t>(K);
    a.nb = static_cast<int32_t>(K / 32);
    a.bn = kBNMax;
    a.wait_limit = wait_limit();
    // the tile count depends on the device-side offsets: launch one CTA per
    // SM, each walks the tile list it computes from expert_off
    const int64_t nt = (N + kBM - 1) / kBM;
    const int64_t bound = nt * (E + (R + kBNMax - 1) / kBNMax);
    // the kernel counts tiles in int (at most R / 128 + 2 E chunks per weight tile)
    if (nt * (R / kBNMax + 2 * static_cast<int64_t>(E) + 1) > 0x7FFFFFFFll)
        return H32_ERR_INVALID_ARG;
    const int grid = static_cast<int>(bound < sms ? bound : sms);
    return launch<4>(map, a, grid, reinterpret_cast<cudaStream_t>(stream));
}
