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
//   warps 2, 3  idle (with 16 epilogue warps: they complete the producers'
//               warpgroup, which hands its registers to the epilogue); the
//               widening warps in the widening instance (below)
//   the rest    epilogue (16 warps, four per TMEM lane quarter, each a
//               quarter of the tile's columns; or 12 warps, three per quarter):
//               tcgen05.ld each block's S, fold the scales in with packed fp32
//               operations, store rows of y
// The MMA and the epilogue hand off two blocks per synchronization; measured
// on GB300, one block per hand-off (four buffers) is slower, as every hand-off
// puts all epilogue warps in step.  Every wait is bounded.
//
// The widening instance (q4_0_x_q4_gemm_tc_widen[_experts]) takes the Q4_0
// planes themselves, half the weight bytes of the repacked form: TMA brings
// each stage's 128 x 64-byte tile of Q4_0 nibbles and the fp16 scales, and
// warps 2 and 3 spread the nibbles into bytes 0x0q of the 128B-swizzled tile
// the MMA reads (two masks and a shift per 8 codes).  Read as e4m3, 0x0q is
// exactly q * 2^-9 for every q = 0..15; the activations of this form are the
// e5m2 bytes of 512 times their codes (exact), so every product is the integer
// q x, and one more MMA per block against a constant tile of -8 * 2^-9 (e4m3
// 0x88) leaves S = sum (q - 8) x in the accumulator exactly as before.
//
// Schedule: one persistent CTA per SM takes tiles t = blockIdx.x, + gridDim.x,
// ...  The host simulates that assignment once per shape to choose the token
// width of a tile and, where it pays, a second kernel instance whose last
// partial wave of tiles is cut into narrower pieces, and (with a workspace) a
// third whose cut pieces also run in two parts along K on two CTAs, the second
// part continuing the first's accumulators (TcItem).  Kernels are launched with
// programmatic dependent launch: nothing touches global memory before the
// previous kernel of the stream has completed.

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

#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>

#include "h32_common.cuh"
#include "h32_epilogue.cuh"
#include "h32_tcform.cuh"

namespace h32 {
namespace {

__device__ uint32_t g_tc_status;

constexpr int kBM = 128;             // weight rows per tile (MMA M, TMEM lanes)
constexpr int kBNMax = 128;          // tokens per tile (MMA N)
constexpr int kMaxStages = 5;        // 128-element K stages in flight (at most)
constexpr int kTileBytes = 16384;    // 128 rows x 128 bytes
constexpr int kNibBytes = 8192;      // widening instance: 128 rows x 64 bytes of Q4_0 nibbles
constexpr int kWidenWarps = 2;       // widening instance: warps 2 and 3
constexpr int kScaleBytes = 2048;    // 4 blocks x 128 fp32
#ifndef H32_TC_GROUP
#define H32_TC_GROUP 2
#endif
constexpr int kGroup = H32_TC_GROUP;       // blocks per MMA -> epilogue hand-off
constexpr int kBufs = 4 / kGroup;          // hand-off buffers in TMEM (4 blocks of 128 columns)
constexpr int kTmemCols = 512;       // kBufs hand-off buffers x kGroup blocks x 128 columns
constexpr uint64_t kDrainPolls = 1ull << 22;
constexpr int kMaxExperts = 1024;
constexpr int kSplitMaxP = 128;      // pieces of a K split (flags in the workspace)

// XB = 4: one activation byte per code.  XB = 8: two bytes per code, the e4m3
// bytes of 16 h and of l where the 8-bit code is 16 h + l (0 <= l <= 15), so a
// 128-element stage carries two activation tiles.
// QN: the instance that also quantizes its output for the next projection; it
// gives up a stage for a 4 KB staging tile per epilogue warp.
// WQ: the widening instance (Q4_0 nibbles and fp16 scales in, widened in
// shared memory); a stage also holds the nibble tile, and a constant tile of
// -8 * 2^-9 follows the stages.
template <int EPQ, int XB, bool QN = false, bool WQ = false>
struct TcCfg {
    static_assert(!WQ || (EPQ == 4 && XB == 4 && !QN), "widening: 4-bit route, 16 epilogue warps");
    static constexpr int kStages = (XB == 8 || QN || WQ) ? 4 : 5;
    static constexpr int kBTile = XB == 8 ? 2 * kTileBytes : kTileBytes;   // activations per stage
    static constexpr int kEpiWarps = 4 * EPQ;
    // With 16 epilogue warps the producers form a warpgroup of their own (TMA,
    // MMA and two idle warps) that hands registers to the epilogue
    // (setmaxnreg): 96 a thread at launch, then 32 for the producer warpgroup
    // and 112 for the epilogue, 4 x 32 x 32 + 16 x 32 x 112 = 640 x 96.
    static constexpr bool kRegSplit = EPQ == 4;
    static constexpr int kProdWarps = kRegSplit ? 4 : 2;
    static constexpr int kThreads = (kProdWarps + kEpiWarps) * 32;
    static constexpr int kLaunchRegs = 96, kProdRegs = 32, kEpiRegs = 112;
    static_assert(!kRegSplit || (kProdWarps * kProdRegs + kEpiWarps * kEpiRegs) * 32 <=
                                    kThreads * kLaunchRegs,
                  "register split above the launch's registers");
    static constexpr int kMaxChunks = (8 + EPQ - 1) / EPQ;  // 16-column chunks per warp
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStages * kTileBytes;
    static constexpr int kOffN = kOffB + kStages * kBTile;                  // WQ: nibble tiles
    static constexpr int kOffC = kOffN + (WQ ? kStages * kNibBytes : 0);    // WQ: the -8 tile
    static constexpr int kOffSA = kOffC + (WQ ? kTileBytes : 0);
    static constexpr int kOffSB = kOffSA + kStages * kScaleBytes;
    static constexpr int kOffBar = kOffSB + kStages * kScaleBytes;
    static constexpr int kOffMisc = kOffBar + 32 * 8;
    static constexpr int kOffGrp = kOffMisc + 16 * 4;            // row offsets, tile prefix
    static constexpr int kOffQ = (kOffGrp + 2 * (kMaxExperts + 1) * 4 + 127) & ~127;
    static constexpr int kBytes = kOffQ + (QN ? kEpiWarps * 4096 : 0);
    static constexpr int kSmem = kBytes + 1024;
    static_assert(kSmem <= 232448, "shared memory above the per-block limit");
};

enum {
    kBarFull = 0,
    kBarEmpty = kBarFull + kMaxStages,
    kBarSFull = kBarEmpty + kMaxStages,
    kBarSEmpty = kBarSFull + kBufs,
    kBarDrain = kBarSEmpty + kBufs,
    kBarWide = kBarDrain + 1    // widening instance: a stage's e4m3 weight tile is written
};
static_assert(kBarWide + kMaxStages <= 32, "barriers above their shared-memory slots");
enum { kMiscTmem = 0, kMiscAbort = 1, kMiscBad = 2, kMiscTotal = 3 };

struct TcArgs {
    float *y;                    // nullable when qn is set
    int32_t *bsum;
    const int32_t *expert_off;   // [E+1] row offsets of the expert groups, or null (dense)
    uint8_t *qn;                 // the output quantized for the next projection, or null:
    float *qnd;                  //   codes [M][N] (tc form), scales [N/32][ldqnd]
    int64_t ldy, ldqnd;
    int32_t M, N, nb, bn, E;     // M: activation rows (all groups)
    int32_t qn_rot;              // 0 or 32: rotate the next projection's 32-blocks
    // dense only: tiles from tail_first on (the last partial wave) are each cut
    // into tail_k pieces along the tokens; tail_k = 1 cuts nothing
    int32_t tail_first, tail_k;
    // dense only, the K split of the cut pieces (split_p pieces, 0 = none):
    // the first split_kh K stages of piece p run on CTA p, the rest on CTA
    // split_p + p; the partial sums pass through the caller's workspace (a
    // header, ws_flag[p][16], ws_acc[p][ws_ld columns][128 rows])
    unsigned long long *ws_hdr, *ws_flag;
    float *ws_acc;
    int32_t split_p, split_kh, ws_ld;
    uint64_t wait_limit;
};

__device__ __forceinline__ void record(uint32_t bits) { atomicOr(&g_tc_status, bits); }

// per-warpgroup register budgets (every warp of the warpgroup executes the same one)
template <int N>
__device__ __forceinline__ void reg_dealloc() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void reg_alloc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void set_abort(volatile int *misc) {
    misc[kMiscAbort] = 1;
    record(kStatusTimeout);
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

// Tiles: per expert group e (one group of all rows when dense), every 128-row
// weight tile times every chunk of up to bn token rows.  A group's chunks start
// at its first row rounded down to a multiple of 4 (so the token-scale box
// starts on a 16-byte boundary); the rows of the chunk outside the group are
// computed but not stored.  Tiles are numbered group-major, then weight-tile
// major (consecutive CTAs share a weight tile).
struct TcTile {
    int n0;     // first weight row within the expert
    int wrow;   // its row in the [E * N] weight planes
    int g0;     // first token row of the chunk
    int clo, chi;   // columns [clo, chi) of the chunk belong to the group
    int ncols;  // MMA width: chi rounded up to 16
};

__device__ __forceinline__ int group_chunks(const int *s_off, int e, int bn) {
    const int lo = s_off[e], hi = s_off[e + 1];
    return hi > lo ? (hi - (lo & ~3) + bn - 1) / bn : 0;
}

template <bool kTail>
__device__ __forceinline__ TcTile tc_tile(int t, const TcArgs &a, const int *s_off,
                                          const int *s_tpre) {
    int sub = -1;   // the piece of a cut tail tile, or -1
    if constexpr (kTail) {
        if (t >= a.tail_first) {
            const int p = t - a.tail_first;
            t = a.tail_first + p / a.tail_k;
            sub = p - (p / a.tail_k) * a.tail_k;
        }
    }
    int lo = 0, hi = a.E;   // the last group whose first tile is <= t
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_tpre[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    const int e = lo;
    const int local = t - s_tpre[e];
    const int chunks = group_chunks(s_off, e, a.bn);
    const int wt = local / chunks, ch = local - wt * chunks;
    TcTile ti;
    ti.n0 = wt * kBM;
    ti.wrow = e * a.N + ti.n0;
    ti.g0 = (s_off[e] & ~3) + ch * a.bn;
    ti.clo = max(0, s_off[e] - ti.g0);
    ti.chi = min(a.bn, s_off[e + 1] - ti.g0);
    if (kTail && sub >= 0) {
        // piece `sub` of the chunk's columns [0, chi) (dense: clo = 0), in widths
        // that are multiples of 16 so every piece starts on a 16-byte boundary of
        // the token scales; trailing pieces of a narrow chunk are empty
        const int pw = ((ti.chi + a.tail_k - 1) / a.tail_k + 15) & ~15;
        ti.g0 += sub * pw;
        ti.chi = max(0, min(pw, ti.chi - sub * pw));
    }
    ti.ncols = (ti.chi + 15) & ~15;
    return ti;
}

// The CTA's work items in order.  Without the K split: tiles t = blockIdx.x,
// + gridDim.x, ... below `total`, every K stage.  With it, each cut piece of the
// last partial wave runs in two parts along K on two CTAs: CTA p < split_p
// starts with stages [0, split_kh) of piece p and leaves its partial sums in the
// workspace (mode 1), CTA split_p + p ends with stages [split_kh, nst) of piece
// p, starting from those sums (mode 2), and the uncut tiles t < tail_first go
// round robin in between (mode 0).  Every output still takes its blocks in
// order: the second part continues the first part's accumulators.
struct TcItem {
    int t, st0, st1, mode;
};

template <bool kSplit>
__device__ __forceinline__ int tc_item_count(const TcArgs &a, int total) {
    const int b = blockIdx.x, g = gridDim.x;
    if constexpr (kSplit) {
        if (a.split_p > 0) {
            const int main = b < a.tail_first ? (a.tail_first - 1 - b) / g + 1 : 0;
            return main + (b < a.split_p ? 1 : 0) + (b >= a.split_p && b < 2 * a.split_p ? 1 : 0);
        }
    }
    return b < total ? (total - 1 - b) / g + 1 : 0;
}

template <bool kSplit>
__device__ __forceinline__ TcItem tc_item(const TcArgs &a, int k, int nst) {
    const int b = blockIdx.x, g = gridDim.x;
    if constexpr (kSplit) {
        if (a.split_p > 0) {
            if (b < a.split_p) {
                if (k == 0) return TcItem{a.tail_first + b, 0, a.split_kh, 1};
                --k;
            }
            const int t = b + k * g;
            if (t < a.tail_first) return TcItem{t, 0, nst, 0};
            return TcItem{a.tail_first + b - a.split_p, a.split_kh, nst, 2};
        }
    }
    return TcItem{b + k * g, 0, nst, 0};
}

// The handoff of a split piece's partial sums between the two CTAs, per
// epilogue warp (its 32 rows x its columns of the piece): the first part stores
// its accumulators and then, after a fence, the launch's generation number in
// its flag (release); the second part waits for that number (acquire, bounded)
// and loads them.  The launch's number is the workspace header's value plus
// one; the header changes only when the last CTA to finish advances it, so
// flags left by an earlier launch (or a replay of the same graph node) never
// match.
__device__ __forceinline__ void st_release_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// The weight scales of the thread's row for the four blocks of K stage `st`
// held in shared-memory stage `s`: fp32 [128 rows][4] from the repacked form,
// or (widening instance) fp16 [128 rows][8], the scales of stages st & ~1 and
// st | 1 (the TMA box starts on a 16-byte boundary), widened exactly.
template <bool kWQ>
__device__ __forceinline__ void stage_dw(const float *s_sa, int s, int row, int st, float (&dw)[4]) {
    if constexpr (kWQ) {
        const uint2 h = *reinterpret_cast<const uint2 *>(
            reinterpret_cast<const uint8_t *>(s_sa) + s * kScaleBytes + row * 16 + (st & 1) * 8);
        const uint16_t hs[4] = {static_cast<uint16_t>(h.x), static_cast<uint16_t>(h.x >> 16),
                                static_cast<uint16_t>(h.y), static_cast<uint16_t>(h.y >> 16)};
#pragma unroll
        for (int j = 0; j < 4; ++j) asm("cvt.f32.f16 %0, %1;" : "=f"(dw[j]) : "h"(hs[j]));
    } else {
        const float4 d4 = *reinterpret_cast<const float4 *>(s_sa + s * (kScaleBytes / 4) + 4 * row);
        dw[0] = d4.x;
        dw[1] = d4.y;
        dw[2] = d4.z;
        dw[3] = d4.w;
    }
}

// The ring positions of an epilogue warp: shared-memory stage and TMEM buffer,
// each a counter and a phase bit.
struct EpiRing {
    uint32_t s, sph, gb, gph;
};

// One work item of an epilogue warp, without block sums: tile (or piece) t,
// K stages [st0, st0 + nstage).  kMode 0: the whole K range, from zero, to y;
// 1: the first part of a split piece, its accumulators to the workspace; 2: the
// second part, starting from the first part's accumulators, to y.  Arrivals
// come from one elected lane.  Returns false when a wait gave up.  A warp holds
// its lane quarter's 32 weight rows (one a thread, the 32x32b TMEM fragment)
// times its share of the tile's columns.
template <int EPQ, int XB, bool kQN, bool kTail, bool kWQ, int kMode>
__device__ __forceinline__ bool epi_item(const TcArgs &a, int t, int st0, int nstage,
                                         const int *s_off, const int *s_tpre, uint64_t *bars,
                                         const float *s_sa, const float *s_sb, float *s_q,
                                         uint32_t tmem, int warp, int lane,
                                         volatile int *abort_flag, EpiRing &r) {
    using C = TcCfg<EPQ, XB, kQN, kWQ>;
    const int ew = warp - C::kProdWarps;
    const int quad = warp & 3;                 // TMEM lanes 32 quad .. 32 quad + 31
    const int part = ew >> 2;                  // share of the columns
    const int row = quad * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const uint64_t lim = a.wait_limit;
    const TcTile ti = tc_tile<kTail>(t, a, s_off, s_tpre);
    if (kTail && ti.ncols == 0) return true;   // an empty piece: no role touches it
    const int n16 = ti.ncols >> 4;
    const int base = n16 / EPQ, rem = n16 % EPQ;
    const int nch = base + (part < rem ? 1 : 0);
    const int c0 = 16 * (part * base + min(part, rem));
    const uint32_t tcol_base = tmem + lane_addr + c0;
    uint64_t acc[8 * C::kMaxChunks];
#pragma unroll
    for (int i = 0; i < 8 * C::kMaxChunks; ++i) acc[i] = 0ull;
    if constexpr (kMode == 2) {
        if (nch > 0) {
            // the first part's accumulators, once its flag holds this launch's number
            const int p = t - a.tail_first;
            const unsigned long long *flag = a.ws_flag + p * 16 + ew;
            uint64_t polls = 0;
            const unsigned long long want = ld_relaxed_u64(a.ws_hdr) + 1;
            while (!__all_sync(0xFFFFFFFFu, ld_acquire_u64(flag) == want)) {
                if (++polls > lim || *abort_flag) return false;
            }
            // [piece][column][128 rows], the layout of y: a column's 32 rows are
            // one coalesced access of the warp
            const float *src = a.ws_acc + (static_cast<int64_t>(p) * a.ws_ld + c0) * kBM + row;
#pragma unroll
            for (int c = 0; c < C::kMaxChunks; ++c) {
                if (c < nch) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float lo = __ldcg(src + (16 * c + 2 * q) * kBM);
                        const float hi = __ldcg(src + (16 * c + 2 * q + 1) * kBM);
                        acc[8 * c + q] = pair_of(__float_as_uint(lo), __float_as_uint(hi));
                    }
                }
            }
        }
    }
    for (int si = 0; si < nstage; ++si) {
        const int st = st0 + si;
        if (!warp_wait(&bars[kBarFull + r.s], r.sph, lim, abort_flag)) return false;
        float dws[4];
        stage_dw<kWQ>(s_sa, r.s, row, st, dws);
        const float *sb = s_sb + r.s * (kScaleBytes / 4) + c0;   // [4 blocks][bn tokens]
#pragma unroll
        for (int j0 = 0; j0 < 4; j0 += kGroup) {
            if (!warp_wait(&bars[kBarSFull + r.gb], r.gph, lim, abort_flag)) return false;
            tc_fence_after();
            const uint32_t tcol0 = tcol_base + r.gb * (kGroup * 128);
            // one 16-column chunk of one block per TMEM wait (measured: fewer
            // live load registers beat fewer waits, and every reordering that
            // overlaps loads with folds measured slower); every accumulator
            // takes the blocks in order
#pragma unroll
            for (int c = 0; c < C::kMaxChunks; ++c) {
                if (c < nch) {
#pragma unroll
                    for (int i = 0; i < kGroup; ++i) {
                        uint32_t v[16];
                        tmem_ld_x16(tcol0 + i * 128 + c * 16, v);
                        tmem_ld_wait();
                        fold16(acc + 8 * c, dws[j0 + i], sb + (j0 + i) * a.bn + 16 * c, v);
                    }
                }
            }
            // the warp-wide wait above: every lane's TMEM reads of the buffer are done
            tc_fence_before();
            elect_arrive(&bars[kBarSEmpty + r.gb]);
            if (++r.gb == kBufs) {
                r.gb = 0;
                r.gph ^= 1;
            }
        }
        __syncwarp();
        elect_arrive(&bars[kBarEmpty + r.s]);
        if (++r.s == C::kStages) {
            r.s = 0;
            r.sph ^= 1;
        }
    }
    if constexpr (kMode == 1) {
        // the first part of a piece: its accumulators to the workspace, then the flag
        if (nch > 0) {
            const int p = t - a.tail_first;
            float *dst = a.ws_acc + (static_cast<int64_t>(p) * a.ws_ld + c0) * kBM + row;
#pragma unroll
            for (int c = 0; c < C::kMaxChunks; ++c) {
                if (c < nch) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const uint64_t pr = acc[8 * c + q];
                        __stcg(dst + (16 * c + 2 * q) * kBM, __uint_as_float(static_cast<uint32_t>(pr)));
                        __stcg(dst + (16 * c + 2 * q + 1) * kBM,
                               __uint_as_float(static_cast<uint32_t>(pr >> 32)));
                    }
                }
            }
            __threadfence();
            __syncwarp();
            if (lane == 0) st_release_u64(a.ws_flag + p * 16 + ew, ld_relaxed_u64(a.ws_hdr) + 1);
        }
        return true;
    }
    const int64_t n = ti.n0 + row;
    if (n < a.N && (!kQN || a.y)) {
#pragma unroll
        for (int c = 0; c < C::kMaxChunks; ++c) {
            if (c < nch) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int col = c0 + c * 16 + 2 * q;
                    const uint64_t pr = acc[8 * c + q];
                    if (col >= ti.clo && col < ti.chi)
                        a.y[(ti.g0 + col) * a.ldy + n] = __uint_as_float(static_cast<uint32_t>(pr));
                    if (col + 1 >= ti.clo && col + 1 < ti.chi)
                        a.y[(ti.g0 + col + 1) * a.ldy + n] =
                            __uint_as_float(static_cast<uint32_t>(pr >> 32));
                }
            }
        }
    }
    // the output quantized for the next projection.  The warp's 32 lanes are 32
    // consecutive output features, one 32-block of the next projection's input
    // for every token column (N % 32 == 0: a block is all inside or all outside
    // the N rows).  The warp turns its 32 rows x 32 columns around through a
    // 4 KB staging tile (16-byte chunks of a column XOR-swizzled by the column,
    // so writes and reads are free of bank conflicts); then lane t holds token
    // column t's whole block and rotates and quantizes it in registers, the
    // step the activation quantizer takes, with the same arithmetic.
    if constexpr (kQN) {
        float *stg = s_q + (warp - C::kProdWarps) * 1024;
#pragma unroll
        for (int c = 0; c < C::kMaxChunks; ++c) {
            if (c < nch) {
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const int t = c * 16 + q;
                    const uint64_t pr = acc[8 * c + (q >> 1)];
                    stg[t * 32 + ((((lane >> 2) ^ (t & 7))) << 2) + (lane & 3)] =
                        __uint_as_float(static_cast<uint32_t>(pr >> (32 * (q & 1))));
                }
            }
        }
        __syncwarp();
        const int col = c0 + lane;
        if (lane < 16 * nch && col >= ti.clo && col < ti.chi && ti.n0 + quad * 32 < a.N) {
            float v[32];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float4 f = *reinterpret_cast<const float4 *>(
                    stg + lane * 32 + ((k ^ (lane & 7)) << 2));
                v[4 * k] = f.x;
                v[4 * k + 1] = f.y;
                v[4 * k + 2] = f.z;
                v[4 * k + 3] = f.w;
            }
            if (a.qn_rot) rotate32(v);
            uint32_t w[8];
            const float d = quant_block_tc4(v, w);
            const int64_t g = ti.g0 + col;
            uint4 *dst = reinterpret_cast<uint4 *>(a.qn + g * a.N + ti.n0 + quad * 32);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            a.qnd[((ti.n0 + quad * 32) >> 5) * a.ldqnd + g] = d;
        }
        __syncwarp();   // the staging tile is free for the next tile
    }
    return true;
}

// The epilogue of one warp over all of the CTA's work items (TcItem): the
// uncut tiles and pieces, each over the whole K range, in one loop (measured:
// a loop over items whose K range is a variable made every tile of the
// instance about 6% slower), the two parts of a split piece before and after
// it.
template <int EPQ, int XB, bool kQN, bool kTail, bool kWQ, bool kSplit>
__device__ __forceinline__ bool epilogue_tiles(const TcArgs &a, int total, const int *s_off,
                                               const int *s_tpre, uint64_t *bars, const float *s_sa,
                                               const float *s_sb, float *s_q, uint32_t tmem,
                                               int warp, int lane, volatile int *abort_flag) {
    const int b = blockIdx.x, g = gridDim.x;
    const int nst = a.nb / 4;
    EpiRing r{0u, 0u, 0u, 0u};
    int main_end = total;
    if constexpr (kSplit) {
        if (a.split_p > 0) {
            main_end = a.tail_first;
            if (b < a.split_p &&
                !epi_item<EPQ, XB, kQN, kTail, kWQ, 1>(a, a.tail_first + b, 0, a.split_kh, s_off,
                                                        s_tpre, bars, s_sa, s_sb, s_q, tmem, warp,
                                                        lane, abort_flag, r))
                return false;
        }
    }
    const int nit = b < main_end ? (main_end - 1 - b) / g + 1 : 0;
    for (int k = 0; k < nit; ++k)
        if (!epi_item<EPQ, XB, kQN, kTail, kWQ, 0>(a, b + k * g, 0, nst, s_off, s_tpre, bars, s_sa,
                                                    s_sb, s_q, tmem, warp, lane, abort_flag, r))
            return false;
    if constexpr (kSplit) {
        if (a.split_p > 0 && b >= a.split_p && b < 2 * a.split_p &&
            !epi_item<EPQ, XB, kQN, kTail, kWQ, 2>(a, a.tail_first + b - a.split_p, a.split_kh,
                                                    nst - a.split_kh, s_off, s_tpre, bars, s_sa,
                                                    s_sb, s_q, tmem, warp, lane, abort_flag, r))
            return false;
    }
    return true;
}

// The epilogue of one warp over all of its tiles in the instances without a
// cut tail (dense shapes that fill their waves, and the expert groups), without
// block sums: the same work as epi_item<.., 0> over a tile loop of its own
// (measured on GB300: this form runs the MoE micro-batch's expert GEMMs 4-5%
// faster than the item-body form, which runs the cut instances 4-5% faster).
// Ring positions of the shared-memory stages and TMEM buffers are carried as
// counters and phase bits, arrivals come from one elected lane.  Returns false
// when a wait gave up.  A warp holds its lane quarter's 32 weight rows (one a
// thread, the 32x32b TMEM fragment) times its share of the tile's columns.
template <int EPQ, int XB, bool kQN, bool kTail, bool kWQ>
__device__ __forceinline__ bool epilogue_tiles_plain(const TcArgs &a, int total, const int *s_off,
                                               const int *s_tpre, uint64_t *bars, const float *s_sa,
                                               const float *s_sb, float *s_q, uint32_t tmem,
                                               int warp, int lane, volatile int *abort_flag) {
    using C = TcCfg<EPQ, XB, kQN, kWQ>;
    const int ew = warp - C::kProdWarps;
    const int quad = warp & 3;                 // TMEM lanes 32 quad .. 32 quad + 31
    const int part = ew >> 2;                  // share of the columns
    const int row = quad * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
    const int nst = a.nb / 4;
    const uint64_t lim = a.wait_limit;
    uint32_t s = 0, sph = 0, gb = 0, gph = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const TcTile ti = tc_tile<kTail>(t, a, s_off, s_tpre);
        if (kTail && ti.ncols == 0) continue;   // an empty piece: no role touches it
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
            float dws[4];
            stage_dw<kWQ>(s_sa, s, row, st, dws);
            const float *sb = s_sb + s * (kScaleBytes / 4) + c0;   // [4 blocks][bn tokens]
#pragma unroll
            for (int j0 = 0; j0 < 4; j0 += kGroup) {
                if (!warp_wait(&bars[kBarSFull + gb], gph, lim, abort_flag)) return false;
                tc_fence_after();
                const uint32_t tcol0 = tcol_base + gb * (kGroup * 128);
                // one 16-column chunk of one block per TMEM wait (measured: fewer
                // live load registers beat fewer waits, and every reordering that
                // overlaps loads with folds measured slower); every accumulator
                // takes the blocks in order
#pragma unroll
                for (int c = 0; c < C::kMaxChunks; ++c) {
                    if (c < nch) {
#pragma unroll
                        for (int i = 0; i < kGroup; ++i) {
                            uint32_t v[16];
                            tmem_ld_x16(tcol0 + i * 128 + c * 16, v);
                            tmem_ld_wait();
                            fold16(acc + 8 * c, dws[j0 + i], sb + (j0 + i) * a.bn + 16 * c, v);
                        }
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
            if (++s == C::kStages) {
                s = 0;
                sph ^= 1;
            }
        }
        const int64_t n = ti.n0 + row;
        if (n < a.N && (!kQN || a.y)) {
#pragma unroll
            for (int c = 0; c < C::kMaxChunks; ++c) {
                if (c < nch) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int col = c0 + c * 16 + 2 * q;
                        const uint64_t pr = acc[8 * c + q];
                        if (col >= ti.clo && col < ti.chi)
                            a.y[(ti.g0 + col) * a.ldy + n] = __uint_as_float(static_cast<uint32_t>(pr));
                        if (col + 1 >= ti.clo && col + 1 < ti.chi)
                            a.y[(ti.g0 + col + 1) * a.ldy + n] =
                                __uint_as_float(static_cast<uint32_t>(pr >> 32));
                    }
                }
            }
        }
        // the output quantized for the next projection.  The warp's 32 lanes are 32
        // consecutive output features, one 32-block of the next projection's input
        // for every token column (N % 32 == 0: a block is all inside or all outside
        // the N rows).  The warp turns its 32 rows x 32 columns around through a
        // 4 KB staging tile (16-byte chunks of a column XOR-swizzled by the column,
        // so writes and reads are free of bank conflicts); then lane t holds token
        // column t's whole block and rotates and quantizes it in registers, the
        // step the activation quantizer takes, with the same arithmetic.
        if constexpr (kQN) {
            float *stg = s_q + (warp - C::kProdWarps) * 1024;
#pragma unroll
            for (int c = 0; c < C::kMaxChunks; ++c) {
                if (c < nch) {
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int t = c * 16 + q;
                        const uint64_t pr = acc[8 * c + (q >> 1)];
                        stg[t * 32 + ((((lane >> 2) ^ (t & 7))) << 2) + (lane & 3)] =
                            __uint_as_float(static_cast<uint32_t>(pr >> (32 * (q & 1))));
                    }
                }
            }
            __syncwarp();
            const int col = c0 + lane;
            if (lane < 16 * nch && col >= ti.clo && col < ti.chi && ti.n0 + quad * 32 < a.N) {
                float v[32];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float4 f = *reinterpret_cast<const float4 *>(
                        stg + lane * 32 + ((k ^ (lane & 7)) << 2));
                    v[4 * k] = f.x;
                    v[4 * k + 1] = f.y;
                    v[4 * k + 2] = f.z;
                    v[4 * k + 3] = f.w;
                }
                if (a.qn_rot) rotate32(v);
                uint32_t w[8];
                const float d = quant_block_tc4(v, w);
                const int64_t g = ti.g0 + col;
                uint4 *dst = reinterpret_cast<uint4 *>(a.qn + g * a.N + ti.n0 + quad * 32);
                dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                a.qnd[((ti.n0 + quad * 32) >> 5) * a.ldqnd + g] = d;
            }
            __syncwarp();   // the staging tile is free for the next tile
        }
    }
    return true;
}

// The widening warps (2 and 3) of the widening instance over all of the CTA's
// tiles: per K stage, once TMA has landed the stage, the 128 x 64-byte tile of
// Q4_0 bytes becomes the 128 x 128-byte tile of code bytes 0x0q in the layout the
// MMA reads (128B swizzle: the 16-byte chunk c of row r sits at chunk c ^ (r & 7)
// of the row, rows in 8-row atoms of 1 KB).  Thread wt (0..63) takes the
// (row, block) items wt, wt + 64, ...: a warp's 32 items are 8 rows x 4 blocks,
// so eight lanes read 128 contiguous bytes and write eight distinct chunk
// positions (free of bank conflicts).  Block j of a row: its 16 Q4_0 bytes give
// chunk 2 j (elements 0..15, the low nibbles) and chunk 2 j + 1 (16..31).
// Returns false when a wait gave up.
template <bool kTail>
__device__ __forceinline__ bool widen_tiles(const TcArgs &a, int total, const int *s_off,
                                            const int *s_tpre, uint64_t *bars, const uint8_t *s_n,
                                            uint8_t *s_a, int wt, volatile int *abort_flag) {
    using C = TcCfg<4, 4, false, true>;
    const int nst = a.nb / 4;
    uint32_t ks = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const TcTile ti = tc_tile<kTail>(t, a, s_off, s_tpre);
        if (kTail && ti.ncols == 0) continue;
        for (int st = 0; st < nst; ++st, ++ks) {
            const int s = ks % C::kStages;
            // (measured: a suspended wait by one lane makes the MMA wait longer for
            // the widened tile; a spinning lane is no faster than the whole warp)
            if (!warp_wait(&bars[kBarFull + s], (ks / C::kStages) & 1, a.wait_limit, abort_flag))
                return false;
            const uint8_t *nib = s_n + s * kNibBytes;
            uint8_t *wide = s_a + s * kTileBytes;
#pragma unroll 2
            for (int it = 0; it < 8; ++it) {
                const int i = it * 64 + wt, r = i >> 2, j = i & 3;
                const uint4 x = *reinterpret_cast<const uint4 *>(nib + r * 64 + j * 16);
                uint4 lo, hi;
                widen_q4_0_word(x.x, lo.x, hi.x);
                widen_q4_0_word(x.y, lo.y, hi.y);
                widen_q4_0_word(x.z, lo.z, hi.z);
                widen_q4_0_word(x.w, lo.w, hi.w);
                uint8_t *rp = wide + (r >> 3) * 1024 + (r & 7) * 128;
                *reinterpret_cast<uint4 *>(rp + (((2 * j) ^ (r & 7)) << 4)) = lo;
                *reinterpret_cast<uint4 *>(rp + (((2 * j + 1) ^ (r & 7)) << 4)) = hi;
            }
            // the MMA reads the tile through the async proxy
            fence_proxy_async_smem();
            __syncwarp();
            elect_arrive(&bars[kBarWide + s]);
        }
    }
    return true;
}

// kEpi: 0 = y only, 1 = y and the block sums, 2 = y (optional) and the output
// quantized for the next projection.  kTail: the last partial wave's tiles are
// cut into pieces (TcArgs::tail_first, tail_k).  kWQ: the widening instance
// (map_a over the Q4_0 nibbles, map_sa over the fp16 scales).  kSplit: the cut
// pieces also run in two parts along K (TcArgs::split_p, TcItem); an instance
// of its own, as the cut instance without that code measured about 4% faster
// on GB300.
template <int EPQ, int XB, int kEpi, bool kTail = false, bool kWQ = false, bool kSplit = false>
__global__ void __launch_bounds__(TcCfg<EPQ, XB, kEpi == 2, kWQ>::kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const __grid_constant__ CUtensorMap map_sa,
                   const __grid_constant__ CUtensorMap map_sb, const TcArgs a) {
    static_assert(!kSplit || (kTail && kEpi != 1 && !kWQ), "the K split: no block sums, cut tail");
    using C = TcCfg<EPQ, XB, kEpi == 2, kWQ>;
    constexpr int kStages = C::kStages;
    constexpr bool kSums = kEpi == 1;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *s_a = smem + C::kOffA;
    uint8_t *s_b = smem + C::kOffB;
    float *s_sa = reinterpret_cast<float *>(smem + C::kOffSA);
    float *s_sb = reinterpret_cast<float *>(smem + C::kOffSB);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
    volatile int *misc = reinterpret_cast<volatile int *>(smem + C::kOffMisc);
    int *s_off = reinterpret_cast<int *>(smem + C::kOffGrp);
    int *s_tpre = s_off + kMaxExperts + 1;
    float *s_q = reinterpret_cast<float *>(smem + C::kOffQ);   // kEpi == 2: staging tiles
    uint8_t *s_n = smem + C::kOffN;                             // kWQ: Q4_0 nibble tiles
    uint8_t *s_c = smem + C::kOffC;                             // kWQ: the constant tile

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nst = a.nb / 4;
    const uint64_t lim = a.wait_limit;
    const uint32_t stage_tx =
        (kWQ ? kNibBytes : kTileBytes) + (XB / 4) * a.bn * 128 + kScaleBytes + a.bn * 16;
    const int E = a.E;
    const int nt = (a.N + kBM - 1) / kBM;

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
        if constexpr (kWQ)
            for (int i = 0; i < kStages; ++i) mbar_init(&bars[kBarWide + i], kWidenWarps);
        misc[kMiscAbort] = 0;
        misc[kMiscBad] = 0;
        fence_barrier_init();
    }
    if constexpr (kWQ) {
        // the constant A operand: every weight -8 * 2^-9 = -2^-6 (e4m3 0x88), so
        // one more MMA per block adds -8 times the activation block sum
        uint4 *c = reinterpret_cast<uint4 *>(s_c);
        for (int i = tid; i < kTileBytes / 16; i += C::kThreads)
            c[i] = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
        fence_proxy_async_smem();
    }
    // the previous kernel of the stream (launched ahead of this one) is done
    // before anything here touches global memory
    pdl_wait();
    pdl_trigger();
    // group offsets: checked (0 = off[0] <= ... <= off[E] = M), then the tile
    // prefix over the groups (warp 0)
    if (a.expert_off == nullptr) {
        if (tid == 0) {
            s_off[0] = 0;
            s_off[1] = a.M;
        }
    } else {
        for (int i = tid; i <= E; i += C::kThreads) s_off[i] = a.expert_off[i];
    }
    __syncthreads();
    for (int i = tid; i <= E; i += C::kThreads) {
        const int v = s_off[i];
        if ((i == 0 && v != 0) || (i == E && v != a.M) || (i < E && s_off[i + 1] < v))
            misc[kMiscBad] = 1;
    }
    __syncthreads();
    if (warp == 0 && !misc[kMiscBad]) {
        const int per = (E + 31) / 32;
        const int e0 = lane * per;
        int sum = 0;
        for (int i = 0; i < per; ++i)
            if (e0 + i < E) sum += nt * group_chunks(s_off, e0 + i, a.bn);
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - sum;
        for (int i = 0; i < per; ++i) {
            if (e0 + i < E) {
                s_tpre[e0 + i] = run;
                run += nt * group_chunks(s_off, e0 + i, a.bn);
            }
        }
        if (lane == 31) {
            s_tpre[E] = incl;
            misc[kMiscTotal] = (kTail && incl > a.tail_first)
                                   ? a.tail_first + (incl - a.tail_first) * a.tail_k
                                   : incl;
        }
    }
    __syncthreads();
    if (misc[kMiscBad]) {
        if (tid == 0 && blockIdx.x == 0) record(kStatusGuard);
        return;
    }
    const int total = misc[kMiscTotal];
    if (a.split_p == 0 && static_cast<int>(blockIdx.x) >= total) return;
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
        if constexpr (C::kRegSplit) reg_dealloc<C::kProdRegs>();
        if (lane == 0) {
            prefetch_tmap(&map_a);
            prefetch_tmap(&map_b);
            prefetch_tmap(&map_sa);
            prefetch_tmap(&map_sb);
            uint32_t ks = 0;
            bool ok = true;
            const int nit = tc_item_count<kSplit>(a, total);
            for (int k = 0; k < nit && ok; ++k) {
                const TcItem it = tc_item<kSplit>(a, k, nst);
                const TcTile ti = tc_tile<kTail>(it.t, a, s_off, s_tpre);
                if (kTail && ti.ncols == 0) continue;
                for (int st = it.st0; st < it.st1; ++st, ++ks) {
                    const int s = ks % kStages;
                    if (!mbar_wait_bounded(&bars[kBarEmpty + s], ((ks / kStages) & 1) ^ 1, lim,
                                           abort_flag)) {
                        set_abort(misc);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars[kBarFull + s], stage_tx);
                    if constexpr (kWQ)
                        tma_load_2d(s_n + s * kNibBytes, &map_a, &bars[kBarFull + s], st * 64, ti.wrow);
                    else
                        tma_load_2d(s_a + s * kTileBytes, &map_a, &bars[kBarFull + s], st * 128,
                                    ti.wrow);
                    tma_load_2d(s_b + s * C::kBTile, &map_b, &bars[kBarFull + s], st * 128 * (XB / 4),
                                ti.g0);
                    if constexpr (XB == 8)
                        tma_load_2d(s_b + s * C::kBTile + kTileBytes, &map_b, &bars[kBarFull + s],
                                    st * 256 + 128, ti.g0);
                    tma_load_2d(s_sa + s * (kScaleBytes / 4), &map_sa, &bars[kBarFull + s],
                                kWQ ? (st * 4) & ~7 : st * 4, ti.wrow);
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
        if constexpr (C::kRegSplit) reg_dealloc<C::kProdRegs>();
        if (lane == 0) {
            uint32_t ks = 0, kg = 0;
            bool ok = true;
            const int nit = tc_item_count<kSplit>(a, total);
            for (int k = 0; k < nit && ok; ++k) {
                const TcItem it = tc_item<kSplit>(a, k, nst);
                const TcTile ti = tc_tile<kTail>(it.t, a, s_off, s_tpre);
                if (kTail && ti.ncols == 0) continue;
                const uint32_t idesc =
                    kWQ ? idesc_e4m3_e5m2_f32(kBM, ti.ncols) : idesc_e4m3_f32(kBM, ti.ncols);
                for (int st = it.st0; st < it.st1 && ok; ++st, ++ks) {
                    const int s = ks % kStages;
                    // the widening instance's weight tile is ready once the widening
                    // warps, which waited for the stage themselves, have written it
                    if (!mbar_wait_bounded(&bars[(kWQ ? kBarWide : kBarFull) + s], (ks / kStages) & 1,
                                           lim, abort_flag)) {
                        set_abort(misc);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t da = smem_desc_sw128(smem_u32(s_a + s * kTileBytes));
                    const uint64_t dc = smem_desc_sw128(smem_u32(s_c));
                    const uint64_t db = smem_desc_sw128(smem_u32(s_b + s * C::kBTile));
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
                            const int j = j0 + i;
                            // block j's 32 weight bytes start 32 j bytes into each 128-byte row
                            const uint64_t koff = (32 * j) >> 4;
                            const uint32_t slot = tmem + (gb * kGroup + i) * 128;
                            if constexpr (kWQ) {
                                // (q 2^-9)(512 x) summed, then (-8 2^-9)(512 x):
                                // S = sum q x - 8 sum x, integers below 2^24, exact
                                mma_f8f6f4(slot, da + koff, db + koff, idesc, 0);
                                mma_f8f6f4(slot, dc + koff, db + koff, idesc, 1);
                            } else if constexpr (XB == 4) {
                                mma_f8f6f4(slot, da + koff, db + koff, idesc, 0);
                            } else {
                                // S = sum w (16 h) + sum w l: two MMAs into one accumulator
                                // (every partial sum is an integer below 2^24: exact)
                                const uint64_t dbj = db + ((j >> 1) * kTileBytes >> 4) +
                                                     (((j & 1) * 64) >> 4);
                                mma_f8f6f4(slot, da + koff, dbj, idesc, 0);
                                mma_f8f6f4(slot, da + koff, dbj + (32 >> 4), idesc, 1);
                            }
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
    } else if (warp < C::kProdWarps) {
        // the producer warpgroup's other two warps: idle, or the widening warps
        if constexpr (C::kRegSplit) reg_dealloc<C::kProdRegs>();
        if constexpr (kWQ) {
            if (!widen_tiles<kTail>(a, total, s_off, s_tpre, bars, s_n, s_a, (warp - 2) * 32 + lane,
                                    abort_flag))
                set_abort(misc);
        }
    } else if constexpr (!kSums) {
        // ------------------------------------------------------- epilogue
        if constexpr (C::kRegSplit) reg_alloc<C::kEpiRegs>();
        bool eok;
        if constexpr (!kTail)
            eok = epilogue_tiles_plain<EPQ, XB, kEpi == 2, kTail, kWQ>(
                a, total, s_off, s_tpre, bars, s_sa, s_sb, s_q, tmem, warp, lane, abort_flag);
        else
            eok = epilogue_tiles<EPQ, XB, kEpi == 2, kTail, kWQ, kSplit>(
                a, total, s_off, s_tpre, bars, s_sa, s_sb, s_q, tmem, warp, lane, abort_flag);
        if (!eok) set_abort(misc);
    } else {
        // ------------------------------------ epilogue with block sums
        if constexpr (C::kRegSplit) reg_alloc<C::kEpiRegs>();
        const int ew = warp - C::kProdWarps;
        const int quad = warp & 3;                 // TMEM lanes 32*quad .. +31
        const int part = ew >> 2;                  // share of the columns
        const int row = quad * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(quad * 32) << 16;
        uint32_t ks = 0, kg = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const TcTile ti = tc_tile<kTail>(t, a, s_off, s_tpre);
            if (kTail && ti.ncols == 0) continue;
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
                const float *sb = s_sb + s * (kScaleBytes / 4);   // [4 blocks][bn tokens]
                float dws[4];
                stage_dw<kWQ>(s_sa, s, row, st, dws);
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
                                    if (n < a.N) {
#pragma unroll
                                        for (int q = 0; q < 16; ++q)
                                            if (col0 + q >= ti.clo && col0 + q < ti.chi)
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
                            if (col >= ti.clo && col < ti.chi)
                                a.y[(ti.g0 + col) * a.ldy + n] =
                                    __uint_as_float(static_cast<uint32_t>(pr));
                            if (col + 1 >= ti.clo && col + 1 < ti.chi)
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
    if constexpr (kSplit) {
        // the last CTA to finish advances the generation: the header holds this
        // launch's number until then (every CTA reads it before it counts itself
        // done)
        if (tid == 0 && a.ws_hdr) {
            unsigned int *done = reinterpret_cast<unsigned int *>(a.ws_hdr + 1);
            __threadfence();
            if (atomicAdd(done, 1u) == gridDim.x - 1) {
                *done = 0u;
                st_relaxed_u64(a.ws_hdr, ld_relaxed_u64(a.ws_hdr) + 1);
                __threadfence();
            }
        }
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

// The dense schedule: tokens per tile (bn), and how many pieces each tile of
// the last partial wave is cut into along the tokens (tail_k), chosen by
// simulating the kernel's static round-robin assignment of tiles to CTAs.
struct TcPlan {
    int bn, tail_k;
    int64_t tail_first, total, grid;
    // the K split of the cut pieces (split_p = 0: none): pieces split_p,
    // stages [0, split_kh) first, piece width (the workspace's row stride) ws_ld
    int64_t split_p = 0, split_kh = 0, ws_ld = 0;
};

// a tile costs its MMA width plus a fixed part that is about the work of 80
// more columns, and the kernel with three epilogue warps per lane quarter (the
// tile widths whose 16-column chunks do not split evenly over four) runs 4-8%
// slower per unit; fitted on GB300 to a sweep of widths 48-128 on seven shapes
// (within 1.4% rms of the measured times of each shape)
inline int64_t tile_cost(int64_t width) { return width > 0 ? ((width + 15) / 16) * 16 + 80 : 0; }
inline int64_t width_factor(int bn) {   // percent
    switch (bn / 16) {
        case 1: case 2: return 105;
        case 5: return 104;
        case 6: return 108;
        default: return 100;
    }
}

// The simulated makespan of a plan, in tile-cost units times the nst K stages
// (a piece run in two parts costs its share of the stages in each).  With
// `split`, every cut piece runs in two parts (TcItem); that needs a full wave
// of uncut tiles (so the second part of a piece starts after its first part
// has ended) and two CTAs a piece; returns -1 where a plan does not apply.
inline int64_t plan_makespan(int64_t M, int64_t nt, int sms, int bn, int k, int64_t nst,
                             bool split, TcPlan *plan) {
    const int64_t chunks = (M + bn - 1) / bn;
    const int64_t T = nt * chunks;
    const int64_t r = T % sms;   // tiles of the last partial wave
    const int64_t tail_first = ((k > 1 || split) && r > 0) ? T - r : T;
    const int64_t total = tail_first + (T - tail_first) * k;
    const int64_t grid = total < sms ? total : sms;
    const int64_t P = total - tail_first;   // cut pieces
    const int64_t kh = nst / 2;
    if (split && (P == 0 || P > kSplitMaxP || 2 * P > grid || tail_first < grid || kh < 1)) return -1;
    auto width = [&](int64_t t) {
        const int64_t ch = t % chunks;
        return ch == chunks - 1 ? M - ch * bn : static_cast<int64_t>(bn);
    };
    int64_t pw_max = 0;
    auto piece_cost = [&](int64_t p) {   // piece p of the cut tiles
        const int64_t sub = p % k;
        const int64_t w = width(tail_first + p / k);
        const int64_t pw = ((w + k - 1) / k + 15) / 16 * 16;
        const int64_t wp = w - sub * pw < pw ? w - sub * pw : pw;
        if (pw > pw_max) pw_max = pw;
        return tile_cost(wp > 0 ? wp : 0);
    };
    int64_t worst = 0;
    for (int64_t c = 0; c < grid; ++c) {
        int64_t cost = 0;
        if (split) {
            if (c < P) cost += piece_cost(c) * kh;
            for (int64_t t = c; t < tail_first; t += grid) cost += tile_cost(width(t)) * nst;
            if (c >= P && c < 2 * P) cost += piece_cost(c - P) * (nst - kh);
        } else {
            for (int64_t t = c; t < total; t += grid)
                cost += (t < tail_first ? tile_cost(width(t)) : piece_cost(t - tail_first)) * nst;
        }
        if (cost > worst) worst = cost;
    }
    if (plan) {
        *plan = TcPlan{bn, k, tail_first, total, grid};
        if (split) {
            plan->split_p = P;
            plan->split_kh = kh;
            plan->ws_ld = pw_max;
        }
    }
    return worst * width_factor(bn);
}

TcPlan plan_tc_uncached(int64_t M, int64_t N, int sms, bool allow_cut, bool allow_split,
                        int64_t nst) {
    const int64_t nt = (N + kBM - 1) / kBM;
    TcPlan plan{};
    int64_t best = INT64_MAX;
    for (int bn = kBNMax; bn >= 32; bn -= 16) {
        TcPlan p{};
        const int64_t m = plan_makespan(M, nt, sms, bn, 1, nst, false, &p);
        if (m < best) {
            best = m;
            plan = p;
        }
    }
    // then a cut of the last partial wave, at any width, kept where the
    // simulation shortens the best uncut makespan by at least 1%; then the same
    // pieces run in two parts along K, kept where that shortens the best plan
    // so far by at least 5% (measured on GB300: the instance with the split
    // runs its tiles 8-9% slower, so the simulation's gain shrinks: 16% for the
    // pp512 attention and FFN-down shapes gave 9-13%, 8% for the 1024-token
    // ones gave 4-7%, and 3% for pp512 FFN gate/up gave a loss)
    for (int split = 0; split <= (allow_split ? 1 : 0); ++split) {
        const int64_t before = best;
        const int64_t keep = split ? 95 : 99;
        for (int bn = kBNMax; allow_cut && bn >= 32; bn -= 16) {
            for (int k = split ? 1 : 2; k <= 8 && bn / k >= 16; k *= 2) {
                TcPlan p{};
                const int64_t m = plan_makespan(M, nt, sms, bn, k, nst, split != 0, &p);
                if (m >= 0 && m < best && m * 100 <= before * keep) {
                    best = m;
                    plan = p;
                }
            }
        }
    }
    return plan;
}

// the simulation costs O(tiles) host time per candidate: remember the plan of
// each shape (a bounded table, emptied when full)
TcPlan plan_tc(int64_t M, int64_t N, int sms, bool allow_cut, bool allow_split, int64_t nst) {
    static std::mutex mu;
    static std::map<std::tuple<int64_t, int64_t, int, bool, bool, int64_t>, TcPlan> plans;
    if (!allow_split) nst = 1;   // the plan does not depend on K then
    const auto key = std::make_tuple(M, N, sms, allow_cut, allow_split, nst);
    {
        std::lock_guard<std::mutex> lock(mu);
        const auto it = plans.find(key);
        if (it != plans.end()) return it->second;
    }
    const TcPlan plan = plan_tc_uncached(M, N, sms, allow_cut, allow_split, nst);
    std::lock_guard<std::mutex> lock(mu);
    if (plans.size() >= 4096) plans.clear();
    plans.emplace(key, plan);
    return plan;
}

// The workspace of a plan with the K split, at fixed offsets whatever the plan
// (so that a workspace reused by plans of other shapes never finds partial sums
// where it looks for flags): a 256-byte header (the generation number, the
// count of finished CTAs), flags [kSplitMaxP][16] (generation numbers), then the
// partial sums [split_p][ws_ld columns][128 rows] (fp32).
constexpr int64_t kSplitFlagOff = 256;
constexpr int64_t kSplitAccOff = kSplitFlagOff + kSplitMaxP * 16 * 8;
inline size_t split_ws_bytes(const TcPlan &p) {
    if (p.split_p == 0) return 0;
    return static_cast<size_t>(kSplitAccOff) + static_cast<size_t>(p.split_p) * kBM * p.ws_ld * 4;
}

template <int EPQ, int XB, int kEpi, bool kTail = false, bool kWQ = false, bool kSplit = false>
h32_status launch_tc(const CUtensorMap *maps, const TcArgs &a, int grid, cudaStream_t s) {
    using C = TcCfg<EPQ, XB, kEpi == 2, kWQ>;
    constexpr int kSmem = C::kSmem;
    const cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<EPQ, XB, kEpi, kTail, kWQ, kSplit>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return launch_status(e);
    if constexpr (C::kRegSplit) {
        // the epilogue's setmaxnreg.inc waits until the pool holds its registers:
        // never launch with fewer registers a thread than the split assumes
        // (read once per kernel; a failed read leaves -1 and refuses every launch)
        static const int regs = [] {
            cudaFuncAttributes fa{};
            return cudaFuncGetAttributes(&fa, gemm_tc_kernel<EPQ, XB, kEpi, kTail, kWQ, kSplit>) ==
                           cudaSuccess
                       ? fa.numRegs
                       : -1;
        }();
        if (regs < 0 || ((regs + 7) / 8) * 8 < C::kLaunchRegs) {
            note_error("tc GEMM compiled with fewer registers than its warpgroup split needs");
            return H32_ERR_UNSUPPORTED;
        }
    }
    const cudaError_t el = launch_pdl(gemm_tc_kernel<EPQ, XB, kEpi, kTail, kWQ, kSplit>, dim3(grid), dim3(C::kThreads),
                                      kSmem, s, maps[0], maps[1], maps[2], maps[3], a);
    return launch_status(el != cudaSuccess ? el : cudaGetLastError());
}

}  // namespace

__device__ uint32_t g_tc_status_taken;
__global__ void take_g_tc_status() { g_tc_status_taken = atomicExch(&g_tc_status, 0u); }

h32_status tc_read_and_clear_status(cudaStream_t s) {
    bool ok = false;
    const uint32_t v = take_status(take_g_tc_status, g_tc_status_taken, s, &ok);
    if (!ok) return H32_ERR_CUDA;
    if (v & kStatusTimeout) return H32_ERR_TIMEOUT;
    if (v & kStatusGuard) return H32_ERR_DEVICE_GUARD;
    return H32_OK;
}

}  // namespace h32

namespace h32 {
namespace {

// Shared by the dense and the expert-batched entry points: checks, tensor
// maps, launch.  E groups of weight rows [E * N][K]; expert_off null = dense.
// With wd16 set (the widening instance), wp holds the Q4_0 nibbles [E * N][K / 2]
// and wd16 the fp16 scales [E * N][K / 32]; wsc and ldws are unused.
h32_status run_gemm_tc(int xbits, const uint8_t *wp, const float *wsc, int64_t ldws, int64_t E,
                       const uint8_t *xw, const float *xdt, int64_t ldxd,
                       const int32_t *expert_off, int64_t M, int64_t N, int64_t K, float *y,
                       int64_t ldy, int32_t *block_sums, void *stream, uint8_t *qn = nullptr,
                       float *qnd = nullptr, int64_t ldqnd = 0, int qn_rot = 0,
                       const uint16_t *wd16 = nullptr, void *ws = nullptr, size_t ws_bytes = 0) {
    if (wd16) ldws = K / 32;
    if (M < 0 || N <= 0 || K <= 0 || (K % 128) != 0 || (N % 16) != 0 || (y && ldy < N) ||
        ldws < K / 32 || (ldws % 4) != 0 || ldxd < M || (ldxd % 4) != 0 || E < 1 ||
        E > kMaxExperts)
        return H32_ERR_INVALID_ARG;
    if (qn && ((N % 32) != 0 || !qnd || ldqnd < M || block_sums ||
               (qn_rot != 0 && qn_rot != 1 && qn_rot != 32)))
        return H32_ERR_INVALID_ARG;
    // the widening instance: fp16 scale rows of K / 16 bytes, a multiple of 16
    // for their tensor map
    if (wd16 && ((K % 256) != 0 || xbits != 4 || qn)) return H32_ERR_INVALID_ARG;
    if (M == 0) return H32_OK;
    if (!wp || (!wsc && !wd16) || !xw || !xdt || (!y && !qn)) return H32_ERR_INVALID_ARG;
    if (!aligned16(wp) || (wsc && !aligned16(wsc)) || (wd16 && !aligned16(wd16)) ||
        !aligned16(xw) || !aligned16(xdt) ||
        (y && !aligned16(y)) || (qn && (!aligned16(qn) || !aligned16(qnd))) ||
        (block_sums && !aligned16(block_sums)) || (expert_off && !aligned16(expert_off)) ||
        (y && (ldy % 4) != 0))
        return H32_ERR_ALIGNMENT;
    if (M > 0x7FFFFFFFll || E * N > 0x7FFFFFFFll || K > 0x7FFFFFFFll) return H32_ERR_INVALID_ARG;
    int sms = 0;
    H32_TRY(check_device(&sms));
    // dense: the tile width and the cut of the last wave from the schedule
    // simulation; groups: full 128-row chunks, nothing cut
    TcPlan plan{kBNMax, 1, 0, 0, sms};
    if (expert_off) {
        // the kernel numbers tiles in int: group e has at most
        // ceil((size_e + 3) / 128) chunks, so at most R / 128 + 2 E chunks in all
        if (((N + kBM - 1) / kBM) * (M / kBNMax + 2 * E + 1) > 0x7FFFFFFFll)
            return H32_ERR_INVALID_ARG;
    } else {
        if (((N + kBM - 1) / kBM) * ((M + 15) / 16) * 8 > 0x7FFFFFFFll) return H32_ERR_INVALID_ARG;
        plan = plan_tc(M, N, sms, !block_sums, ws && !block_sums && !wd16, K / 128);
        if (plan.split_p > 0) {
            if (ws_bytes < split_ws_bytes(plan)) return H32_ERR_INVALID_ARG;
            if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return H32_ERR_ALIGNMENT;
        }
    }
    const int bn = plan.bn;
    const int64_t grid = plan.grid;
    CUtensorMap maps[4];
    if (wd16) {
        H32_TRY(make_map(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, wp, K / 2, E * N, K / 2, 64,
                         kBM, false));
        H32_TRY(make_map(&maps[2], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, wd16, K / 32, E * N, K / 16,
                         8, kBM, false));
    } else {
        H32_TRY(make_map(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, wp, K, E * N, K, 128, kBM,
                         true));
        H32_TRY(make_map(&maps[2], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, wsc, ldws, E * N, ldws * 4,
                         4, kBM, false));
    }
    const int64_t xrow = K * (xbits / 4);   // activation bytes per row
    H32_TRY(make_map(&maps[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, xw, xrow, M, xrow, 128, bn, true));
    H32_TRY(make_map(&maps[3], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, xdt, ldxd, K / 32, ldxd * 4, bn, 4,
                     false));
    TcArgs a{};
    a.y = y;
    a.bsum = block_sums;
    a.expert_off = expert_off;
    a.ldy = ldy;
    a.qn = qn;
    a.qnd = qnd;
    a.ldqnd = ldqnd;
    a.qn_rot = qn_rot;
    a.M = static_cast<int32_t>(M);
    a.N = static_cast<int32_t>(N);
    a.nb = static_cast<int32_t>(K / 32);
    a.bn = bn;
    a.E = static_cast<int32_t>(E);
    a.tail_first = static_cast<int32_t>(plan.tail_first);
    a.tail_k = plan.tail_k;
    if (plan.split_p > 0) {
        // the planner splits only with a workspace of the plan's size (checked above)
        if (!ws) return H32_ERR_INVALID_ARG;
        uint8_t *w = static_cast<uint8_t *>(ws);
        a.ws_hdr = reinterpret_cast<unsigned long long *>(w);
        a.ws_flag = reinterpret_cast<unsigned long long *>(w + kSplitFlagOff);
        a.ws_acc = reinterpret_cast<float *>(w + kSplitAccOff);
        a.split_p = static_cast<int32_t>(plan.split_p);
        a.split_kh = static_cast<int32_t>(plan.split_kh);
        a.ws_ld = static_cast<int32_t>(plan.ws_ld);
    }
    a.wait_limit = wait_limit();
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int g = static_cast<int>(grid);
    if (wd16) {
        if (block_sums) return launch_tc<4, 4, 1, false, true>(maps, a, g, s);
        return plan.tail_k > 1 ? launch_tc<4, 4, 0, true, true>(maps, a, g, s)
                               : launch_tc<4, 4, 0, false, true>(maps, a, g, s);
    }
    if (xbits == 8) {
        if (block_sums) return launch_tc<H32_TC_EPI_PER_QUAD, 8, 1>(maps, a, g, s);
        if (plan.split_p > 0) return launch_tc<H32_TC_EPI_PER_QUAD, 8, 0, true, false, true>(maps, a, g, s);
        return plan.tail_k > 1 ? launch_tc<H32_TC_EPI_PER_QUAD, 8, 0, true>(maps, a, g, s)
                               : launch_tc<H32_TC_EPI_PER_QUAD, 8, 0>(maps, a, g, s);
    }
    if (qn) {
        if (plan.split_p > 0) return launch_tc<H32_TC_EPI_PER_QUAD, 4, 2, true, false, true>(maps, a, g, s);
        return plan.tail_k > 1 ? launch_tc<H32_TC_EPI_PER_QUAD, 4, 2, true>(maps, a, g, s)
                               : launch_tc<H32_TC_EPI_PER_QUAD, 4, 2>(maps, a, g, s);
    }
    if (block_sums) return launch_tc<H32_TC_EPI_PER_QUAD, 4, 1>(maps, a, g, s);
    // the tile's 16-column chunks in even shares: 12 epilogue warps (3 per lane
    // quarter) when 16 would leave one warp with twice the others' chunks
    // (5 or 6 chunks: measured 5-8% faster on the pp512 attention and FFN-down
    // shapes), 16 otherwise
    const int n16 = bn / 16;
    const bool narrow = n16 % 4 == 1 || n16 % 4 == 2;
    if (plan.split_p > 0)
        return narrow ? launch_tc<3, 4, 0, true, false, true>(maps, a, g, s)
                      : launch_tc<H32_TC_EPI_PER_QUAD, 4, 0, true, false, true>(maps, a, g, s);
    if (plan.tail_k > 1)
        return narrow ? launch_tc<3, 4, 0, true>(maps, a, g, s)
                      : launch_tc<H32_TC_EPI_PER_QUAD, 4, 0, true>(maps, a, g, s);
    if (narrow) return launch_tc<3, 4, 0>(maps, a, g, s);
    return launch_tc<H32_TC_EPI_PER_QUAD, 4, 0>(maps, a, g, s);
}

}  // namespace
}  // namespace h32

extern "C" h32_status q4_0_x_q4_gemm_tc(const uint8_t *wp, const float *wsc, int64_t ldws,
                                        const uint8_t *xw, const float *xdt, int64_t ldxd,
                                        int64_t M, int64_t N, int64_t K, float *y, int64_t ldy,
                                        int32_t *block_sums, void *stream) {
    return h32::run_gemm_tc(4, wp, wsc, ldws, 1, xw, xdt, ldxd, nullptr, M, N, K, y, ldy,
                            block_sums, stream);
}

extern "C" h32_status h32_gemm_tc_schedule(int64_t M, int64_t N, int64_t K, int32_t sms,
                                           int32_t with_workspace, int64_t *out) {
    if (!out || sms < 1 || M < 1 || N <= 0 || K <= 0 || (K % 128) != 0 || (N % 16) != 0 ||
        M > 0x7FFFFFFFll || N > 0x7FFFFFFFll || K > 0x7FFFFFFFll ||
        ((N + 127) / 128) * ((M + 15) / 16) * 8 > 0x7FFFFFFFll)
        return H32_ERR_INVALID_ARG;
    const h32::TcPlan p = h32::plan_tc(M, N, sms, true, with_workspace != 0, K / 128);
    const int64_t v[9] = {p.bn, p.tail_k, p.tail_first, p.total, p.grid,
                          p.split_p, p.split_kh, p.ws_ld,
                          static_cast<int64_t>(h32::split_ws_bytes(p))};
    for (int i = 0; i < 9; ++i) out[i] = v[i];
    return H32_OK;
}

extern "C" h32_status h32_gemm_tc_workspace_bytes(int64_t M, int64_t N, int64_t K, size_t *bytes) {
    if (!bytes) return H32_ERR_INVALID_ARG;
    *bytes = 0;
    if (M < 0 || N <= 0 || K <= 0 || (K % 128) != 0 || (N % 16) != 0 || M > 0x7FFFFFFFll ||
        N > 0x7FFFFFFFll || K > 0x7FFFFFFFll || ((N + 127) / 128) * ((M + 15) / 16) * 8 > 0x7FFFFFFFll)
        return H32_ERR_INVALID_ARG;
    if (M == 0) return H32_OK;
    int sms = 0;
    H32_TRY(h32::check_device(&sms));
    *bytes = h32::split_ws_bytes(h32::plan_tc(M, N, sms, true, true, K / 128));
    return H32_OK;
}

extern "C" h32_status q4_0_x_q4_gemm_tc_ws(const uint8_t *wp, const float *wsc, int64_t ldws,
                                           const uint8_t *xw, const float *xdt, int64_t ldxd,
                                           int64_t M, int64_t N, int64_t K, float *y, int64_t ldy,
                                           int32_t *block_sums, void *workspace,
                                           size_t workspace_bytes, void *stream) {
    return h32::run_gemm_tc(4, wp, wsc, ldws, 1, xw, xdt, ldxd, nullptr, M, N, K, y, ldy,
                            block_sums, stream, nullptr, nullptr, 0, 0, nullptr, workspace,
                            workspace_bytes);
}

extern "C" h32_status q4_0_x_q8_gemm_tc_ws(const uint8_t *wp, const float *wsc, int64_t ldws,
                                           const uint8_t *xw8, const float *xdt, int64_t ldxd,
                                           int64_t M, int64_t N, int64_t K, float *y, int64_t ldy,
                                           int32_t *block_sums, void *workspace,
                                           size_t workspace_bytes, void *stream) {
    return h32::run_gemm_tc(8, wp, wsc, ldws, 1, xw8, xdt, ldxd, nullptr, M, N, K, y, ldy,
                            block_sums, stream, nullptr, nullptr, 0, 0, nullptr, workspace,
                            workspace_bytes);
}

// The no-alloc entry points' workspace: one static array per device, zero at
// module load (a valid workspace), never allocated or freed by a call.
namespace h32 {
namespace {
constexpr size_t kStaticWsBytes = 4u << 20;
__device__ __align__(256) uint8_t g_tc_static_ws[kStaticWsBytes];

h32_status static_workspace(void **ptr) {
    static std::mutex mu;
    static void *addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return H32_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        const cudaError_t e = cudaGetSymbolAddress(&addr[dev], g_tc_static_ws);
        if (e != cudaSuccess) return launch_status(e);
    }
    *ptr = addr[dev];
    return H32_OK;
}

h32_status run_noalloc(int xbits, const uint8_t *wp, const float *wsc, int64_t ldws,
                       const uint8_t *xw, const float *xdt, int64_t ldxd, int64_t M, int64_t N,
                       int64_t K, float *y, int64_t ldy, int32_t *block_sums, void *stream) {
    size_t need = 0;
    if (!block_sums) {
        const h32_status st = h32_gemm_tc_workspace_bytes(M, N, K, &need);
        if (st != H32_OK) return st;
    }
    if (need > kStaticWsBytes) return H32_ERR_UNSUPPORTED;   // never allocates
    void *ws = nullptr;
    if (need > 0) H32_TRY(static_workspace(&ws));
    return run_gemm_tc(xbits, wp, wsc, ldws, 1, xw, xdt, ldxd, nullptr, M, N, K, y, ldy,
                       block_sums, stream, nullptr, nullptr, 0, 0, nullptr, ws,
                       need > 0 ? kStaticWsBytes : 0);
}
}  // namespace
}  // namespace h32

extern "C" h32_status q4_0_x_q4_gemm_tc_noalloc(const uint8_t *wp, const float *wsc, int64_t ldws,
                                                const uint8_t *xw, const float *xdt, int64_t ldxd,
                                                int64_t M, int64_t N, int64_t K, float *y,
                                                int64_t ldy, int32_t *block_sums, void *stream) {
    return h32::run_noalloc(4, wp, wsc, ldws, xw, xdt, ldxd, M, N, K, y, ldy, block_sums, stream);
}

extern "C" h32_status q4_0_x_q8_gemm_tc_noalloc(const uint8_t *wp, const float *wsc, int64_t ldws,
                                                const uint8_t *xw8, const float *xdt, int64_t ldxd,
                                                int64_t M, int64_t N, int64_t K, float *y,
                                                int64_t ldy, int32_t *block_sums, void *stream) {
    return h32::run_noalloc(8, wp, wsc, ldws, xw8, xdt, ldxd, M, N, K, y, ldy, block_sums, stream);
}

extern "C" h32_status q4_0_x_q4_gemm_tc_quant_next(const uint8_t *wp, const float *wsc,
                                                   int64_t ldws, const uint8_t *xw,
                                                   const float *xdt, int64_t ldxd, int64_t M,
                                                   int64_t N, int64_t K, float *y, int64_t ldy,
                                                   uint8_t *xw_next, float *xdt_next,
                                                   int64_t ldxd_next, int rotate_next,
                                                   void *stream) {
    if (!xw_next) return H32_ERR_INVALID_ARG;
    return h32::run_gemm_tc(4, wp, wsc, ldws, 1, xw, xdt, ldxd, nullptr, M, N, K, y, ldy, nullptr,
                            stream, xw_next, xdt_next, ldxd_next, rotate_next);
}

extern "C" h32_status q4_0_x_q4_gemm_tc_quant_next_ws(const uint8_t *wp, const float *wsc,
                                                      int64_t ldws, const uint8_t *xw,
                                                      const float *xdt, int64_t ldxd, int64_t M,
                                                      int64_t N, int64_t K, float *y, int64_t ldy,
                                                      uint8_t *xw_next, float *xdt_next,
                                                      int64_t ldxd_next, int rotate_next,
                                                      void *workspace, size_t workspace_bytes,
                                                      void *stream) {
    if (!xw_next) return H32_ERR_INVALID_ARG;
    return h32::run_gemm_tc(4, wp, wsc, ldws, 1, xw, xdt, ldxd, nullptr, M, N, K, y, ldy, nullptr,
                            stream, xw_next, xdt_next, ldxd_next, rotate_next, nullptr, workspace,
                            workspace_bytes);
}

extern "C" h32_status q4_0_x_q4_gemm_tc_widen(const uint8_t *wq, const uint16_t *wd,
                                              const uint8_t *xw, const float *xdt, int64_t ldxd,
                                              int64_t M, int64_t N, int64_t K, float *y,
                                              int64_t ldy, int32_t *block_sums, void *stream) {
    if (!wd) return H32_ERR_INVALID_ARG;
    return h32::run_gemm_tc(4, wq, nullptr, 0, 1, xw, xdt, ldxd, nullptr, M, N, K, y, ldy,
                            block_sums, stream, nullptr, nullptr, 0, 0, wd);
}

extern "C" h32_status q4_0_x_q4_gemm_tc_widen_experts(const uint8_t *wq, const uint16_t *wd,
                                                      int32_t E, const uint8_t *xw,
                                                      const float *xdt, int64_t ldxd,
                                                      const int32_t *expert_off, int64_t R,
                                                      int64_t N, int64_t K, float *y, int64_t ldy,
                                                      int32_t *block_sums, void *stream) {
    if (!wd || !expert_off) return H32_ERR_INVALID_ARG;
    return h32::run_gemm_tc(4, wq, nullptr, 0, E, xw, xdt, ldxd, expert_off, R, N, K, y, ldy,
                            block_sums, stream, nullptr, nullptr, 0, 0, wd);
}

extern "C" h32_status q4_0_x_q8_gemm_tc(const uint8_t *wp, const float *wsc, int64_t ldws,
                                        const uint8_t *xw8, const float *xdt, int64_t ldxd,
                                        int64_t M, int64_t N, int64_t K, float *y, int64_t ldy,
                                        int32_t *block_sums, void *stream) {
    return h32::run_gemm_tc(8, wp, wsc, ldws, 1, xw8, xdt, ldxd, nullptr, M, N, K, y, ldy,
                            block_sums, stream);
}

extern "C" h32_status q4_0_x_q4_gemm_tc_experts(const uint8_t *wp, const float *wsc, int64_t ldws,
                                                int32_t E, const uint8_t *xw, const float *xdt,
                                                int64_t ldxd, const int32_t *expert_off, int64_t R,
                                                int64_t N, int64_t K, float *y, int64_t ldy,
                                                int32_t *block_sums, void *stream) {
    if (!expert_off) return H32_ERR_INVALID_ARG;
    return h32::run_gemm_tc(4, wp, wsc, ldws, E, xw, xdt, ldxd, expert_off, R, N, K, y, ldy,
                            block_sums, stream);
}
