// Routing and weighted combine around the expert-batched GEMM (sm_103a).
//
// "Where the engine is going: HRX and the NPU", section "4-bit activations
// reach the MoE experts": the Hadamard route covers the expert matmuls of a
// mixture-of-experts model.  These kernels are the layer around those
// matmuls: pick each token's experts and weights from its router logits,
// group the (token, expert) rows by expert for the grouped GEMM, and add a
// token's expert outputs back together.  The pages leave the router open;
// the reading taken here: the k largest logits (ties to the lower expert id),
// listed by decreasing logit; weights = softmax over those k logits (the full
// softmax's top-k probabilities renormalised to sum to 1); rows grouped by
// expert, then by token; the combine sums a token's rows in choice order with
// fp32 fma from +0.
//
// Every result is deterministic: no atomics decide an order.
//   route_topk_kernel   one warp per token: k rounds of a warp-wide argmax
//                       over the logits held in registers, then the weights
//   route_group_kernel  one block per expert: its offset is the number of
//                       choices of lower experts; its rows are the tokens
//                       that chose it, in token order (ballot prefix sums)
//   combine_kernel      one block per token (x) and 128 float4 columns (y): 16-byte
//                       loads of the token's k rows, fma in choice order
#include "h32_common.cuh"

namespace h32 {
namespace {

__device__ uint32_t g_moe_status;   // kStatusGuard: a combine row index out of range

constexpr int kMaxE = 1024;         // experts a router call handles
constexpr int kMaxK = 32;           // choices per token (one lane each)
constexpr int kTopkWarps = 8;       // tokens per block of route_topk_kernel
constexpr int kGroupThreads = 1024;
constexpr int kCombineThreads = 128;   // one float4 column each

// (value, id) a beats b: larger value, or equal value and lower id; a NaN
// ranks below every number (-inf included), NaNs among themselves by id;
// id < 0 = none
__device__ __forceinline__ bool beats(float va, int ia, float vb, int ib) {
    if (ia < 0) return false;
    if (ib < 0) return true;
    const bool na = isnan(va), nb = isnan(vb);
    if (na || nb) return (na && nb) ? ia < ib : nb;
    return va > vb || (va == vb && ia < ib);
}

// Unnormalised weight of a chosen logit l given the largest chosen logit
// lmax: exp(l - lmax) when lmax is finite (0 for a chosen -inf or NaN); when
// lmax = +inf, 1 for the +inf choices and 0 for the others; when lmax is -inf
// or NaN (every logit masked), 1: equal weights.  These are the limits of the
// softmax over the chosen logits.
__device__ __forceinline__ float unnormalised_weight(float l, float lmax) {
    if (isfinite(lmax)) return isnan(l) ? 0.0f : expf(__fsub_rn(l, lmax));
    if (lmax > 0.0f) return l == lmax ? 1.0f : 0.0f;
    return 1.0f;
}

// NPER: logits per lane (expert lane + 32 i, i < NPER), a power of two >= E / 32
template <int NPER>
__global__ void __launch_bounds__(kTopkWarps * 32)
    route_topk_kernel(const float *__restrict__ logits, int T, int E, int64_t ldl, int k,
                      int32_t *__restrict__ topk_id, float *__restrict__ topk_w) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kTopkWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const float *row = logits + t * ldl;
    float v[NPER];
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? row[e] : 0.0f;
    }
    uint32_t taken = 0;   // bit i: expert lane + 32 i already chosen
    int my_id = -1;       // lane j keeps choice j
    float my_v = 0.0f;
    for (int j = 0; j < k; ++j) {
        float bv = 0.0f;
        int bi = -1;
#pragma unroll
        for (int i = 0; i < NPER; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u) && beats(v[i], e, bv, bi)) {
                bv = v[i];
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
            const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
            if (beats(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == j) {
            my_id = bi;
            my_v = bv;
        }
    }
    // weights: exp of each chosen logit minus the largest, their sum in choice
    // order from +0, one IEEE divide each
    const float lmax = __shfl_sync(0xFFFFFFFFu, my_v, 0);
    const float ex = (lane < k) ? unnormalised_weight(my_v, lmax) : 0.0f;
    float s = 0.0f;
    for (int j = 0; j < k; ++j) s = __fadd_rn(s, __shfl_sync(0xFFFFFFFFu, ex, j));
    if (lane < k) {
        topk_id[t * k + lane] = my_id;
        topk_w[t * k + lane] = __fdiv_rn(ex, s);
    }
}

// exclusive prefix of `flag` over the block's threads in thread order, and the
// block's total (all threads get it); warp_tot is shared memory, one int per warp
__device__ __forceinline__ int block_prefix(bool flag, int *warp_tot, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, flag);
    if (lane == 0) warp_tot[warp] = __popc(bal);
    __syncthreads();
    int before = 0, all = 0;
    for (int w = 0; w < kGroupThreads / 32; ++w) {
        const int c = warp_tot[w];
        if (w < warp) before += c;
        all += c;
    }
    __syncthreads();
    *total = all;
    return before + __popc(bal & ((1u << lane) - 1u));
}

__global__ void __launch_bounds__(kGroupThreads)
    route_group_kernel(const int32_t *__restrict__ topk_id, int T, int E, int k,
                       int32_t *__restrict__ expert_off, int32_t *__restrict__ row_idx,
                       int32_t *__restrict__ row_of) {
    __shared__ int red[2][kGroupThreads / 32];
    __shared__ int warp_tot[kGroupThreads / 32];
    pdl_wait();
    pdl_trigger();
    const int e = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t n = static_cast<int64_t>(T) * k;
    // choices of lower experts (this expert's first row) and of this expert;
    // 16-byte loads (topk_id is 16-byte aligned), independent within a thread
    int lt = 0, eq = 0;
    const int64_t n4 = n / 4;
    const int4 *id4 = reinterpret_cast<const int4 *>(topk_id);
#pragma unroll 4
    for (int64_t i = threadIdx.x; i < n4; i += kGroupThreads) {
        const int4 q = id4[i];
        lt += (q.x < e) + (q.y < e) + (q.z < e) + (q.w < e);
        eq += (q.x == e) + (q.y == e) + (q.z == e) + (q.w == e);
    }
    for (int64_t i = 4 * n4 + threadIdx.x; i < n; i += kGroupThreads) {
        const int id = topk_id[i];
        lt += id < e;
        eq += id == e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        lt += __shfl_xor_sync(0xFFFFFFFFu, lt, o);
        eq += __shfl_xor_sync(0xFFFFFFFFu, eq, o);
    }
    if (lane == 0) {
        red[0][warp] = lt;
        red[1][warp] = eq;
    }
    __syncthreads();
    int first = 0, count = 0;
    for (int w = 0; w < kGroupThreads / 32; ++w) {
        first += red[0][w];
        count += red[1][w];
    }
    if (threadIdx.x == 0) {
        expert_off[e] = first;
        if (e == E - 1) expert_off[E] = first + count;
    }
    // this expert's rows: the tokens that chose it, in token order
    int base = first;
    for (int64_t t0 = 0; t0 < T; t0 += kGroupThreads) {
        const int64_t t = t0 + threadIdx.x;
        int j = -1;
        if (t < T) {
            const int32_t *ids = topk_id + t * k;
#pragma unroll 8
            for (int c = 0; c < k; ++c)
                if (ids[c] == e) j = c;
        }
        int tot;
        const int pos = block_prefix(j >= 0, warp_tot, &tot);
        if (j >= 0) {
            const int r = base + pos;
            row_idx[r] = static_cast<int32_t>(t);
            row_of[t * k + j] = r;
        }
        base += tot;
    }
}

__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const float *__restrict__ y, int64_t R, int64_t ldy,
                   const int32_t *__restrict__ row_of, const float *__restrict__ topk_w, int k,
                   int64_t H, float *__restrict__ out, int64_t ldo) {
    __shared__ int64_t s_row[kMaxK];
    __shared__ float s_w[kMaxK];
    pdl_wait();
    pdl_trigger();
    const int64_t t = blockIdx.x;
    if (threadIdx.x < k) {
        int64_t r = row_of[t * k + threadIdx.x];
        if (r < 0 || r >= R) {
            atomicOr(&g_moe_status, kStatusGuard);
            r = -1;
        }
        s_row[threadIdx.x] = r;
        s_w[threadIdx.x] = topk_w[t * k + threadIdx.x];
    }
    __syncthreads();
    const int64_t c = static_cast<int64_t>(blockIdx.y) * kCombineThreads + threadIdx.x;
    if (c >= H / 4) return;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    // the loads of several rows are in flight together; the fmas stay in order
#pragma unroll 8
    for (int j = 0; j < k; ++j) {
        const int64_t r = s_row[j];
        if (r < 0) continue;   // a guarded index adds nothing
        const float w = s_w[j];
        const float4 v = __ldg(reinterpret_cast<const float4 *>(y + r * ldy) + c);
        acc.x = __fmaf_rn(w, v.x, acc.x);
        acc.y = __fmaf_rn(w, v.y, acc.y);
        acc.z = __fmaf_rn(w, v.z, acc.z);
        acc.w = __fmaf_rn(w, v.w, acc.w);
    }
    reinterpret_cast<float4 *>(out + t * ldo)[c] = acc;
}

}  // namespace

__device__ uint32_t g_moe_status_taken;
__global__ void take_g_moe_status() { g_moe_status_taken = atomicExch(&g_moe_status, 0u); }

h32_status moe_read_and_clear_status(cudaStream_t s) {
    bool ok = false;
    const uint32_t v = take_status(take_g_moe_status, g_moe_status_taken, s, &ok);
    if (!ok) return H32_ERR_CUDA;
    return (v & kStatusGuard) ? H32_ERR_DEVICE_GUARD : H32_OK;
}

}  // namespace h32

extern "C" h32_status h32_moe_route(const float *logits, int64_t T, int32_t E, int64_t ldl,
                                    int32_t k, int32_t *topk_id, float *topk_w,
                                    int32_t *expert_off, int32_t *row_idx, int32_t *row_of,
                                    void *stream) {
    using namespace h32;
    if (T < 0 || E < 1 || E > kMaxE || k < 1 || k > kMaxK || k > E || ldl < E || !expert_off)
        return H32_ERR_INVALID_ARG;
    if (T * k > 0x7FFFFFFFll) return H32_ERR_INVALID_ARG;
    if (T > 0 && (!logits || !topk_id || !topk_w || !row_idx || !row_of))
        return H32_ERR_INVALID_ARG;
    if ((logits && (reinterpret_cast<uintptr_t>(logits) & 3u)) ||
        (reinterpret_cast<uintptr_t>(expert_off) & 3u) || (topk_id && !aligned16(topk_id)) ||
        (topk_w && (reinterpret_cast<uintptr_t>(topk_w) & 3u)) ||
        (row_idx && (reinterpret_cast<uintptr_t>(row_idx) & 3u)) ||
        (row_of && (reinterpret_cast<uintptr_t>(row_of) & 3u)))
        return H32_ERR_ALIGNMENT;
    H32_TRY(check_device(nullptr));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int t32 = static_cast<int>(T);
    if (T > 0) {
        const dim3 grid(static_cast<unsigned>((T + kTopkWarps - 1) / kTopkWarps));
        const dim3 block(kTopkWarps * 32);
        const int ei = static_cast<int>(E), ki = static_cast<int>(k);
        cudaError_t e1;
        if (E <= 32)
            e1 = launch_pdl(route_topk_kernel<1>, grid, block, 0, s, logits, t32, ei, ldl, ki, topk_id, topk_w);
        else if (E <= 64)
            e1 = launch_pdl(route_topk_kernel<2>, grid, block, 0, s, logits, t32, ei, ldl, ki, topk_id, topk_w);
        else if (E <= 128)
            e1 = launch_pdl(route_topk_kernel<4>, grid, block, 0, s, logits, t32, ei, ldl, ki, topk_id, topk_w);
        else if (E <= 256)
            e1 = launch_pdl(route_topk_kernel<8>, grid, block, 0, s, logits, t32, ei, ldl, ki, topk_id, topk_w);
        else if (E <= 512)
            e1 = launch_pdl(route_topk_kernel<16>, grid, block, 0, s, logits, t32, ei, ldl, ki, topk_id, topk_w);
        else
            e1 = launch_pdl(route_topk_kernel<32>, grid, block, 0, s, logits, t32, ei, ldl, ki, topk_id, topk_w);
        if (e1 != cudaSuccess) return launch_status(e1);
    }
    // with T = 0 this writes all-zero offsets
    const cudaError_t e2 = launch_pdl(route_group_kernel, dim3(E), dim3(kGroupThreads), 0, s,
                                      static_cast<const int32_t *>(topk_id), t32,
                                      static_cast<int>(E), static_cast<int>(k), expert_off,
                                      row_idx, row_of);
    return launch_status(e2 != cudaSuccess ? e2 : cudaGetLastError());
}

extern "C" h32_status h32_moe_combine(const float *y, int64_t R, int64_t ldy, const int32_t *row_of,
                                      const float *topk_w, int64_t T, int32_t k, int64_t H,
                                      float *out, int64_t ldo, void *stream) {
    using namespace h32;
    if (T < 0 || R < 0 || k < 1 || k > kMaxK || H <= 0 || (H % 4) != 0 || ldy < H || ldo < H)
        return H32_ERR_INVALID_ARG;
    if (T == 0) return H32_OK;
    if (!y || !row_of || !topk_w || !out || T > 0x7FFFFFFFll) return H32_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned16(out) || (ldy % 4) != 0 || (ldo % 4) != 0 ||
        (reinterpret_cast<uintptr_t>(row_of) & 3u) || (reinterpret_cast<uintptr_t>(topk_w) & 3u))
        return H32_ERR_ALIGNMENT;
    H32_TRY(check_device(nullptr));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t col_blocks = (H / 4 + kCombineThreads - 1) / kCombineThreads;
    if (col_blocks > 65535) return H32_ERR_INVALID_ARG;
    const dim3 grid(static_cast<unsigned>(T), static_cast<unsigned>(col_blocks));
    const cudaError_t e = launch_pdl(combine_kernel, grid, dim3(kCombineThreads), 0, s, y, R, ldy,
                                     row_of, topk_w, static_cast<int>(k), H, out, ldo);
    return launch_status(e != cudaSuccess ? e : cudaGetLastError());
}
