// Rotate + quantize kernels of the Hadamard route (sm_103a).
//
//  * h32_quantize_act_q4 / _q8: the activation quantizer of "509 tokens a
//    second of prompt: the Hadamard route ships", section "The rotation":
//    each block of 32 activations is rotated by the 32-point Walsh-Hadamard
//    transform and rounded to 4-bit codes with one fp32 scale (8-bit codes on
//    the exact route of "Prompt processing: 4-bit activations, rotated
//    first").
//  * h32_rotate_quantize_weights_q4_0: the offline weight step of "Making the
//    file is part of the engine" (rotate the projections, quantize to Q4_0).
//
// Layout on the device: one thread owns one whole 32-block.  It loads the
// block with 128-bit loads, runs all five butterfly stages (strides 1, 2, 4,
// 8, 16) in registers, takes the block's amax, one IEEE divide and one IEEE
// reciprocal, and writes the packed codes with one 128-bit store (4-bit) or
// two (8-bit).  Adjacent lanes own adjacent blocks, so each warp's stores are
// contiguous.  The pages run the rotation as two in-thread butterfly steps
// and three lane shuffles on a 32-wide AMD wave; owning the whole block in one
// thread removes the shuffles and the per-lane redundant divide, which keeps
// the kernel's instruction count under the HBM roofline on GB300.
//
// Rounding: every add, multiply, divide and reciprocal is IEEE round-to-
// nearest-even (explicit _rn intrinsics; the library is built without
// fast-math and with denormals kept), so codes and scales are bit-identical
// to a plain sequential fp32 evaluation of the same steps.
#include <cuda_fp16.h>

#include "h32_common.cuh"
#include "h32_tcform.cuh"

namespace h32 {
namespace {

__device__ uint32_t g_quant_status;   // kStatusGuard: a gathered row index out of range


// ----------------------------------------------------------------------------
// loading one block as 32 fp32 values
// ----------------------------------------------------------------------------
__device__ __forceinline__ void load_block_bf16(const uint16_t *__restrict__ p, float (&v)[32]) {
    const uint4 *q = reinterpret_cast<const uint4 *>(p);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint4 u = __ldg(q + c);
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[8 * c + 2 * i] = __uint_as_float(w[i] << 16);
            v[8 * c + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
}

__device__ __forceinline__ void load_block_f32(const float *__restrict__ p, float (&v)[32]) {
    const float4 *q = reinterpret_cast<const float4 *>(p);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        float4 f = __ldg(q + c);
        v[4 * c] = f.x;
        v[4 * c + 1] = f.y;
        v[4 * c + 2] = f.z;
        v[4 * c + 3] = f.w;
    }
}

// ----------------------------------------------------------------------------
// the rotation: butterfly with strides 1, 2, 4, 8, 16, then the 1/sqrt(32) scale
// ----------------------------------------------------------------------------
// The kRot-point rotation (0 = none, 32, 64, 128) of the thread's 32-block,
// which is 32-block `pos` (0 .. kRot/32 - 1) of its kRot-block.  The other
// 32-blocks of the kRot-block are held by the lanes that differ from this one
// in the low bits pos covers (lane ^ 1, lane ^ 2); those lanes are in `mask`.
// Strides 32 and 64 pair element i of two blocks: the lower block takes
// a + c, the upper a - c (a the lower block's value), as in strides 1..16.
template <int kRot>
__device__ __forceinline__ void rotate_block(float (&v)[32], uint32_t pos, unsigned mask) {
    if constexpr (kRot == 32) {
        rotate32(v);
    } else if constexpr (kRot > 32) {
        butterfly32(v);
#pragma unroll
        for (int hb = 1; hb < kRot / 32; hb <<= 1) {
            const bool lower = (pos & hb) == 0;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float c = __shfl_xor_sync(mask, v[i], hb);
                v[i] = lower ? __fadd_rn(v[i], c) : __fsub_rn(c, v[i]);
            }
        }
        const float sc = (kRot == 64) ? 0.125f : kInvSqrt128;
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(v[i], sc);
    }
}

// the rotate argument of the entry points: 0 = none, 1 or 32, 64, 128 points
// (-1 = not supported)
int rot_points(int rotate) {
    return rotate == 0 ? 0 : rotate == 1 || rotate == 32 ? 32 : rotate == 64 ? 64
         : rotate == 128 ? 128 : -1;
}

// low byte of each of four words -> one word
__device__ __forceinline__ uint32_t pack_low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    const uint32_t ab = __byte_perm(a, b, 0x0040);
    const uint32_t cd = __byte_perm(c, d, 0x0040);
    return __byte_perm(ab, cd, 0x5410);
}

// ----------------------------------------------------------------------------
// activation quantizer
// ----------------------------------------------------------------------------
template <bool kBf16, int kBits, int kRot>
__global__ void __launch_bounds__(256) quant_act_kernel(const void *__restrict__ x, uint32_t nblk,
                                                       uint32_t nb, int64_t ldx,
                                                       uint8_t *__restrict__ xq,
                                                       float *__restrict__ xd) {
    constexpr float kQmax = (kBits == 4) ? 7.0f : 127.0f;
    constexpr float kQmin = (kBits == 4) ? -8.0f : -127.0f;
    // block g = row * nb + b; the grid stride is split once into whole rows
    // and a remainder so the walk needs no division per block
    const uint32_t stride = gridDim.x * blockDim.x;
    const uint32_t srow = stride / nb, sb = stride % nb;
    uint32_t g = blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t row = g / nb, b = g % nb;
    for (; g < nblk; g += stride) {
        const unsigned mask = __activemask();
        float v[32];
        if constexpr (kBf16) {
            load_block_bf16(reinterpret_cast<const uint16_t *>(x) + int64_t(row) * ldx + 32 * b, v);
        } else {
            load_block_f32(reinterpret_cast<const float *>(x) + int64_t(row) * ldx + 32 * b, v);
        }
        // the kRot/32 blocks of a kRot-block sit in adjacent lanes: nb, the
        // grid stride and nblk are multiples of kRot/32
        rotate_block<kRot>(v, b, mask);

        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
        const float d = __fdiv_rn(amax, kQmax);
        const float id = (d != 0.0f) ? __frcp_rn(d) : 0.0f;

        // codes: round-half-even(y * id).  With a finite amax and a finite id
        // every product lies in [-qmax, qmax] up to rounding; when 1/d
        // overflowed (a block of subnormal size) or the rotation itself
        // overflowed to +-inf, the code is the clamped y / d instead
        uint32_t bits[32];
        if (!(amax < INFINITY) || isinf(id)) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                bits[i] = __float_as_uint(__fadd_rn(degenerate_code(v[i], d, kQmin, kQmax),
                                                    kRoundMagic));
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                bits[i] = __float_as_uint(__fadd_rn(__fmul_rn(v[i], id), kRoundMagic));
        }

        if constexpr (kBits == 4) {
            // Q4_0 nibble order: byte j = element j (low) | element j + 16 (high)
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t lo =
                    pack_low_bytes(bits[4 * k], bits[4 * k + 1], bits[4 * k + 2], bits[4 * k + 3]);
                const uint32_t hi = pack_low_bytes(bits[16 + 4 * k], bits[17 + 4 * k],
                                                   bits[18 + 4 * k], bits[19 + 4 * k]);
                w[k] = (lo & 0x0F0F0F0Fu) | ((hi << 4) & 0xF0F0F0F0u);
            }
            *reinterpret_cast<uint4 *>(xq + (int64_t(g) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                w[k] = pack_low_bytes(bits[4 * k], bits[4 * k + 1], bits[4 * k + 2], bits[4 * k + 3]);
            uint4 *dst = reinterpret_cast<uint4 *>(xq + (int64_t(g) << 5));
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
        xd[g] = d;
        row += srow;
        b += sb;
        if (b >= nb) {
            b -= nb;
            ++row;
        }
    }
}

// ----------------------------------------------------------------------------
// offline weights: rotate, then the Q4_0 rule
// ----------------------------------------------------------------------------
template <int kRot>
__global__ void __launch_bounds__(256) quant_w_kernel(const float *__restrict__ w, uint32_t nblk,
                                                     uint8_t *__restrict__ wq,
                                                     uint16_t *__restrict__ wd) {
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t g = blockIdx.x * blockDim.x + threadIdx.x; g < nblk; g += stride) {
        const unsigned mask = __activemask();
        float v[32];
        load_block_f32(w + int64_t(g) * 32, v);
        rotate_block<kRot>(v, g, mask);   // g = row * nb + b with nb a multiple of kRot/32
        // signed value of largest magnitude, first one on ties
        float amax = 0.0f, mx = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float a = fabsf(v[i]);
            if (a > amax) {
                amax = a;
                mx = v[i];
            }
        }
        const float d = __fdiv_rn(mx, -8.0f);
        const float id = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
        // a degenerate block (1/d overflows, or the rotation overflowed): the
        // code from y / d by an IEEE divide, inf / inf read as its limit
        // (-8 where y has the sign of the signed maximum, else +8)
        const bool degen = isinf(id) || !(amax < INFINITY);
        uint32_t c[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            float u;
            if (!degen) {
                u = __fadd_rn(__fmul_rn(v[i], id), 8.5f);
            } else {
                float t = __fdiv_rn(v[i], d);
                if (isnan(t)) t = ((__float_as_uint(v[i]) ^ __float_as_uint(mx)) >> 31) ? 8.0f : -8.0f;
                u = __fadd_rn(t, 8.5f);
            }
            u = fminf(fmaxf(u, 0.0f), 15.0f);
            c[i] = static_cast<uint32_t>(__float2int_rz(u));
        }
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t lo = pack_low_bytes(c[4 * k], c[4 * k + 1], c[4 * k + 2], c[4 * k + 3]);
            const uint32_t hi =
                pack_low_bytes(c[16 + 4 * k], c[17 + 4 * k], c[18 + 4 * k], c[19 + 4 * k]);
            o[k] = lo | (hi << 4);
        }
        *reinterpret_cast<uint4 *>(wq + (int64_t(g) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        wd[g] = __half_as_ushort(__float2half_rn(d));
    }
}

// Rotate + quantize to 4-bit (or 8-bit) codes in tc form.  Each warp walks
// tiles of 4 rows x 8 blocks (measured on a 16384 x 17408 stream: 154 us,
// against 180 us for one row of 32 blocks per warp and 236 us for a block-major
// walk).  With kGather,
// output row r is the quantized input row row_idx[r] (an index outside
// [0, T) records kStatusGuard and yields zero codes and a zero scale).  kE5
// (4-bit only): the codes as the e5m2 bytes of 512 times the code, the
// activation side of the GEMM that widens Q4_0 weights in shared memory.
template <bool kBf16, int kBits, int kRot, bool kGather, bool kE5 = false>
__global__ void __launch_bounds__(256) quant_act_tc_kernel(const void *__restrict__ x, uint32_t nblk,
                                                          uint32_t M, uint32_t K, int64_t ldx,
                                                          const int32_t *__restrict__ row_idx,
                                                          int64_t T, uint8_t *__restrict__ xw,
                                                          float *__restrict__ xdt, int64_t ldxd) {
    // Each warp takes tiles of 4 rows x 8 blocks (lane = 8 r + j): every row
    // segment is 8 blocks read and written contiguously, the 4 scales of a
    // block column land in one 16-byte run of the block-major scale array, and
    // the kRot/32 blocks of a kRot-block sit in adjacent lanes (kRot/32 divides 8).
    (void)nblk;
    pdl_wait();
    pdl_trigger();
    const uint32_t nb = K / 32;
    const uint32_t tiles_b = (nb + 7) / 8, ntiles = ((M + 3) / 4) * tiles_b;
    const uint32_t lane = threadIdx.x & 31;
    const uint32_t nwarps = gridDim.x * (blockDim.x >> 5);
    for (uint32_t wt = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); wt < ntiles;
         wt += nwarps) {
        const uint32_t tr = wt / tiles_b, tb = wt - tr * tiles_b;
        const uint32_t row = tr * 4 + (lane >> 3), b = tb * 8 + (lane & 7);
        const bool in = row < M && b < nb;
        const unsigned mask = __ballot_sync(0xFFFFFFFFu, in);
        if (!in) continue;
        float v[32];
        int64_t src = row;
        bool valid = true;
        if constexpr (kGather) {
            src = __ldg(row_idx + row);
            valid = src >= 0 && src < T;
            if (!valid) {
                atomicOr(&g_quant_status, kStatusGuard);
                src = 0;
            }
        }
        if constexpr (kBf16) {
            load_block_bf16(reinterpret_cast<const uint16_t *>(x) + src * ldx + 32 * b, v);
        } else {
            load_block_f32(reinterpret_cast<const float *>(x) + src * ldx + 32 * b, v);
        }
        if constexpr (kGather) {
            if (!valid) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0.0f;
            }
        }
        rotate_block<kRot>(v, b, mask);
        float d;
        if constexpr (kBits == 4) {
            uint32_t w[8];
            d = quant_block_tc4<kE5>(v, w);
            uint4 *dst = reinterpret_cast<uint4 *>(xw + int64_t(row) * K + 32 * b);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        } else {
            constexpr float kQmax = 127.0f, kQmin = -127.0f;
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
            d = __fdiv_rn(amax, kQmax);
            const float id = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
            uint32_t bits[32];
            if (!(amax < INFINITY) || isinf(id)) {   // degenerate block: the clamped y / d
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    bits[i] = __float_as_uint(__fadd_rn(degenerate_code(v[i], d, kQmin, kQmax),
                                                        kRoundMagic));
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    bits[i] = __float_as_uint(__fadd_rn(__fmul_rn(v[i], id), kRoundMagic));
            }
            // 64 bytes per block: the 32 bytes of 16 h, then the 32 bytes of l
            // integer byte arithmetic here: measured faster than converting floats
            uint32_t wh[8], wl[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                tc_bytes_q8(pack_low_bytes(bits[4 * k], bits[4 * k + 1], bits[4 * k + 2],
                                           bits[4 * k + 3]),
                            wh[k], wl[k]);
            uint4 *dst = reinterpret_cast<uint4 *>(xw + int64_t(row) * 2 * K + 64 * b);
            dst[0] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
            dst[1] = make_uint4(wh[4], wh[5], wh[6], wh[7]);
            dst[2] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
            dst[3] = make_uint4(wl[4], wl[5], wl[6], wl[7]);
        }
        xdt[int64_t(b) * ldxd + row] = d;
    }
}

// Q4_0 -> tc form: e4m3 bytes of q - 8 in element order, scale d widened to fp32
__global__ void __launch_bounds__(256) prepack_w_tc_kernel(const uint8_t *__restrict__ wq,
                                                          const uint16_t *__restrict__ wd,
                                                          uint32_t N, uint32_t nb, uint32_t ldws,
                                                          uint8_t *__restrict__ wp,
                                                          float *__restrict__ wsc) {
    const uint32_t total = N * ldws;
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t g = blockIdx.x * blockDim.x + threadIdx.x; g < total; g += stride) {
        const uint32_t n = g / ldws, b = g - n * ldws;
        if (b >= nb) {
            wsc[g] = 0.0f;
            continue;
        }
        const uint4 q = __ldg(reinterpret_cast<const uint4 *>(wq + (int64_t(n) * nb + b) * 16));
        const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
        uint32_t lo[4], hi[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            // flipping the top bit of a Q4_0 code gives q - 8 in two's complement;
            // nibbles -> sign-extended bytes -> tc bytes
            const uint32_t t = qw[k] ^ 0x88888888u;
            const uint32_t l = t & 0x0F0F0F0Fu, h = (t >> 4) & 0x0F0F0F0Fu;
            // sign-extend each 4-bit value to a byte: (v ^ 8) - 8 per byte, done as
            // v | (0xF0 where bit 3 set)
            const uint32_t ls = l | (byte_sign_mask(l << 4) & 0xF0F0F0F0u);
            const uint32_t hs = h | (byte_sign_mask(h << 4) & 0xF0F0F0F0u);
            lo[k] = tc_bytes(ls);
            hi[k] = tc_bytes(hs);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(wp + int64_t(n) * nb * 32 + int64_t(b) * 32);
        dst[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        dst[1] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        wsc[g] = __half2float(__ushort_as_half(__ldg(wd + int64_t(n) * nb + b)));
    }
}

// Q4_0 interchange: the file format's 18-byte blocks (fp16 d, then the 16
// code bytes) <-> the planes wq [N][K/2], wd [N][K/32].  A block starts on a
// 2-byte boundary only, so it moves as nine 2-byte words; the planes as one
// 16-byte word and one 2-byte word.
__global__ void __launch_bounds__(256) q4_0_blocks_to_planes_kernel(
    const uint16_t *__restrict__ blocks, uint32_t nblk, uint8_t *__restrict__ wq,
    uint16_t *__restrict__ wd) {
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t g = blockIdx.x * blockDim.x + threadIdx.x; g < nblk; g += stride) {
        const uint16_t *b = blocks + int64_t(g) * 9;
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = static_cast<uint32_t>(__ldg(b + 1 + 2 * k)) |
                   (static_cast<uint32_t>(__ldg(b + 2 + 2 * k)) << 16);
        *reinterpret_cast<uint4 *>(wq + int64_t(g) * 16) = make_uint4(w[0], w[1], w[2], w[3]);
        wd[g] = __ldg(b);
    }
}

__global__ void __launch_bounds__(256) q4_0_planes_to_blocks_kernel(
    const uint8_t *__restrict__ wq, const uint16_t *__restrict__ wd, uint32_t nblk,
    uint16_t *__restrict__ blocks) {
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t g = blockIdx.x * blockDim.x + threadIdx.x; g < nblk; g += stride) {
        const uint4 q = __ldg(reinterpret_cast<const uint4 *>(wq + int64_t(g) * 16));
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        uint16_t *b = blocks + int64_t(g) * 9;
        b[0] = __ldg(wd + g);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            b[1 + 2 * k] = static_cast<uint16_t>(w[k]);
            b[2 + 2 * k] = static_cast<uint16_t>(w[k] >> 16);
        }
    }
}

int grid_for(uint32_t nblk, int sm_count) {
    const uint32_t want = (nblk + 255) / 256;
    const uint32_t cap = static_cast<uint32_t>(sm_count) * 8;
    return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

template <int kBits>
h32_status quantize_act(const void *x, h32_in_dtype dt, int64_t M, int64_t K, int64_t ldx,
                        void *xq, float *xd, int rotate, void *stream) {
    if (M < 0 || K <= 0 || (K % 32) != 0 || ldx < K) return H32_ERR_INVALID_ARG;
    if (rot_points(rotate) < 0 || (rot_points(rotate) > 0 && K % rot_points(rotate) != 0))
        return H32_ERR_INVALID_ARG;
    if (dt != H32_IN_F32 && dt != H32_IN_BF16) return H32_ERR_INVALID_ARG;
    if (M == 0) return H32_OK;
    if (!x || !xq || !xd) return H32_ERR_INVALID_ARG;
    const int64_t esize = (dt == H32_IN_BF16) ? 2 : 4;
    if (!aligned16(x) || !aligned16(xq) || !aligned16(xd) || ((ldx * esize) % 16) != 0)
        return H32_ERR_ALIGNMENT;
    const int64_t nb = K / 32;
    if (M * nb > 0x7FFFFFFFll) return H32_ERR_INVALID_ARG;
    int sms = 0;
    H32_TRY(check_device(&sms));
    const uint32_t nblk = static_cast<uint32_t>(M * nb);
    const uint32_t f = static_cast<uint32_t>(nb);
    const int grid = grid_for(nblk, sms);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *q = reinterpret_cast<uint8_t *>(xq);
    const bool bf = dt == H32_IN_BF16;
#define H32_QA(BF, R) quant_act_kernel<BF, kBits, R><<<grid, 256, 0, s>>>(x, nblk, f, ldx, q, xd)
    switch (rot_points(rotate)) {
        case 0: if (bf) H32_QA(true, 0); else H32_QA(false, 0); break;
        case 32: if (bf) H32_QA(true, 32); else H32_QA(false, 32); break;
        case 64: if (bf) H32_QA(true, 64); else H32_QA(false, 64); break;
        default: if (bf) H32_QA(true, 128); else H32_QA(false, 128); break;
    }
#undef H32_QA
    return launch_status(cudaGetLastError());
}

}  // namespace

__device__ uint32_t g_quant_status_taken;
__global__ void take_g_quant_status() { g_quant_status_taken = atomicExch(&g_quant_status, 0u); }

h32_status quant_read_and_clear_status(cudaStream_t s) {
    bool ok = false;
    const uint32_t v = take_status(take_g_quant_status, g_quant_status_taken, s, &ok);
    if (!ok) return H32_ERR_CUDA;
    if (v & kStatusGuard) return H32_ERR_DEVICE_GUARD;
    return H32_OK;
}

namespace {
int grid_for_tc(uint32_t nblk, int sm_count) { return grid_for(nblk, sm_count); }
}  // namespace

}  // namespace h32

extern "C" h32_status h32_quantize_act_q4(const void *x, h32_in_dtype dt, int64_t M, int64_t K,
                                          int64_t ldx, uint8_t *xq, float *xd, int rotate,
                                          void *stream) {
    return h32::quantize_act<4>(x, dt, M, K, ldx, xq, xd, rotate, stream);
}

extern "C" h32_status h32_quantize_act_q8(const void *x, h32_in_dtype dt, int64_t M, int64_t K,
                                          int64_t ldx, int8_t *xq, float *xd, int rotate,
                                          void *stream) {
    return h32::quantize_act<8>(x, dt, M, K, ldx, xq, xd, rotate, stream);
}

extern "C" h32_status h32_rotate_quantize_weights_q4_0(const float *w, int64_t N, int64_t K,
                                                       int rotate, uint8_t *wq, uint16_t *wd,
                                                       void *stream) {
    using namespace h32;
    if (N < 0 || K <= 0 || (K % 32) != 0) return H32_ERR_INVALID_ARG;
    if (rot_points(rotate) < 0 || (rot_points(rotate) > 0 && K % rot_points(rotate) != 0))
        return H32_ERR_INVALID_ARG;
    if (N == 0) return H32_OK;
    if (!w || !wq || !wd) return H32_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(wq) || !aligned16(wd)) return H32_ERR_ALIGNMENT;
    if (N * (K / 32) > 0x7FFFFFFFll) return H32_ERR_INVALID_ARG;
    int sms = 0;
    H32_TRY(check_device(&sms));
    const uint32_t nblk = static_cast<uint32_t>(N * (K / 32));
    const int grid = grid_for(nblk, sms);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    switch (rot_points(rotate)) {
        case 0: quant_w_kernel<0><<<grid, 256, 0, s>>>(w, nblk, wq, wd); break;
        case 32: quant_w_kernel<32><<<grid, 256, 0, s>>>(w, nblk, wq, wd); break;
        case 64: quant_w_kernel<64><<<grid, 256, 0, s>>>(w, nblk, wq, wd); break;
        default: quant_w_kernel<128><<<grid, 256, 0, s>>>(w, nblk, wq, wd); break;
    }
    return launch_status(cudaGetLastError());
}

namespace h32 {
namespace {
template <int kBits, bool kE5 = false>
h32_status quantize_act_tc(const void *x, h32_in_dtype dt, int64_t M, int64_t K, int64_t ldx,
                           const int32_t *row_idx, int64_t T, uint8_t *xw, float *xdt,
                           int64_t ldxd, int rotate, void *stream) {
    if (M < 0 || K <= 0 || (K % 32) != 0 || ldx < K || ldxd < M || (ldxd % 4) != 0 || T < 0)
        return H32_ERR_INVALID_ARG;
    if (rot_points(rotate) < 0 || (rot_points(rotate) > 0 && K % rot_points(rotate) != 0))
        return H32_ERR_INVALID_ARG;
    if (dt != H32_IN_F32 && dt != H32_IN_BF16) return H32_ERR_INVALID_ARG;
    if (M == 0) return H32_OK;
    if (!x || !xw || !xdt || (row_idx && T == 0)) return H32_ERR_INVALID_ARG;
    const int64_t esize = (dt == H32_IN_BF16) ? 2 : 4;
    if (!aligned16(x) || !aligned16(xw) || !aligned16(xdt) || ((ldx * esize) % 16) != 0 ||
        (row_idx && !aligned16(row_idx)))
        return H32_ERR_ALIGNMENT;
    if (M * (K / 32) > 0x7FFFFFFFll || M > 0x7FFFFFFFll || K > 0x7FFFFFFFll)
        return H32_ERR_INVALID_ARG;
    int sms = 0;
    H32_TRY(check_device(&sms));
    const uint32_t nblk = static_cast<uint32_t>(M * (K / 32));
    const int grid = grid_for_tc(nblk, sms);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint32_t m32 = static_cast<uint32_t>(M), k32 = static_cast<uint32_t>(K);
#define H32_QTC(BF, ROT, GA)                                                                  \
    e = launch_pdl(quant_act_tc_kernel<BF, kBits, ROT, GA, kE5>, dim3(grid), dim3(256), 0, s, x, nblk, \
                   m32, k32, ldx, row_idx, T, xw, xdt, ldxd)
#define H32_QTC_R(ROT)                    \
    do {                                  \
        if (bf && ga) H32_QTC(true, ROT, true);   \
        else if (bf) H32_QTC(true, ROT, false);   \
        else if (ga) H32_QTC(false, ROT, true);   \
        else H32_QTC(false, ROT, false);          \
    } while (0)
    const bool bf = dt == H32_IN_BF16, ga = row_idx != nullptr;
    cudaError_t e = cudaSuccess;
    switch (rot_points(rotate)) {
        case 0: H32_QTC_R(0); break;
        case 32: H32_QTC_R(32); break;
        case 64: H32_QTC_R(64); break;
        default: H32_QTC_R(128); break;
    }
#undef H32_QTC_R
#undef H32_QTC
    return launch_status(e != cudaSuccess ? e : cudaGetLastError());
}
}  // namespace
}  // namespace h32

extern "C" h32_status h32_quantize_act_q4_tc(const void *x, h32_in_dtype dt, int64_t M, int64_t K,
                                             int64_t ldx, uint8_t *xw, float *xdt, int64_t ldxd,
                                             int rotate, void *stream) {
    return h32::quantize_act_tc<4>(x, dt, M, K, ldx, nullptr, M, xw, xdt, ldxd, rotate, stream);
}

extern "C" h32_status h32_quantize_act_q8_tc(const void *x, h32_in_dtype dt, int64_t M, int64_t K,
                                             int64_t ldx, uint8_t *xw8, float *xdt, int64_t ldxd,
                                             int rotate, void *stream) {
    return h32::quantize_act_tc<8>(x, dt, M, K, ldx, nullptr, M, xw8, xdt, ldxd, rotate, stream);
}

extern "C" h32_status h32_quantize_act_q4_tc_gather(const void *x, h32_in_dtype dt, int64_t T,
                                                    int64_t K, int64_t ldx, const int32_t *row_idx,
                                                    int64_t R, uint8_t *xw, float *xdt,
                                                    int64_t ldxd, int rotate, void *stream) {
    if (!row_idx) return H32_ERR_INVALID_ARG;
    return h32::quantize_act_tc<4>(x, dt, R, K, ldx, row_idx, T, xw, xdt, ldxd, rotate, stream);
}

extern "C" h32_status h32_quantize_act_q4_tc_e5m2(const void *x, h32_in_dtype dt, int64_t M,
                                                  int64_t K, int64_t ldx, uint8_t *xw, float *xdt,
                                                  int64_t ldxd, int rotate, void *stream) {
    return h32::quantize_act_tc<4, true>(x, dt, M, K, ldx, nullptr, M, xw, xdt, ldxd, rotate,
                                         stream);
}

extern "C" h32_status h32_quantize_act_q4_tc_e5m2_gather(const void *x, h32_in_dtype dt,
                                                         int64_t T, int64_t K, int64_t ldx,
                                                         const int32_t *row_idx, int64_t R,
                                                         uint8_t *xw, float *xdt, int64_t ldxd,
                                                         int rotate, void *stream) {
    if (!row_idx) return H32_ERR_INVALID_ARG;
    return h32::quantize_act_tc<4, true>(x, dt, R, K, ldx, row_idx, T, xw, xdt, ldxd, rotate,
                                         stream);
}

extern "C" h32_status h32_prepack_weights_q4_0_tc(const uint8_t *wq, const uint16_t *wd, int64_t N,
                                                  int64_t K, uint8_t *wp, float *wsc, int64_t ldws,
                                                  void *stream) {
    using namespace h32;
    if (N < 0 || K <= 0 || (K % 32) != 0 || ldws < K / 32 || (ldws % 4) != 0)
        return H32_ERR_INVALID_ARG;
    if (N == 0) return H32_OK;
    if (!wq || !wd || !wp || !wsc) return H32_ERR_INVALID_ARG;
    if (!aligned16(wq) || !aligned16(wd) || !aligned16(wp) || !aligned16(wsc))
        return H32_ERR_ALIGNMENT;
    if (N * ldws > 0x7FFFFFFFll) return H32_ERR_INVALID_ARG;
    int sms = 0;
    H32_TRY(check_device(&sms));
    const uint32_t total = static_cast<uint32_t>(N * ldws);
    const int grid = grid_for(total, sms);
    prepack_w_tc_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        wq, wd, static_cast<uint32_t>(N), static_cast<uint32_t>(K / 32),
        static_cast<uint32_t>(ldws), wp, wsc);
    return launch_status(cudaGetLastError());
}

namespace h32 {
namespace {
h32_status q4_0_layout_args(const void *blocks, const uint8_t *wq, const uint16_t *wd, int64_t N,
                            int64_t K) {
    if (N < 0 || K <= 0 || (K % 32) != 0) return H32_ERR_INVALID_ARG;
    if (N == 0) return H32_OK;
    if (!blocks || !wq || !wd) return H32_ERR_INVALID_ARG;
    if (!aligned16(blocks) || !aligned16(wq) || !aligned16(wd)) return H32_ERR_ALIGNMENT;
    if (N * (K / 32) > 0x7FFFFFFFll) return H32_ERR_INVALID_ARG;
    return H32_OK;
}
}  // namespace
}  // namespace h32

extern "C" h32_status h32_q4_0_blocks_to_planes(const uint8_t *blocks, int64_t N, int64_t K,
                                                uint8_t *wq, uint16_t *wd, void *stream) {
    using namespace h32;
    H32_TRY(q4_0_layout_args(blocks, wq, wd, N, K));
    if (N == 0) return H32_OK;
    int sms = 0;
    H32_TRY(check_device(&sms));
    const uint32_t nblk = static_cast<uint32_t>(N * (K / 32));
    q4_0_blocks_to_planes_kernel<<<grid_for(nblk, sms), 256, 0,
                                   reinterpret_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const uint16_t *>(blocks), nblk, wq, wd);
    return launch_status(cudaGetLastError());
}

extern "C" h32_status h32_q4_0_planes_to_blocks(const uint8_t *wq, const uint16_t *wd, int64_t N,
                                                int64_t K, uint8_t *blocks, void *stream) {
    using namespace h32;
    H32_TRY(q4_0_layout_args(blocks, wq, wd, N, K));
    if (N == 0) return H32_OK;
    int sms = 0;
    H32_TRY(check_device(&sms));
    const uint32_t nblk = static_cast<uint32_t>(N * (K / 32));
    q4_0_planes_to_blocks_kernel<<<grid_for(nblk, sms), 256, 0,
                                   reinterpret_cast<cudaStream_t>(stream)>>>(
        wq, wd, nblk, reinterpret_cast<uint16_t *>(blocks));
    return launch_status(cudaGetLastError());
}
