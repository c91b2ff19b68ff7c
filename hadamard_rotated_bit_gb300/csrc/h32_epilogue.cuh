// Epilogue arithmetic shared by the GEMM kernels (sm_103a): the per-block
// scale step acc = fma(fp32(d_w * d_x), S, acc) on packed fp32 pairs.
#pragma once

#include <stdint.h>

namespace h32 {

// packed fp32 pairs (low half = first element); IEEE round-to-nearest-even per lane
__device__ __forceinline__ uint64_t pair_of(uint32_t lo, uint32_t hi) {
    return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// 16 columns of one block into the accumulators: acc = fma(fp32(dw * dx), S, acc),
// two columns per packed operation; dx and S come in as pairs already
__device__ __forceinline__ void fold16(uint64_t *acc, float dw, const float *dx,
                                       const uint32_t (&v)[16]) {
    const uint32_t w = __float_as_uint(dw);
    const uint64_t dw2 = pair_of(w, w);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const ulonglong2 d = *reinterpret_cast<const ulonglong2 *>(dx + 4 * q);
        acc[2 * q] = fma_f32x2(mul_f32x2(dw2, d.x), pair_of(v[4 * q], v[4 * q + 1]), acc[2 * q]);
        acc[2 * q + 1] =
            fma_f32x2(mul_f32x2(dw2, d.y), pair_of(v[4 * q + 2], v[4 * q + 3]), acc[2 * q + 1]);
    }
}

// One 16-column chunk of one block when a thread holds two rows (16x32bx2
// load pair): va = row a, vb = row b, each 8 consecutive columns whose token
// scales start at dx; acc[0..3] row a, acc[4..7] row b, in column pairs
__device__ __forceinline__ void fold8x2(uint64_t *acc, float dwa, float dwb, const float *dx,
                                        const uint32_t (&va)[8], const uint32_t (&vb)[8]) {
    const uint64_t wa = pair_of(__float_as_uint(dwa), __float_as_uint(dwa));
    const uint64_t wb = pair_of(__float_as_uint(dwb), __float_as_uint(dwb));
    const ulonglong2 d0 = *reinterpret_cast<const ulonglong2 *>(dx);
    const ulonglong2 d1 = *reinterpret_cast<const ulonglong2 *>(dx + 4);
    const uint64_t d[4] = {d0.x, d0.y, d1.x, d1.y};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        acc[q] = fma_f32x2(mul_f32x2(wa, d[q]), pair_of(va[2 * q], va[2 * q + 1]), acc[q]);
        acc[4 + q] = fma_f32x2(mul_f32x2(wb, d[q]), pair_of(vb[2 * q], vb[2 * q + 1]), acc[4 + q]);
    }
}

// One 16-column chunk of one block when a thread holds four rows (16x256b load
// pair): rows k = 0..3 with weight scales dw[k]; p0, p1 the token-scale pairs
// of its columns 2g, 2g + 1 and 8 + 2g, 9 + 2g; va = rows 0 and 1, vb = rows 2
// and 3 in the 16x256b order; acc[2k + e] = row k, column pair e
__device__ __forceinline__ void fold4x4(uint64_t *acc, const uint64_t (&dw2)[4], uint64_t p0,
                                        uint64_t p1, const uint32_t (&va)[8],
                                        const uint32_t (&vb)[8]) {
    acc[0] = fma_f32x2(mul_f32x2(dw2[0], p0), pair_of(va[0], va[1]), acc[0]);
    acc[1] = fma_f32x2(mul_f32x2(dw2[0], p1), pair_of(va[4], va[5]), acc[1]);
    acc[2] = fma_f32x2(mul_f32x2(dw2[1], p0), pair_of(va[2], va[3]), acc[2]);
    acc[3] = fma_f32x2(mul_f32x2(dw2[1], p1), pair_of(va[6], va[7]), acc[3]);
    acc[4] = fma_f32x2(mul_f32x2(dw2[2], p0), pair_of(vb[0], vb[1]), acc[4]);
    acc[5] = fma_f32x2(mul_f32x2(dw2[2], p1), pair_of(vb[4], vb[5]), acc[5]);
    acc[6] = fma_f32x2(mul_f32x2(dw2[3], p0), pair_of(vb[2], vb[3]), acc[6]);
    acc[7] = fma_f32x2(mul_f32x2(dw2[3], p1), pair_of(vb[6], vb[7]), acc[7]);
}

// the same when some d_w * d_x falls outside the normal range: round the
// product of the unscaled scales itself, then apply the 2^18 exactly
__device__ __forceinline__ void fold16_exact(uint64_t *acc, float dw, const float *dx,
                                          const uint32_t (&v)[16]) {
    const float dw0 = dw * 0x1p-18f;
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        const uint64_t pr = acc[i / 2];
        const float s0 = __fmul_rn(__fmul_rn(dw0, dx[i]), 262144.0f);
        const float s1 = __fmul_rn(__fmul_rn(dw0, dx[i + 1]), 262144.0f);
        const float a0 = __fmaf_rn(s0, __uint_as_float(v[i]), __uint_as_float(static_cast<uint32_t>(pr)));
        const float a1 =
            __fmaf_rn(s1, __uint_as_float(v[i + 1]), __uint_as_float(static_cast<uint32_t>(pr >> 32)));
        acc[i / 2] = pair_of(__float_as_uint(a0), __float_as_uint(a1));
    }
}

}  // namespace h32
