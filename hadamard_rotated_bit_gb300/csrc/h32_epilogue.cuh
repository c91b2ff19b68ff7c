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
