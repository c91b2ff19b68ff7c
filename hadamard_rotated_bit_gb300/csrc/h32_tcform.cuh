// The tensor-core operand form shared by the quantizers and the GEMM
// epilogue that quantizes its own output for the next projection: rounding
// constants and the byte encodings of integer codes as e4m3.
#pragma once

#include <stdint.h>

namespace h32 {

// fp32 nearest to 1/sqrt(32) (bit pattern 0x3E3504F3)
constexpr float kInvSqrt32 = 0x1.6a09e6p-3f;
constexpr float kInvSqrt128 = 0x1.6a09e6p-4f;   // half of kInvSqrt32: the fp32 nearest 1/sqrt(128)
// 1.5 * 2^23: adding it to |t| < 2^22 leaves round-half-even(t) in the low
// mantissa bits as a two's-complement integer
constexpr float kRoundMagic = 12582912.0f;

// The code value of y in a degenerate block, where 1/d is not finite (d below
// 2^-128: a block of subnormal size) or d is infinite (the rotation
// overflowed): y / d by an IEEE divide, so an exact zero stays 0 and the
// element of largest magnitude gets +-qmax; inf / inf (an infinite element of
// an overflowed block) reads as its limit, +-qmax.  Clamped to [qmin, qmax],
// not yet rounded.
__device__ __forceinline__ float degenerate_code(float y, float d, float qmin, float qmax) {
    float t = __fdiv_rn(y, d);
    if (isnan(t)) t = copysignf(qmax, y);
    return fminf(fmaxf(t, qmin), qmax);
}

// strides 1, 2, 4, 8, 16: the in-thread stages of every rotation size
__device__ __forceinline__ void butterfly32(float (&v)[32]) {
#pragma unroll
    for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            if ((i & h) == 0) {
                const float a = v[i], c = v[i + h];
                v[i] = __fadd_rn(a, c);
                v[i + h] = __fsub_rn(a, c);
            }
        }
    }
}

__device__ __forceinline__ void rotate32(float (&v)[32]) {
    butterfly32(v);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __fmul_rn(v[i], kInvSqrt32);
}


// tensor-core form: one byte per code, the e4m3 encoding of the integer code
__device__ __forceinline__ uint32_t byte_sign_mask(uint32_t x) {
    uint32_t r;
    asm("prmt.b32 %0, %1, 0, 0xBA98;" : "=r"(r) : "r"(x));
    return r;
}

// four magnitudes 0..8 (one per byte) -> their e4m3 bytes.  e4m3 (bias 7,
// 3 mantissa bits) holds every integer up to 16 exactly: 1 = 0x38, 2 = 0x40,
// 3 = 0x44, 4 = 0x48, 5 = 0x4A, 6 = 0x4C, 7 = 0x4E, 8 = 0x50.  A byte permute
// looks 0..7 up in an 8-byte table; the selector nibble 8 picks table byte 0
// (0x00) in sign-replicate mode, which stays 0x00, and 8 is then or-ed in.
__device__ __forceinline__ uint32_t e4m3_of_magnitudes(uint32_t mag) {
    const uint32_t sel = (mag & 0xFu) | ((mag >> 4) & 0xF0u) | ((mag >> 8) & 0xF00u) |
                         ((mag >> 12) & 0xF000u);
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(0x44403800u), "r"(0x4E4C4A48u), "r"(sel));
    return r | (((mag >> 3) & 0x01010101u) * 0x50u);
}

// four int8 codes in [-8, 8] -> four e4m3 bytes (sign bit | e4m3 of |c|)
__device__ __forceinline__ uint32_t tc_bytes(uint32_t c) {
    const uint32_t m = byte_sign_mask(c);                       // 0xFF where negative
    const uint32_t mag = (c ^ m) + (m & 0x01010101u);           // |c| per byte, no carries
    return e4m3_of_magnitudes(mag) | (m & 0x80808080u);
}

// Sixteen-entry byte table lookup: each byte v (0..15) of `v` -> byte v of the
// table t0..t3 (t0 holding entries 0..3 from its low byte up).  Two byte
// permutes look up v & 7 in each half of the table; bit 3 of v picks the half.
__device__ __forceinline__ uint32_t lut16(uint32_t v, uint32_t t0, uint32_t t1, uint32_t t2,
                                          uint32_t t3) {
    const uint32_t s = v & 0x07070707u;
    uint32_t sel, a, b;
    asm("prmt.b32 %0, %1, 0, 0x4420;" : "=r"(sel) : "r"(s | (s >> 4)));   // 4 nibbles
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(a) : "r"(t0), "r"(t1), "r"(sel));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(b) : "r"(t2), "r"(t3), "r"(sel));
    const uint32_t m = byte_sign_mask(v << 4);                               // 0xFF where v >= 8
    return (a & ~m) | (b & m);
}

// four int8 codes c = 16 h + l (0 <= l <= 15, -8 <= h <= 7) -> the e4m3 bytes
// of 16 h (hi) and of l (lo), by table: l = 0..7 as in e4m3_of_magnitudes,
// 8..15 = 0x50..0x57; 16 h for the 4-bit pattern of h = 0..7: 0x00, 0x58, 0x60,
// 0x64, 0x68, 0x6A, 0x6C, 0x6E, and for h = -8..-1: 0xF0, 0xEE, 0xEC, 0xEA, 0xE8,
// 0xE4, 0xE0, 0xD8.
__device__ __forceinline__ void tc_bytes_q8(uint32_t c, uint32_t &hi, uint32_t &lo) {
    lo = lut16(c & 0x0F0F0F0Fu, 0x44403800u, 0x4E4C4A48u, 0x53525150u, 0x57565554u);
    hi = lut16((c >> 4) & 0x0F0F0F0Fu, 0x64605800u, 0x6E6C6A68u, 0xEAECEEF0u, 0xD8E0E4E8u);
}


// The widening form of the weight codes: the Q4_0 code q (0..15) itself as
// the byte 0x0q, which read as e4m3 is q * 2^-9 exactly (exponent field 0:
// subnormals m * 2^-9 for q < 8; field 1: (8 + m) * 2^-9 for q >= 8).  Eight
// codes of one word of a Q4_0 block (byte j of the block: element j in the low
// nibble, element j + 16 in the high one) -> the bytes of the low-nibble
// elements j..j+3 in `lo` and of the high-nibble elements j+16..j+19 in `hi`.
__device__ __forceinline__ void widen_q4_0_word(uint32_t x, uint32_t &lo, uint32_t &hi) {
    lo = x & 0x0F0F0F0Fu;
    hi = (x >> 4) & 0x0F0F0F0Fu;
}

// four integer-valued floats (each exactly representable in e4m3: |c| <= 16,
// or a multiple of 16 up to 128) -> their e4m3 bytes, c0 in the lowest byte.
// The hardware conversion is exact for such values.
__device__ __forceinline__ uint32_t e4m3x4_of_ints(float c0, float c1, float c2, float c3) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(c1), "f"(c0));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(c3), "f"(c2));
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// The activation side of the widening form: four integer codes |c| <= 8 ->
// the e5m2 bytes of 512 c (exact: at most three significant bits, exponent
// within range), so that with weights read as q * 2^-9 every product is the
// integer q c.  0 = 0x00, 1 = 0x60, 2 = 0x64, 3 = 0x66, 4 = 0x68, 5 = 0x69,
// 6 = 0x6A, 7 = 0x6B, 8 = 0x6C, the sign in bit 7.
__device__ __forceinline__ uint32_t e5m2x4_of_ints_x512(float c0, float c1, float c2, float c3) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;"
        : "=h"(lo)
        : "f"(__fmul_rn(c1, 512.0f)), "f"(__fmul_rn(c0, 512.0f)));
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;"
        : "=h"(hi)
        : "f"(__fmul_rn(c3, 512.0f)), "f"(__fmul_rn(c2, 512.0f)));
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// One 32-block y of activations to 4-bit codes in tensor-core form, the step
// every 4-bit tc-form producer shares (the activation quantizer and the GEMM
// that quantizes its own output): d = amax(|y|) / 7 (IEEE divide), codes
// round-half-even(y * fl(1/d)) (the clamped y / d in a degenerate block), each
// code as the e4m3 byte of the integer (kE5: the e5m2 byte of 512 times the
// integer, the widening form); w[k] holds codes 4k .. 4k + 3 from its low byte
// up.  Returns d.
template <bool kE5 = false>
__device__ __forceinline__ float quant_block_tc4(const float (&v)[32], uint32_t (&w)[8]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const float d = __fdiv_rn(amax, 7.0f);
    const float id = (d != 0.0f) ? __frcp_rn(d) : 0.0f;
    uint32_t bits[32];
    if (!(amax < INFINITY) || isinf(id)) {   // degenerate block: the clamped y / d
#pragma unroll
        for (int i = 0; i < 32; ++i)
            bits[i] = __float_as_uint(__fadd_rn(degenerate_code(v[i], d, -8.0f, 7.0f), kRoundMagic));
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            bits[i] = __float_as_uint(__fadd_rn(__fmul_rn(v[i], id), kRoundMagic));
    }
    // the codes as integer-valued floats (exact: bits holds code + 1.5 * 2^23),
    // converted to e4m3 by the hardware (exact for |code| <= 8)
    float c[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) c[i] = __fsub_rn(__uint_as_float(bits[i]), kRoundMagic);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        if constexpr (kE5)
            w[k] = e5m2x4_of_ints_x512(c[4 * k], c[4 * k + 1], c[4 * k + 2], c[4 * k + 3]);
        else
            w[k] = e4m3x4_of_ints(c[4 * k], c[4 * k + 1], c[4 * k + 2], c[4 * k + 3]);
    }
    return d;
}

}  // namespace h32
