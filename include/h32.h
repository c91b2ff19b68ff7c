/*
 * h32.h -- C ABI of the Hadamard-route prompt path for one GB300 GPU (sm_103a).
 *
 * The method (pages: "509 tokens a second of prompt: the Hadamard route ships"
 * and "Qwen3.8-27B at 45.7 tok/s ...", section "Prompt processing: 4-bit
 * activations, rotated first"):
 *   - activations are rounded in blocks of 32 values that share one scale;
 *   - each block is first rotated by a 32-point Walsh-Hadamard transform,
 *     which spreads a few large values over the block ("The rotation");
 *   - the weights are rotated the same way once, offline, and stored as
 *     Q4_0 (an fp16 scale and 32 4-bit codes q per block, value (q - 8) * d),
 *     so every dot product is unchanged: x . w = (Hx) . (Hw);
 *   - the matrix product runs on 4-bit (or, on the exact route, 8-bit)
 *     activation codes against the Q4_0 codes, whose top bit flipped is the
 *     two's-complement value q - 8 ("Why prompts are a matrix-unit problem").
 *
 * Conventions for every call:
 *   Ownership  All array pointers are device pointers owned by the caller.
 *              The library keeps no pointer after a call returns and allocates
 *              no device memory (the K split's workspace is the caller's, or,
 *              for the _noalloc calls, a static array of the library's own).
 *   Streams    `stream` is a cudaStream_t (0 = the legacy default stream).
 *              Every compute call only enqueues work on it and returns.
 *   Errors     Argument, shape and alignment errors are returned at once,
 *              before anything is enqueued.  A failed launch returns
 *              H32_ERR_CUDA.  Problems found on the device (a bounded wait
 *              that gave up, a range guard) set a per-library device status
 *              word instead; h32_device_status() synchronizes the stream and
 *              reports (and clears) it.  There is no CPU fallback: a device
 *              that is not sm_103 returns H32_ERR_UNSUPPORTED.
 *   Layouts    Row-major.  K is the reduction length, a multiple of 32;
 *              nb = K / 32 blocks per row.  4-bit codes are stored in the
 *              Q4_0 nibble order: byte j (0..15) of a block holds element j in
 *              its low nibble and element j + 16 in its high nibble.
 *   Alignment  Every array pointer is 16-byte aligned; row pitches given in
 *              elements must make the pitch in bytes a multiple of 16.
 *   Empty      M = 0 (or R = 0) is valid and enqueues nothing.
 */
#ifndef H32_H
#define H32_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum h32_status {
    H32_OK = 0,
    H32_ERR_INVALID_ARG = 1,  /* null pointer, bad shape or dtype               */
    H32_ERR_ALIGNMENT = 2,    /* pointer or row pitch not 16-byte aligned       */
    H32_ERR_UNSUPPORTED = 3,  /* no CUDA device, or the device is not sm_103    */
    H32_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed    */
    H32_ERR_TIMEOUT = 5,      /* device status: a bounded wait gave up          */
    H32_ERR_DEVICE_GUARD = 6  /* device status: a device-side range check fired */
} h32_status;

typedef enum h32_in_dtype {
    H32_IN_F32 = 0,  /* fp32 activations                                     */
    H32_IN_BF16 = 1  /* bf16 activations, widened to fp32 exactly            */
} h32_in_dtype;

/*
 * Rotate and quantize activations to 4-bit codes (the activation quantizer of
 * "The rotation" / "Prompt processing: 4-bit activations, rotated first").
 * For each row m and block b: y = H x_block / sqrt(32) (fp32 butterfly,
 * strides 1, 2, 4, 8, 16, then one multiply by the fp32 nearest 1/sqrt(32));
 * d = amax(|y|) / 7 in fp32; codes = round-half-even(clamp(y * (1/d), -8, 7)),
 * all codes 0 when d = 0.  In a degenerate block, where 1/d is not finite (a
 * block of subnormal size, d below 2^-128) or the rotation overflowed to
 * +-inf, the code is round-half-even(clamp(y / d)) by an IEEE divide instead:
 * exact zeros stay 0 and an infinite element gets +-7 (the limit of y / d).
 *   x      [M][ldx] activations of type `dt`, ldx >= K
 *   xq     [M][K/2] out: two's-complement 4-bit codes, Q4_0 nibble order
 *   xd     [M][K/32] out: fp32 scales d
 *   rotate 1 (or 32) = rotate first (the Hadamard route); 0 = plain 4-bit route;
 *          64 or 128 = the larger rotation the pages name as the next step
 *          ("Qwen3.8-27B at 45.7 tok/s ...", section "What's next"): the same
 *          Sylvester butterfly over each 64- or 128-block (strides 1 .. n/2,
 *          then one multiply by the fp32 nearest 1/sqrt(n)), scales still one
 *          per 32-block; K must be a multiple of n.  Any other value:
 *          H32_ERR_INVALID_ARG.  The same argument, with the same meaning, is
 *          taken by every quantizer below and by the weight quantizer; weights
 *          and activations of one product must use the same rotation.
 */
h32_status h32_quantize_act_q4(const void *x, h32_in_dtype dt, int64_t M, int64_t K, int64_t ldx,
                               uint8_t *xq, float *xd, int rotate, void *stream);

/*
 * The exact route's 8-bit activation quantizer ("Prompt processing ...": the
 * exact int8 path).  As h32_quantize_act_q4 with d = amax / 127 and codes
 * clamped to [-127, 127], stored as int8 in element order.
 *   xq     [M][K] out: int8 codes;  xd [M][K/32] out: fp32 scales
 */
h32_status h32_quantize_act_q8(const void *x, h32_in_dtype dt, int64_t M, int64_t K, int64_t ldx,
                               int8_t *xq, float *xd, int rotate, void *stream);

/*
 * Offline weight step ("Making the file is part of the engine": rotate the
 * projections, then quantize to Q4_0).  Each 32-block of a weight row is
 * rotated with the same transform as the activations (rotate as for
 * h32_quantize_act_q4: 0, 1/32, 64 or 128 points), then
 * rounded by the Q4_0 rule: the signed value of largest magnitude (first on
 * ties) maps to code 0, d = max / -8, code = min(15, trunc(y * (1/d) + 8.5)),
 * d stored as fp16 rounded to nearest even.  Degenerate blocks as for the
 * activations: where 1/d is not finite or the rotation overflowed, y / d by an
 * IEEE divide replaces y * (1/d) (a zero gets code 8); inf / inf reads as -8
 * where y has the sign of the signed maximum, else +8.
 *   w      [N][K] fp32 weights (rows are output features)
 *   wq     [N][K/2] out: codes 0..15 in Q4_0 nibble order
 *   wd     [N][K/32] out: fp16 scales (bit patterns)
 */
h32_status h32_rotate_quantize_weights_q4_0(const float *w, int64_t N, int64_t K, int rotate,
                                            uint8_t *wq, uint16_t *wd, void *stream);

/*
 * Q4_0 interchange with the file format ("Qwen3.8-27B at 45.7 tok/s ...",
 * section "Prompt processing: 4-bit activations, rotated first": the route
 * reads plain Q4_0 files).  A file block is 18 bytes: the fp16 scale d (little
 * endian), then the 16 code bytes in Q4_0 nibble order.  Every entry point of
 * this library takes the two planes instead (the 18-byte blocks do not sit on
 * the 16-byte boundaries the tensor copies need):
 *   blocks  [N][K/32][18] bytes, the base 16-byte aligned
 *   wq      [N][K/2] codes;  wd [N][K/32] fp16 bit patterns
 * Requires K % 32 == 0.  Pure moves: the bytes are unchanged.
 */
h32_status h32_q4_0_blocks_to_planes(const uint8_t *blocks, int64_t N, int64_t K, uint8_t *wq,
                                     uint16_t *wd, void *stream);
h32_status h32_q4_0_planes_to_blocks(const uint8_t *wq, const uint16_t *wd, int64_t N, int64_t K,
                                     uint8_t *blocks, void *stream);

/*
 * Block-scaled integer product of Q4_0 weights and 4-bit activations (the
 * W4A4 matrix product of "Why prompts are a matrix-unit problem").
 *   y[m][n] = sum over b = 0 .. nb-1, in that order, of
 *             acc = fma(fp32(d_w[n][b] * d_x[m][b]), S[m][n][b], acc), acc0 = +0,
 *   S[m][n][b] = sum_j x_code[m][32b+j] * (w_code[n][32b+j] - 8), exact.
 *   wq, wd      Q4_0 weights as written by h32_rotate_quantize_weights_q4_0
 *   xq, xd      4-bit activations as written by h32_quantize_act_q4
 *   y           [M][ldy] fp32 out, ldy >= N
 *   block_sums  nullable debug output: int32 [M][N][K/32], the exact S
 * Requires N % 16 == 0.
 */
h32_status q4_0_x_q4_gemm(const uint8_t *wq, const uint16_t *wd, const uint8_t *xq,
                          const float *xd, int64_t M, int64_t N, int64_t K, float *y,
                          int64_t ldy, int32_t *block_sums, void *stream);

/*
 * The exact route: Q4_0 weights against 8-bit activation codes
 * (h32_quantize_act_q8).  Same definition with x_code in [-127, 127].
 */
h32_status q4_0_x_q8_gemm(const uint8_t *wq, const uint16_t *wd, const int8_t *xq,
                          const float *xd, int64_t M, int64_t N, int64_t K, float *y,
                          int64_t ldy, int32_t *block_sums, void *stream);

/*
 * Expert-batched W4A4 product for mixture-of-experts layers ("4-bit
 * activations reach the MoE experts").  Output rows are in grouped order:
 * row r in [expert_off[e], expert_off[e+1]) uses expert e's weights and the
 * activation row row_idx[r] (row_idx = NULL means row r itself).
 *   wq          [E][N][K/2] Q4_0 codes;  wd [E][N][K/32] fp16 scales
 *   xq, xd      4-bit activations [T][K/2], [T][K/32]
 *   row_idx     device int32 [R] or NULL; entries outside [0, T) set
 *               H32_ERR_DEVICE_GUARD and read as an all-zero row
 *   T           rows of xq / xd (with row_idx = NULL, T must be >= R)
 *   expert_off  device int32 [E+1], non-decreasing, expert_off[0] = 0,
 *               expert_off[E] = R (checked on the device: a violation sets
 *               H32_ERR_DEVICE_GUARD and the kernel writes nothing)
 *   y           [R][ldy] fp32 out;  block_sums nullable int32 [R][N][K/32]
 * Requires N % 16 == 0 and 1 <= E <= 1024.
 */
h32_status q4_0_x_q4_gemm_experts(const uint8_t *wq, const uint16_t *wd, int32_t E,
                                  const uint8_t *xq, const float *xd, const int32_t *row_idx,
                                  int64_t T, const int32_t *expert_off, int64_t R, int64_t N,
                                  int64_t K,
                                  float *y, int64_t ldy, int32_t *block_sums, void *stream);

/*
 * ---------------------------------------------------------------------------
 * Tensor-core form ("tc form").  GB300 has no integer tensor-core MMA; the
 * exact 4-bit products run on the FP8 tensor cores, with every code v stored
 * as one byte: the e4m3 encoding of the integer v itself (every integer of
 * magnitude 0..8 is exact in e4m3, so each 32-term block sum S comes out of
 * the MMA exact, as an integer-valued fp32).  The calls below produce and
 * consume that form directly, so the GEMM needs no widening step: weights are
 * repacked once, offline (lossless: the same codes and scales), and the
 * activation quantizer writes the tc form.  Results are bit-identical to the
 * Q4_0 entry points above.
 * ---------------------------------------------------------------------------
 */

/*
 * Rotate and quantize activations exactly as h32_quantize_act_q4, writing the
 * codes in tc form and the scales block-major:
 *   xw     [M][K] out: one byte per code, the e4m3 encoding of the code, element order
 *   xdt    [K/32][ldxd] out: fp32 scales, xdt[b][m] = d of row m, block b
 *   ldxd   >= M, a multiple of 4 (entries m >= M are left untouched)
 */
h32_status h32_quantize_act_q4_tc(const void *x, h32_in_dtype dt, int64_t M, int64_t K,
                                  int64_t ldx, uint8_t *xw, float *xdt, int64_t ldxd, int rotate,
                                  void *stream);

/*
 * The exact 8-bit route in tc form ("509 tokens a second of prompt: the
 * Hadamard route ships", section "Why prompts are a matrix-unit problem"):
 * codes and scales exactly as h32_quantize_act_q8; each code c = 16 h + l with
 * 0 <= l <= 15 (so -8 <= h <= 7) is stored as two e4m3 bytes, both exact:
 *   xw8    [M][2K] out: per 32-block 64 bytes, the 32 bytes of 16 h, then the
 *          32 bytes of l (element order within each half)
 *   xdt    [K/32][ldxd] out as for h32_quantize_act_q4_tc
 */
h32_status h32_quantize_act_q8_tc(const void *x, h32_in_dtype dt, int64_t M, int64_t K,
                                  int64_t ldx, uint8_t *xw8, float *xdt, int64_t ldxd, int rotate,
                                  void *stream);

/*
 * The same with a row gather, for expert-batched products ("Where the engine is
 * going: HRX and the NPU", section "4-bit activations reach the MoE experts"):
 * output row r is input row row_idx[r] of x[T][ldx], so the rows come out in the
 * experts' grouped order, ready for q4_0_x_q4_gemm_tc_experts.
 *   row_idx  [R] int32 device, each in [0, T); an index outside records
 *            H32_ERR_DEVICE_GUARD (see h32_device_status) and its row gets zero
 *            codes and a zero scale
 *   xw       [R][K] out; xdt [K/32][ldxd] out, ldxd >= R, a multiple of 4
 */
h32_status h32_quantize_act_q4_tc_gather(const void *x, h32_in_dtype dt, int64_t T, int64_t K,
                                         int64_t ldx, const int32_t *row_idx, int64_t R,
                                         uint8_t *xw, float *xdt, int64_t ldxd, int rotate,
                                         void *stream);

/*
 * Repack Q4_0 weights (as written by h32_rotate_quantize_weights_q4_0) into
 * tc form, once, offline:
 *   wp     [N][K] out: one byte per weight, the e4m3 encoding of q - 8, element order
 *   wsc    [N][ldws] out: fp32 d (exact widening of the fp16), ldws >= K/32, a multiple of 4;
 *          entries b >= K/32 are written as 0
 */
h32_status h32_prepack_weights_q4_0_tc(const uint8_t *wq, const uint16_t *wd, int64_t N,
                                       int64_t K, uint8_t *wp, float *wsc, int64_t ldws,
                                       void *stream);

/*
 * The W4A4 product of q4_0_x_q4_gemm on tc-form operands:
 *   y[m][n] = sum over blocks b in order of acc = fma(fp32(d_w * d_x), S, acc)
 * with d_w = wsc[n][b], d_x = xdt[b][m], bit-identical to q4_0_x_q4_gemm for
 * every finite scale (subnormal products d_w * d_x included).
 *   wp, wsc, ldws   from h32_prepack_weights_q4_0_tc
 *   xw, xdt, ldxd   from h32_quantize_act_q4_tc
 *   y               [M][ldy] fp32 out;  block_sums nullable int32 [M][N][K/32]
 * Requires K % 128 == 0 and N % 16 == 0.
 */
h32_status q4_0_x_q4_gemm_tc(const uint8_t *wp, const float *wsc, int64_t ldws,
                             const uint8_t *xw, const float *xdt, int64_t ldxd, int64_t M,
                             int64_t N, int64_t K, float *y, int64_t ldy, int32_t *block_sums,
                             void *stream);

/*
 * q4_0_x_q4_gemm_tc with its output also quantized, in the same kernel, for the
 * next projection (a fused producer: the output never makes an extra HBM round
 * trip before the next projection's activation quantizer).  The rows of the
 * output (the next projection's K dimension) are cut into 32-blocks; each is
 * rotated (rotate_next = 1 or 32) or not (0) and quantized exactly as
 * h32_quantize_act_q4_tc would quantize the fp32 output y, bit for bit.
 *   y          [M][ldy] fp32 out, or null (then only the quantized form is written)
 *   xw_next    [M][N] out: tc-form codes of y, as h32_quantize_act_q4_tc's xw
 *   xdt_next   [N/32][ldxd_next] out: fp32 scales, ldxd_next >= M
 * Requires N % 32 == 0 (and the conditions of q4_0_x_q4_gemm_tc).
 */
h32_status q4_0_x_q4_gemm_tc_quant_next(const uint8_t *wp, const float *wsc, int64_t ldws,
                                        const uint8_t *xw, const float *xdt, int64_t ldxd,
                                        int64_t M, int64_t N, int64_t K, float *y, int64_t ldy,
                                        uint8_t *xw_next, float *xdt_next, int64_t ldxd_next,
                                        int rotate_next, void *stream);

/*
 * q4_0_x_q4_gemm_tc_quant_next with a caller-owned workspace for the K split of
 * the last wave (the workspace as for q4_0_x_q4_gemm_tc_ws below; same results
 * bit for bit, the output and its next-projection quantization both).
 */
h32_status q4_0_x_q4_gemm_tc_quant_next_ws(const uint8_t *wp, const float *wsc, int64_t ldws,
                                           const uint8_t *xw, const float *xdt, int64_t ldxd,
                                           int64_t M, int64_t N, int64_t K, float *y, int64_t ldy,
                                           uint8_t *xw_next, float *xdt_next, int64_t ldxd_next,
                                           int rotate_next, void *workspace,
                                           size_t workspace_bytes, void *stream);

/*
 * ---------------------------------------------------------------------------
 * Widening form.  The GEMMs below read the Q4_0 weight planes themselves
 * (half the weight bytes of the tc form; no repack) and widen each K stage's
 * nibbles in shared memory ("Why prompts are a matrix-unit problem": the codes
 * go to the matrix units as small integers).  A code q (0..15) becomes the byte
 * 0x0q, which the FP8 tensor cores read as e4m3 q * 2^-9, exactly; the
 * activations of this form are the e5m2 bytes of 512 times their codes, also
 * exact, so every product is the integer q x.  One more tensor-core product
 * per block, against weights of -8 * 2^-9, subtracts 8 times the activation
 * block sum: S = sum (q - 8) x exactly, and the results are bit-identical to
 * the tc form and to the Q4_0 entry points.
 * ---------------------------------------------------------------------------
 */

/*
 * Rotate and quantize activations exactly as h32_quantize_act_q4_tc (same
 * codes, same scales, same layouts), each code c stored as the e5m2 byte of
 * 512 c: 0 = 0x00, 1 = 0x60, 2 = 0x64, 3 = 0x66, 4 = 0x68, 5 = 0x69, 6 = 0x6A,
 * 7 = 0x6B, 8 = 0x6C, bit 7 the sign.
 *   xw     [M][K] out: one byte per code, element order
 *   xdt    [K/32][ldxd] out: fp32 scales, as for h32_quantize_act_q4_tc
 */
h32_status h32_quantize_act_q4_tc_e5m2(const void *x, h32_in_dtype dt, int64_t M, int64_t K,
                                       int64_t ldx, uint8_t *xw, float *xdt, int64_t ldxd,
                                       int rotate, void *stream);

/*
 * The same with the row gather of h32_quantize_act_q4_tc_gather (output row r
 * is input row row_idx[r]; an index outside [0, T) records
 * H32_ERR_DEVICE_GUARD and its row gets zero codes and a zero scale).
 */
h32_status h32_quantize_act_q4_tc_e5m2_gather(const void *x, h32_in_dtype dt, int64_t T,
                                              int64_t K, int64_t ldx, const int32_t *row_idx,
                                              int64_t R, uint8_t *xw, float *xdt, int64_t ldxd,
                                              int rotate, void *stream);

/*
 * The W4A4 product of q4_0_x_q4_gemm on the Q4_0 planes, widened in shared
 * memory:
 *   y[m][n] = sum over blocks b in order of acc = fma(fp32(d_w * d_x), S, acc)
 * with d_w = wd[n][b] (fp16, widened exactly), d_x = xdt[b][m]; bit-identical to
 * q4_0_x_q4_gemm_tc and q4_0_x_q4_gemm.
 *   wq, wd          [N][K/2], [N][K/32] Q4_0 planes as written by
 *                   h32_rotate_quantize_weights_q4_0 (fp16 scale bit patterns)
 *   xw, xdt, ldxd   from h32_quantize_act_q4_tc_e5m2
 *   y               [M][ldy] fp32 out;  block_sums nullable int32 [M][N][K/32]
 * Requires K % 256 == 0 (the scale rows, K/16 bytes, feed a tensor copy of
 * 16-byte units) and N % 16 == 0.
 */
h32_status q4_0_x_q4_gemm_tc_widen(const uint8_t *wq, const uint16_t *wd, const uint8_t *xw,
                                   const float *xdt, int64_t ldxd, int64_t M, int64_t N,
                                   int64_t K, float *y, int64_t ldy, int32_t *block_sums,
                                   void *stream);

/*
 * The expert-batched product of q4_0_x_q4_gemm_tc_experts on the experts' Q4_0
 * planes, widened in shared memory as in q4_0_x_q4_gemm_tc_widen.
 *   wq     [E][N][K/2] Q4_0 codes;  wd [E][N][K/32] fp16 scales (the experts'
 *          planes stacked as E * N rows)
 *   xw, xdt, ldxd   in grouped order, from h32_quantize_act_q4_tc_e5m2_gather
 *                   (or h32_quantize_act_q4_tc_e5m2 of rows already grouped)
 *   expert_off, R, y, block_sums as for q4_0_x_q4_gemm_tc_experts
 * Requires 1 <= E <= 1024, K % 256 == 0 and N % 16 == 0.
 */
h32_status q4_0_x_q4_gemm_tc_widen_experts(const uint8_t *wq, const uint16_t *wd, int32_t E,
                                           const uint8_t *xw, const float *xdt, int64_t ldxd,
                                           const int32_t *expert_off, int64_t R, int64_t N,
                                           int64_t K, float *y, int64_t ldy,
                                           int32_t *block_sums, void *stream);

/*
 * The W4A8 product of q4_0_x_q8_gemm on tc-form operands (weights from
 * h32_prepack_weights_q4_0_tc, activations from h32_quantize_act_q8_tc):
 * S = sum w (16 h) + sum w l per block (two MMAs into one accumulator, every
 * partial sum an integer below 2^24, so S is exact), then the same epilogue;
 * bit-identical to q4_0_x_q8_gemm.  Requires K % 128 == 0 and N % 16 == 0.
 */
h32_status q4_0_x_q8_gemm_tc(const uint8_t *wp, const float *wsc, int64_t ldws,
                             const uint8_t *xw8, const float *xdt, int64_t ldxd, int64_t M,
                             int64_t N, int64_t K, float *y, int64_t ldy, int32_t *block_sums,
                             void *stream);

/*
 * ---------------------------------------------------------------------------
 * The K split of the last wave.  The tc GEMMs run one persistent block per SM
 * over 128 x (up to 128)-token tiles; where the tiles do not fill the last
 * wave, its tiles are cut along the tokens, and with a workspace each cut piece
 * also runs in two parts along K on two SMs: the first part before that SM's
 * full tiles, the second after another SM's, continuing the first part's
 * accumulators.  Every output still takes its 32-blocks in order, so the result
 * is bit-identical to q4_0_x_q4_gemm_tc; only the schedule changes (on the
 * 512-token projections of the chain the last wave shrinks from about half a
 * tile to a quarter).
 * ---------------------------------------------------------------------------
 */

/*
 * Workspace bytes the _ws entry points need for an M x N x K product on the
 * current device: 0 when the schedule does not split (then no workspace is
 * used).  The plan depends on M, N, K and the device's SM count only.
 * Returns H32_ERR_INVALID_ARG for shapes the GEMMs reject (K % 128, N % 16).
 */
h32_status h32_gemm_tc_workspace_bytes(int64_t M, int64_t N, int64_t K, size_t *bytes);

/*
 * The schedule the dense tc GEMMs (plain output) take for an M x N x K product
 * on a device of `sms` SMs, with a workspace (with_workspace != 0) or without:
 * host arithmetic only, no device call.  out[9] receives: tokens per tile,
 * pieces per cut tile, the first cut tile, the number of work units (uncut
 * tiles + pieces), the grid, the pieces split along K (0: none), the K stages
 * (of 128) of a piece's first part, the piece width (workspace row stride) and
 * the workspace bytes.  Requires M >= 1, K % 128 == 0, N % 16 == 0.
 */
h32_status h32_gemm_tc_schedule(int64_t M, int64_t N, int64_t K, int32_t sms,
                                int32_t with_workspace, int64_t *out);

/*
 * q4_0_x_q4_gemm_tc / q4_0_x_q8_gemm_tc with a caller-owned workspace for the
 * K split (same arguments, same results, bit for bit):
 *   workspace        device memory, 256-byte aligned, or null (no split: the
 *                    plain entry point's schedule); zero-filled once before its
 *                    first use, after which every call leaves it valid for the
 *                    next (a header with a generation number that the kernel
 *                    advances, so flags of earlier calls, or of earlier replays
 *                    of a captured graph, never match)
 *   workspace_bytes  its size; below h32_gemm_tc_workspace_bytes(M, N, K) ->
 *                    H32_ERR_INVALID_ARG
 * A workspace serves one call at a time: calls that share one must be ordered
 * (one stream, or events).  With block_sums the schedule never splits.  The
 * second part of a piece waits, bounded, for the first part's flag; a timeout
 * is reported as H32_ERR_TIMEOUT like every other wait of the kernel.
 */
h32_status q4_0_x_q4_gemm_tc_ws(const uint8_t *wp, const float *wsc, int64_t ldws,
                                const uint8_t *xw, const float *xdt, int64_t ldxd, int64_t M,
                                int64_t N, int64_t K, float *y, int64_t ldy, int32_t *block_sums,
                                void *workspace, size_t workspace_bytes, void *stream);
h32_status q4_0_x_q8_gemm_tc_ws(const uint8_t *wp, const float *wsc, int64_t ldws,
                                const uint8_t *xw8, const float *xdt, int64_t ldxd, int64_t M,
                                int64_t N, int64_t K, float *y, int64_t ldy, int32_t *block_sums,
                                void *workspace, size_t workspace_bytes, void *stream);

/*
 * q4_0_x_q4_gemm_tc / q4_0_x_q8_gemm_tc with the K split, without a caller's
 * workspace and without allocating: the workspace is a 4 MB array the library
 * holds in each device's static memory (zero when the library's module is
 * loaded, kept valid by every call).  Same arguments and results as the plain
 * entry points.  A product whose schedule needs more than 4 MB of workspace
 * is refused with H32_ERR_UNSUPPORTED (nothing is allocated in its place); on
 * 152 SMs the pp512 chain's shapes need 0.5 MB.  All calls on one device share
 * the array: calls that may overlap must be ordered (one stream, or events).
 */
h32_status q4_0_x_q4_gemm_tc_noalloc(const uint8_t *wp, const float *wsc, int64_t ldws,
                                     const uint8_t *xw, const float *xdt, int64_t ldxd,
                                     int64_t M, int64_t N, int64_t K, float *y, int64_t ldy,
                                     int32_t *block_sums, void *stream);
h32_status q4_0_x_q8_gemm_tc_noalloc(const uint8_t *wp, const float *wsc, int64_t ldws,
                                     const uint8_t *xw8, const float *xdt, int64_t ldxd,
                                     int64_t M, int64_t N, int64_t K, float *y, int64_t ldy,
                                     int32_t *block_sums, void *stream);

/*
 * Expert-batched W4A4 product on tc-form operands (the tc counterpart of
 * q4_0_x_q4_gemm_experts): rows r in [expert_off[e], expert_off[e+1]) of
 * xw/xdt (already in grouped order, e.g. from h32_quantize_act_q4_tc_gather)
 * are multiplied by expert e's weights:
 *   y[r][n] = same definition as q4_0_x_q4_gemm_tc with the weights of expert e
 *   wp     [E][N][K] bytes, wsc [E][N][ldws] fp32 (h32_prepack_weights_q4_0_tc of
 *          the E experts' planes stacked as E * N rows)
 *   expert_off [E+1] int32 device: 0 = off[0] <= off[1] <= ... <= off[E] = R,
 *          else H32_ERR_DEVICE_GUARD is recorded and nothing is computed
 *   y      [R][ldy] fp32 out in grouped order; block_sums nullable int32 [R][N][K/32]
 * Requires 1 <= E <= 1024, K % 128 == 0 and N % 16 == 0.
 */
h32_status q4_0_x_q4_gemm_tc_experts(const uint8_t *wp, const float *wsc, int64_t ldws, int32_t E,
                                     const uint8_t *xw, const float *xdt, int64_t ldxd,
                                     const int32_t *expert_off, int64_t R, int64_t N, int64_t K,
                                     float *y, int64_t ldy, int32_t *block_sums, void *stream);

/*
 * Routing around the expert GEMMs ("Where the engine is going: HRX and the
 * NPU", section "4-bit activations reach the MoE experts": the route covers
 * the expert matmuls of a mixture-of-experts model; the pages do not spell
 * out the router, so the reading taken is stated here).  Per token t:
 *   - its k experts are those of largest logit, ties to the lower expert id,
 *     listed by decreasing logit (the softmax is monotonic, so these are the
 *     k most probable experts);
 *   - choice j weighs w_j = e_j / s with e_j = exp(l_j - l_0) in fp32 and
 *     s = the fp32 sum of e_0 .. e_{k-1} in that order (the full softmax's
 *     top-k probabilities renormalised to sum to 1);
 * then the (token, choice) pairs are grouped by expert id, and within an
 * expert by token, which is the grouped order of h32_quantize_act_q4_tc_gather
 * and q4_0_x_q4_gemm_tc_experts.  Deterministic; the ids, offsets and row maps
 * are exact, the weights are within a few ulps of an IEEE fp32 evaluation
 * (the exp is the CUDA libm expf).
 *   logits     [T][ldl] fp32 device, ldl >= E (4-byte aligned)
 *   topk_id    [T][k] int32 out: the chosen experts (16-byte aligned; the other
 *              outputs 4-byte aligned)
 *   topk_w     [T][k] fp32 out: their weights
 *   expert_off [E+1] int32 out: group e holds grouped rows [off[e], off[e+1]); off[E] = T k
 *   row_idx    [T k] int32 out: the token of grouped row r
 *   row_of     [T][k] int32 out: the grouped row of choice j of token t
 * Logits that are not finite (masked experts) follow the limits of the same
 * rule: a NaN ranks below every number, -inf included (NaNs among themselves
 * by id); a chosen -inf or NaN weighs 0 when the largest chosen logit l_0 is
 * finite; when l_0 = +inf the +inf choices share the weight equally; when
 * l_0 is -inf or NaN (every logit masked) the k weights are equal.
 * Requires 1 <= E <= 1024, 1 <= k <= min(E, 32), T k < 2^31.  T = 0 writes
 * all-zero offsets.
 */
h32_status h32_moe_route(const float *logits, int64_t T, int32_t E, int64_t ldl, int32_t k,
                         int32_t *topk_id, float *topk_w, int32_t *expert_off, int32_t *row_idx,
                         int32_t *row_of, void *stream);

/*
 * The weighted combine after the expert GEMMs: the k expert outputs of each
 * token, in grouped order, added back in token order:
 *   out[t][h] = acc after acc = fma(topk_w[t][j], y[row_of[t][j]][h], acc)
 *               for j = 0 .. k-1, from acc = +0 (fp32)
 *   y       [R][ldy] fp32 device (grouped rows, e.g. the down projection of
 *           q4_0_x_q4_gemm_tc_experts); row_of, topk_w as from h32_moe_route
 *   out     [T][ldo] fp32 out
 * Requires 1 <= k <= 32, H % 4 == 0, ldy, ldo >= H and multiples of 4, y and
 * out 16-byte aligned.  A row index outside [0, R) records
 * H32_ERR_DEVICE_GUARD (see h32_device_status) and adds nothing.
 */
h32_status h32_moe_combine(const float *y, int64_t R, int64_t ldy, const int32_t *row_of,
                           const float *topk_w, int64_t T, int32_t k, int64_t H, float *out,
                           int64_t ldo, void *stream);

/*
 * Synchronize `stream`, then report and clear the device status words that
 * this library's kernels on the current device write: H32_OK, H32_ERR_TIMEOUT
 * or H32_ERR_DEVICE_GUARD (or H32_ERR_CUDA when the synchronization, or a
 * copy, fails).  The words are shared by every stream of the device.  Each is
 * read and cleared in one atomic step on the device, so a problem recorded
 * by a kernel that is still running on another stream is reported by this
 * call or by a later one, never lost.  Calls from several host threads are
 * serialized.
 */
h32_status h32_device_status(void *stream);

/* Human-readable name of a status code (static storage). */
const char *h32_status_string(h32_status status);

/*
 * Bound on every spin wait inside the kernels, in polling iterations
 * (0 restores the default of about a second).  Kernels launched after the
 * call use the new bound; a wait that exceeds it makes the kernel record
 * H32_ERR_TIMEOUT, drain its own in-flight copies and return.  Meant for
 * tests of the timeout path.
 */
void h32_set_wait_limit(uint64_t polls);

/* Text of the most recent CUDA failure seen by the library on the calling
 * thread (after an H32_ERR_CUDA status); static storage, never NULL. */
const char *h32_last_cuda_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int h32_version(void);

#ifdef __cplusplus
}
#endif

#endif /* H32_H */
