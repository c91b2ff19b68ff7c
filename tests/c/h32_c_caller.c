/*
 * A plain C caller of the h32 library: no Python, no torch, only the C ABI of
 * include/h32.h and the CUDA runtime.  It reads fp32 activations x [M][K] and
 * fp32 weights w [N][K] from a binary input file, runs the tensor-core route
 * (rotate + quantize the activations, rotate + quantize the weights to Q4_0,
 * repack them, the W4A4 GEMM) and writes y [M][N] fp32 to the output file;
 * when K % 256 == 0 it then runs the widening route on the same Q4_0 planes
 * (activations as e5m2 bytes, the GEMM that widens the nibbles itself) and
 * appends its y [M][N]; when the schedule splits the last wave along K on
 * this device, it also runs the tensor-core GEMM with a workspace of its own
 * (cudaMalloc'd, zeroed once, used twice) and the no-alloc form, appending
 * their y [M][N].
 *
 * Input file: int64 M, N, K, then x and w as fp32, row-major.
 * Output file: int64 R (the number of results), then R results y [M][N] fp32.
 * Usage: h32_c_caller <input> <output>.  Exit status 0 = success, 1 = a
 * library status that is not H32_OK (printed), 2 = I/O or CUDA runtime error.
 * Test infrastructure: built and run by tests/test_c_caller.py.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "h32.h"

#define CUDA_OK(call)                                                              \
    do {                                                                           \
        cudaError_t e_ = (call);                                                   \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));            \
            return 2;                                                              \
        }                                                                          \
    } while (0)

#define H32_OK_OR_FAIL(call)                                                       \
    do {                                                                           \
        h32_status s_ = (call);                                                    \
        if (s_ != H32_OK) {                                                        \
            fprintf(stderr, "%s: %s\n", #call, h32_status_string(s_));             \
            return 1;                                                              \
        }                                                                          \
    } while (0)

static int64_t round4(int64_t n) { return (n + 3) / 4 * 4; }

int main(int argc, char **argv) {
    if (argc != 3) {
        fprintf(stderr, "usage: %s <input> <output>\n", argv[0]);
        return 2;
    }
    FILE *f = fopen(argv[1], "rb");
    if (!f) return 2;
    int64_t dims[3];
    if (fread(dims, sizeof(int64_t), 3, f) != 3) return 2;
    const int64_t M = dims[0], N = dims[1], K = dims[2], nb = K / 32;
    float *hx = malloc(sizeof(float) * M * K), *hw = malloc(sizeof(float) * N * K);
    float *hy = malloc(sizeof(float) * M * N * 5);
    if (!hx || !hw || !hy) return 2;
    if (fread(hx, sizeof(float), M * K, f) != (size_t)(M * K)) return 2;
    if (fread(hw, sizeof(float), N * K, f) != (size_t)(N * K)) return 2;
    fclose(f);

    const int64_t ldxd = round4(M), ldws = round4(nb);
    float *x, *w, *xdt, *wsc, *y;
    uint8_t *xw, *wq, *wp;
    uint16_t *wd;
    cudaStream_t stream;
    CUDA_OK(cudaStreamCreate(&stream));
    CUDA_OK(cudaMalloc((void **)&x, sizeof(float) * M * K));
    CUDA_OK(cudaMalloc((void **)&w, sizeof(float) * N * K));
    CUDA_OK(cudaMalloc((void **)&xw, (size_t)(M * K)));
    CUDA_OK(cudaMalloc((void **)&xdt, sizeof(float) * nb * ldxd));
    CUDA_OK(cudaMalloc((void **)&wq, (size_t)(N * K / 2)));
    CUDA_OK(cudaMalloc((void **)&wd, sizeof(uint16_t) * N * nb));
    CUDA_OK(cudaMalloc((void **)&wp, (size_t)(N * K)));
    CUDA_OK(cudaMalloc((void **)&wsc, sizeof(float) * N * ldws));
    CUDA_OK(cudaMalloc((void **)&y, sizeof(float) * M * N * 5));
    CUDA_OK(cudaMemsetAsync(xdt, 0, sizeof(float) * nb * ldxd, stream));
    CUDA_OK(cudaMemcpyAsync(x, hx, sizeof(float) * M * K, cudaMemcpyHostToDevice, stream));
    CUDA_OK(cudaMemcpyAsync(w, hw, sizeof(float) * N * K, cudaMemcpyHostToDevice, stream));

    H32_OK_OR_FAIL(h32_rotate_quantize_weights_q4_0(w, N, K, 1, wq, wd, stream));
    H32_OK_OR_FAIL(h32_prepack_weights_q4_0_tc(wq, wd, N, K, wp, wsc, ldws, stream));
    H32_OK_OR_FAIL(h32_quantize_act_q4_tc(x, H32_IN_F32, M, K, K, xw, xdt, ldxd, 1, stream));
    H32_OK_OR_FAIL(q4_0_x_q4_gemm_tc(wp, wsc, ldws, xw, xdt, ldxd, M, N, K, y, N, NULL, stream));
    int64_t routes = 1;
    size_t ws_bytes = 0;
    H32_OK_OR_FAIL(h32_gemm_tc_workspace_bytes(M, N, K, &ws_bytes));
    if (ws_bytes > 0) {
        void *ws;
        CUDA_OK(cudaMalloc(&ws, ws_bytes));
        CUDA_OK(cudaMemsetAsync(ws, 0, ws_bytes, stream));
        for (int i = 0; i < 2; ++i)   /* the second call finds the workspace as the first left it */
            H32_OK_OR_FAIL(q4_0_x_q4_gemm_tc_ws(wp, wsc, ldws, xw, xdt, ldxd, M, N, K,
                                                y + routes * M * N, N, NULL, ws, ws_bytes, stream));
        ++routes;
        H32_OK_OR_FAIL(q4_0_x_q4_gemm_tc_noalloc(wp, wsc, ldws, xw, xdt, ldxd, M, N, K,
                                                 y + routes * M * N, N, NULL, stream));
        ++routes;
        CUDA_OK(cudaStreamSynchronize(stream));
        cudaFree(ws);
    }
    if ((K % 256) == 0) {
        H32_OK_OR_FAIL(h32_quantize_act_q4_tc_e5m2(x, H32_IN_F32, M, K, K, xw, xdt, ldxd, 1, stream));
        H32_OK_OR_FAIL(q4_0_x_q4_gemm_tc_widen(wq, wd, xw, xdt, ldxd, M, N, K, y + routes * M * N,
                                               N, NULL, stream));
        ++routes;
    }
    H32_OK_OR_FAIL(h32_device_status(stream));

    const int64_t nout = M * N * routes;
    CUDA_OK(cudaMemcpyAsync(hy, y, sizeof(float) * nout, cudaMemcpyDeviceToHost, stream));
    CUDA_OK(cudaStreamSynchronize(stream));
    f = fopen(argv[2], "wb");
    if (!f || fwrite(&routes, sizeof(int64_t), 1, f) != 1 ||
        fwrite(hy, sizeof(float), nout, f) != (size_t)nout)
        return 2;
    fclose(f);
    cudaFree(x); cudaFree(w); cudaFree(xw); cudaFree(xdt); cudaFree(wq);
    cudaFree(wd); cudaFree(wp); cudaFree(wsc); cudaFree(y);
    cudaStreamDestroy(stream);
    free(hx); free(hw); free(hy);
    printf("h32 C caller: %lld x %lld x %lld ok\n", (long long)M, (long long)N, (long long)K);
    return 0;
}
