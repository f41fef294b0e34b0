/*
 * c_abi_check.c -- the C ABI driven from plain C: no Python, no torch.
 *
 * Reads bf16 inputs (raw uint16 files written by the test that builds and
 * runs this program), allocates every device buffer itself with cudaMalloc,
 * describes the grouped tensors with gq_quantized, and runs the MXFP8
 * quantisation of X and W, the grouped fprop and the k-grouped wgrad, plus
 * two calls that must be refused on the host.  Results go to raw files for
 * the test to compare with the oracle.  Then it resets the device
 * (cudaDeviceReset: the library's per-context set-up and the no-alloc
 * wgrad's array address must be redone in the new context), allocates and
 * quantises again, and checks that the no-alloc wgrad gives the same bits.
 *
 * usage: c_abi_check DIR G R K N
 *   DIR/splits.bin  int32[G]          DIR/x.bin  uint16[R][K]  (bf16 bits)
 *   DIR/w.bin       uint16[G*N][K]    DIR/dy.bin uint16[R][N]
 * writes DIR/y.bin (float[R][N]), DIR/dw.bin (float[G][N][K]),
 *        DIR/xrow.bin (uint8[R][K] rowwise codes), DIR/status.txt
 *        ("status refused_cols refused_shape reset_status reset_equal")
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "gq.h"

#define CHECK_CUDA(x)                                                              \
    do {                                                                           \
        cudaError_t e_ = (x);                                                      \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "%s failed: %s\n", #x, cudaGetErrorString(e_));        \
            return 2;                                                              \
        }                                                                          \
    } while (0)

#define CHECK_GQ(x)                                                                \
    do {                                                                           \
        gq_status s_ = (x);                                                        \
        if (s_ != GQ_OK) {                                                         \
            fprintf(stderr, "%s failed: %s\n", #x, gq_status_string(s_));          \
            return 3;                                                              \
        }                                                                          \
    } while (0)

static void* read_file(const char* dir, const char* name, size_t bytes)
{
    char path[1024];
    void* buf = malloc(bytes ? bytes : 1);
    FILE* f;
    snprintf(path, sizeof path, "%s/%s", dir, name);
    f = fopen(path, "rb");
    if (!f || !buf || fread(buf, 1, bytes, f) != bytes) {
        fprintf(stderr, "cannot read %s\n", path);
        exit(4);
    }
    fclose(f);
    return buf;
}

static int write_file(const char* dir, const char* name, const void* buf, size_t bytes)
{
    char path[1024];
    FILE* f;
    snprintf(path, sizeof path, "%s/%s", dir, name);
    f = fopen(path, "wb");
    if (!f || fwrite(buf, 1, bytes, f) != bytes)
        return 1;
    fclose(f);
    return 0;
}

/* Device buffers of an MX-quantised [rows, cols] tensor with both orientations. */
static int alloc_mx(gq_quantized* q, int32_t G, int64_t rows, int64_t cols)
{
    gq_recipe rec = {GQ_RECIPE_MXFP8_1X32, 1, 1, 0.0f};
    uint64_t sb = gq_scale_bytes_bound(&rec, G, rows, cols);
    q->num_groups = G;
    q->reserved0 = 0;
    q->rows_cap = rows;
    q->cols = cols;
    q->recipe = rec;
    q->row_scale_bytes = q->col_scale_bytes = sb;
    q->amax = NULL;
    if (cudaMalloc(&q->row_data, (size_t)(rows * cols)) != cudaSuccess ||
        cudaMalloc(&q->col_data, (size_t)(rows * cols)) != cudaSuccess ||
        cudaMalloc(&q->row_scale, (size_t)sb) != cudaSuccess || cudaMalloc(&q->col_scale, (size_t)sb) != cudaSuccess)
        return 1;
    return 0;
}

int main(int argc, char** argv)
{
    const char* dir;
    int32_t G;
    int64_t R, K, N;
    int32_t *h_splits, *d_splits, *d_status, h_status = 0;
    uint16_t *h_x, *h_w, *h_dy;
    void *d_x, *d_w, *d_dy;
    float *d_y, *d_dw, *h_y, *h_dw;
    uint8_t* h_xrow;
    gq_quantized qx, qw, qdy;
    gq_recipe mx = {GQ_RECIPE_MXFP8_1X32, 1, 1, 0.0f};
    cudaStream_t stream;
    gq_status refused_cols, refused_shape;
    FILE* f;
    char path[1024];

    if (argc != 6) {
        fprintf(stderr, "usage: %s DIR G R K N\n", argv[0]);
        return 1;
    }
    dir = argv[1];
    G = atoi(argv[2]);
    R = atoll(argv[3]);
    K = atoll(argv[4]);
    N = atoll(argv[5]);
    if ((gq_version() >> 16) != 1) {
        fprintf(stderr, "unexpected ABI major version %d\n", gq_version() >> 16);
        return 1;
    }

    h_splits = (int32_t*)read_file(dir, "splits.bin", sizeof(int32_t) * (size_t)G);
    h_x = (uint16_t*)read_file(dir, "x.bin", 2 * (size_t)(R * K));
    h_w = (uint16_t*)read_file(dir, "w.bin", 2 * (size_t)(G * N * K));
    h_dy = (uint16_t*)read_file(dir, "dy.bin", 2 * (size_t)(R * N));

    CHECK_CUDA(cudaStreamCreate(&stream));
    CHECK_CUDA(cudaMalloc((void**)&d_splits, sizeof(int32_t) * (size_t)G));
    CHECK_CUDA(cudaMalloc((void**)&d_status, sizeof(int32_t)));
    CHECK_CUDA(cudaMalloc(&d_x, 2 * (size_t)(R * K)));
    CHECK_CUDA(cudaMalloc(&d_w, 2 * (size_t)(G * N * K)));
    CHECK_CUDA(cudaMalloc(&d_dy, 2 * (size_t)(R * N)));
    CHECK_CUDA(cudaMalloc((void**)&d_y, sizeof(float) * (size_t)(R * N)));
    CHECK_CUDA(cudaMalloc((void**)&d_dw, sizeof(float) * (size_t)(G * N * K)));
    CHECK_CUDA(cudaMemcpyAsync(d_splits, h_splits, sizeof(int32_t) * (size_t)G, cudaMemcpyHostToDevice, stream));
    CHECK_CUDA(cudaMemcpyAsync(d_x, h_x, 2 * (size_t)(R * K), cudaMemcpyHostToDevice, stream));
    CHECK_CUDA(cudaMemcpyAsync(d_w, h_w, 2 * (size_t)(G * N * K), cudaMemcpyHostToDevice, stream));
    CHECK_CUDA(cudaMemcpyAsync(d_dy, h_dy, 2 * (size_t)(R * N), cudaMemcpyHostToDevice, stream));
    CHECK_CUDA(cudaMemsetAsync(d_status, 0, sizeof(int32_t), stream));
    if (alloc_mx(&qx, G, R, K) || alloc_mx(&qw, G, (int64_t)G * N, K) || alloc_mx(&qdy, G, R, N)) {
        fprintf(stderr, "cudaMalloc of the quantised buffers failed\n");
        return 2;
    }

    /* host-side refusals: nothing is launched */
    refused_cols = gq_quantize(d_x, R, K - 64, d_splits, G, &mx, &qx, d_status, (gq_stream_t)stream);
    qdy.cols = N + 128;
    refused_shape = gq_quantize(d_dy, R, N, d_splits, G, &mx, &qdy, d_status, (gq_stream_t)stream);
    qdy.cols = N;

    CHECK_GQ(gq_quantize(d_x, R, K, d_splits, G, &mx, &qx, d_status, (gq_stream_t)stream));
    CHECK_GQ(gq_quantize(d_w, (int64_t)G * N, K, NULL, G, &mx, &qw, d_status, (gq_stream_t)stream));
    CHECK_GQ(gq_quantize(d_dy, R, N, d_splits, G, &mx, &qdy, d_status, (gq_stream_t)stream));
    CHECK_GQ(gq_gemm_fprop(&qx, &qw, d_splits, G, N, K, d_y, GQ_DTYPE_F32, d_status, (gq_stream_t)stream));
    CHECK_GQ(gq_gemm_wgrad_noalloc(&qdy, &qx, d_splits, G, N, K, d_dw, 0, d_status, (gq_stream_t)stream));

    h_y = (float*)malloc(sizeof(float) * (size_t)(R * N));
    h_dw = (float*)malloc(sizeof(float) * (size_t)(G * N * K));
    h_xrow = (uint8_t*)malloc((size_t)(R * K));
    CHECK_CUDA(cudaMemcpyAsync(h_y, d_y, sizeof(float) * (size_t)(R * N), cudaMemcpyDeviceToHost, stream));
    CHECK_CUDA(cudaMemcpyAsync(h_dw, d_dw, sizeof(float) * (size_t)(G * N * K), cudaMemcpyDeviceToHost, stream));
    CHECK_CUDA(cudaMemcpyAsync(h_xrow, qx.row_data, (size_t)(R * K), cudaMemcpyDeviceToHost, stream));
    CHECK_CUDA(cudaMemcpyAsync(&h_status, d_status, sizeof(int32_t), cudaMemcpyDeviceToHost, stream));
    CHECK_CUDA(cudaStreamSynchronize(stream));

    if (write_file(dir, "y.bin", h_y, sizeof(float) * (size_t)(R * N)) ||
        write_file(dir, "dw.bin", h_dw, sizeof(float) * (size_t)(G * N * K)) ||
        write_file(dir, "xrow.bin", h_xrow, (size_t)(R * K)))
        return 5;

    /* a new context: everything again, the no-alloc wgrad must give the same bits */
    CHECK_CUDA(cudaDeviceReset());
    CHECK_CUDA(cudaStreamCreate(&stream));
    CHECK_CUDA(cudaMalloc((void**)&d_splits, sizeof(int32_t) * (size_t)G));
    CHECK_CUDA(cudaMalloc((void**)&d_status, sizeof(int32_t)));
    CHECK_CUDA(cudaMalloc(&d_x, 2 * (size_t)(R * K)));
    CHECK_CUDA(cudaMalloc(&d_dy, 2 * (size_t)(R * N)));
    CHECK_CUDA(cudaMalloc((void**)&d_dw, sizeof(float) * (size_t)(G * N * K)));
    CHECK_CUDA(cudaMemcpyAsync(d_splits, h_splits, sizeof(int32_t) * (size_t)G, cudaMemcpyHostToDevice, stream));
    CHECK_CUDA(cudaMemcpyAsync(d_x, h_x, 2 * (size_t)(R * K), cudaMemcpyHostToDevice, stream));
    CHECK_CUDA(cudaMemcpyAsync(d_dy, h_dy, 2 * (size_t)(R * N), cudaMemcpyHostToDevice, stream));
    CHECK_CUDA(cudaMemsetAsync(d_status, 0, sizeof(int32_t), stream));
    if (alloc_mx(&qx, G, R, K) || alloc_mx(&qdy, G, R, N)) {
        fprintf(stderr, "cudaMalloc of the quantised buffers failed after the reset\n");
        return 2;
    }
    CHECK_GQ(gq_quantize(d_x, R, K, d_splits, G, &mx, &qx, d_status, (gq_stream_t)stream));
    CHECK_GQ(gq_quantize(d_dy, R, N, d_splits, G, &mx, &qdy, d_status, (gq_stream_t)stream));
    CHECK_GQ(gq_gemm_wgrad_noalloc(&qdy, &qx, d_splits, G, N, K, d_dw, 0, d_status, (gq_stream_t)stream));
    {
        float* h_dw2 = (float*)malloc(sizeof(float) * (size_t)(G * N * K));
        int32_t h_status2 = 0;
        int equal = 1;
        size_t i;
        CHECK_CUDA(cudaMemcpyAsync(h_dw2, d_dw, sizeof(float) * (size_t)(G * N * K), cudaMemcpyDeviceToHost, stream));
        CHECK_CUDA(cudaMemcpyAsync(&h_status2, d_status, sizeof(int32_t), cudaMemcpyDeviceToHost, stream));
        CHECK_CUDA(cudaStreamSynchronize(stream));
        for (i = 0; i < (size_t)(G * N * K); ++i)
            if (memcmp(&h_dw2[i], &h_dw[i], sizeof(float)) != 0) {
                equal = 0;
                break;
            }
        snprintf(path, sizeof path, "%s/status.txt", dir);
        f = fopen(path, "w");
        if (!f)
            return 5;
        fprintf(f, "%d %d %d %d %d\n", (int)h_status, (int)refused_cols, (int)refused_shape, (int)h_status2, equal);
        fclose(f);
        free(h_dw2);
    }
    return 0;
}
