/*
 * A plain C99 client of the gbgemm C ABI: device buffers from the CUDA runtime,
 * one linear call (bias, GELU-tanh, epilogue input), the device status check, and
 * one call the library must reject.  Usage:
 *
 *   gemm_client DIR M N K
 *
 * reads DIR/A.bin [M,K], DIR/B.bin [N,K], DIR/bias.bin [N], DIR/R.bin [M,N] (raw
 * bf16, row-major, contiguous) and writes DIR/D.bin [M,N].  Exit status 0 on
 * success; otherwise a message on stderr.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "gbgemm.h"

static void* read_all(const char* dir, const char* name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "rb");
    void* buf = malloc(bytes ? bytes : 1);
    if (!f || !buf || fread(buf, 1, bytes, f) != bytes) {
        fprintf(stderr, "cannot read %zu bytes from %s\n", bytes, path);
        exit(10);
    }
    fclose(f);
    return buf;
}

static void* to_device(const void* host, size_t bytes) {
    void* dev = NULL;
    if (cudaMalloc(&dev, bytes ? bytes : 16) != cudaSuccess ||
        cudaMemcpy(dev, host, bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
        fprintf(stderr, "device copy of %zu bytes failed\n", bytes);
        exit(11);
    }
    return dev;
}

int main(int argc, char** argv) {
    if (argc != 5) {
        fprintf(stderr, "usage: %s DIR M N K\n", argv[0]);
        return 1;
    }
    const char* dir = argv[1];
    const int64_t M = atoll(argv[2]), N = atoll(argv[3]), K = atoll(argv[4]);
    const size_t a_bytes = (size_t)(M * K) * 2, b_bytes = (size_t)(N * K) * 2;
    const size_t v_bytes = (size_t)N * 2, mn_bytes = (size_t)(M * N) * 2;

    void* A = to_device(read_all(dir, "A.bin", a_bytes), a_bytes);
    void* B = to_device(read_all(dir, "B.bin", b_bytes), b_bytes);
    void* bias = to_device(read_all(dir, "bias.bin", v_bytes), v_bytes);
    void* R = to_device(read_all(dir, "R.bin", mn_bytes), mn_bytes);
    void* D = NULL;
    if (cudaMalloc(&D, mn_bytes) != cudaSuccess) return 12;
    cudaStream_t stream;
    if (cudaStreamCreate(&stream) != cudaSuccess) return 13;

    gb_status_t st = gb_gemm_linear(A, K, B, K, bias, R, N, GB_ACT_GELU_TANH, D, N, M, N, K, stream);
    if (st != GB_OK) {
        fprintf(stderr, "gb_gemm_linear: status %d: %s\n", (int)st, gb_last_error());
        return 2;
    }
    if ((st = gb_get_device_status(stream)) != GB_OK) {
        fprintf(stderr, "gb_get_device_status: status %d: %s\n", (int)st, gb_last_error());
        return 3;
    }
    char plan[256];
    gb_last_plan(plan, sizeof plan);
    printf("plan: %s\n", plan);

    /* a call the library must reject before touching the GPU */
    st = gb_gemm_linear(NULL, K, B, K, NULL, NULL, 0, GB_ACT_NONE, D, N, M, N, K, stream);
    if (st != GB_ERR_INVALID_ARG || !strstr(gb_last_error(), "A is null")) {
        fprintf(stderr, "null A: status %d, message '%s'\n", (int)st, gb_last_error());
        return 4;
    }

    void* out = malloc(mn_bytes);
    if (!out || cudaMemcpy(out, D, mn_bytes, cudaMemcpyDeviceToHost) != cudaSuccess) return 14;
    char path[4096];
    snprintf(path, sizeof path, "%s/D.bin", dir);
    FILE* f = fopen(path, "wb");
    if (!f || fwrite(out, 1, mn_bytes, f) != mn_bytes) return 15;
    fclose(f);
    printf("gbgemm %s: ok\n", gb_version());
    return 0;
}
