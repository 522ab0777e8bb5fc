/*
 * c_abi_example.c -- the library used from plain C through include/ar.h,
 * with no Python involved: device buffers from cudaMalloc, inputs copied in,
 * ar_residual_rmsnorm, ar_sum and the Lamport-style call (its buffer sized,
 * allocated and filled through the ABI) on a stream, outputs copied back.
 *
 * Usage: c_abi_example <in.bin> <out.bin>
 *   in.bin   R=4 fp32 partials [T, H], then residual [T, H], bias [H],
 *            weight [H] (T = 3, H = 1000, eps = 1e-5 fixed below)
 *   out.bin  out [T, H], residual_out [T, H], the plain sum [T, H], then out
 *            and residual_out again from the Lamport-style call [T, H] each
 * Exit status 0 on success; a failing call prints its status text.
 */
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "ar.h"

enum { R = 4, T = 3, H = 1000 };

static int check_cuda(cudaError_t e, const char* what)
{
    if (e != cudaSuccess) {
        fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
        return 1;
    }
    return 0;
}

int main(int argc, char** argv)
{
    if (argc != 3) {
        fprintf(stderr, "usage: %s in.bin out.bin\n", argv[0]);
        return 2;
    }
    const size_t n = (size_t)T * H;
    const size_t in_count = R * n + n + 2 * (size_t)H;
    float* host_in = (float*)malloc(in_count * sizeof(float));
    float* host_out = (float*)malloc(5 * n * sizeof(float));
    FILE* f = fopen(argv[1], "rb");
    if (!f || fread(host_in, sizeof(float), in_count, f) != in_count) {
        fprintf(stderr, "cannot read %s\n", argv[1]);
        return 2;
    }
    fclose(f);

    float* dev = NULL;
    const size_t ws_bytes = ar_workspace_size_rows(R, H, T, AR_FP32);
    if (check_cuda(cudaMalloc((void**)&dev, (in_count + 5 * n) * sizeof(float) + ws_bytes), "cudaMalloc"))
        return 1;
    void* lamport = NULL;
    const size_t lamport_bytes = ar_lamport_buffer_size(R, H, T, AR_FP32);
    if (lamport_bytes == 0 || check_cuda(cudaMalloc(&lamport, lamport_bytes), "cudaMalloc lamport"))
        return 1;
    if (check_cuda(cudaMemcpy(dev, host_in, in_count * sizeof(float), cudaMemcpyHostToDevice), "copy in"))
        return 1;
    const void* partials[R];
    for (int r = 0; r < R; ++r)
        partials[r] = dev + (size_t)r * n;
    const float* residual = dev + R * n;
    const float* bias = residual + n;
    const float* weight = bias + H;
    float* out = dev + in_count;
    float* residual_out = out + n;
    float* sum = residual_out + n;
    float* lam_out = sum + n;
    float* lam_residual_out = lam_out + n;
    void* ws = lam_residual_out + n;

    cudaStream_t stream;
    if (check_cuda(cudaStreamCreate(&stream), "cudaStreamCreate"))
        return 1;
    int st = ar_residual_rmsnorm(partials, R, bias, residual, weight, 1e-5f, H, T, out, residual_out, ws,
                                 ws_bytes, AR_FP32, AR_AUTO, (ar_stream_t)stream);
    if (st != AR_OK) {
        fprintf(stderr, "ar_residual_rmsnorm: %s\n", ar_strerror(st));
        return 1;
    }
    st = ar_sum(partials, R, sum, n, AR_FP32, AR_TWOSHOT, (ar_stream_t)stream);
    if (st != AR_OK) {
        fprintf(stderr, "ar_sum: %s\n", ar_strerror(st));
        return 1;
    }
    int warps = 0;
    st = ar_lamport_supported(R, H, T, AR_FP32, &warps);
    if (st == AR_OK)
        st = ar_lamport_init(lamport, lamport_bytes, AR_FP32, (ar_stream_t)stream);
    if (st == AR_OK)
        st = ar_residual_rmsnorm_lamport(partials, R, bias, residual, weight, 1e-5f, H, T, lam_out,
                                         lam_residual_out, lamport, lamport_bytes, AR_FP32, (ar_stream_t)stream);
    if (st != AR_OK) {
        fprintf(stderr, "Lamport-style call: %s\n", ar_strerror(st));
        return 1;
    }
    if (check_cuda(cudaStreamSynchronize(stream), "sync") ||
        check_cuda(cudaMemcpy(host_out, out, 5 * n * sizeof(float), cudaMemcpyDeviceToHost), "copy out"))
        return 1;
    if (ar_device_status() != AR_OK) {
        fprintf(stderr, "ar_device_status: %s\n", ar_strerror(ar_device_status()));
        return 1;
    }
    f = fopen(argv[2], "wb");
    if (!f || fwrite(host_out, sizeof(float), 5 * n, f) != 5 * n) {
        fprintf(stderr, "cannot write %s\n", argv[2]);
        return 2;
    }
    fclose(f);
    cudaStreamDestroy(stream);
    cudaFree(dev);
    cudaFree(lamport);
    free(host_in);
    free(host_out);
    printf("c_abi_example: ok (version %d)\n", ar_version());
    return 0;
}
