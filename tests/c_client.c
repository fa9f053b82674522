/*
 * A plain C client of libgar.so: it uses only include/gar.h and the CUDA
 * runtime, no Python.  It all-reduces P = 4 replicas of N fp32 values
 * (Sum, in place) and runs one bucketed Mean with the fused SGD step, then
 * checks the results against values it computes itself (integer-valued
 * inputs, so every sum is exact).  Exit code 0 on success.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdio.h>
#include <stdlib.h>

#include "gar.h"

#define P 4
#define N 100003

#define CHECK_AR(call)                                                              \
    do {                                                                            \
        ar_status_t s_ = (call);                                                    \
        if (s_ != AR_OK) {                                                          \
            fprintf(stderr, "%s failed: %s\n", #call, ar_status_string(s_));        \
            return 1;                                                               \
        }                                                                           \
    } while (0)

#define CHECK_CUDA(call)                                                            \
    do {                                                                            \
        cudaError_t e_ = (call);                                                    \
        if (e_ != cudaSuccess) {                                                    \
            fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_));      \
            return 1;                                                               \
        }                                                                           \
    } while (0)

int main(void)
{
    static float host[P][N], out[N];
    float *dev[P];
    for (int r = 0; r < P; ++r) {
        for (int i = 0; i < N; ++i)
            host[r][i] = (float)((i * 7 + r * 13) % 101 - 50);
        CHECK_CUDA(cudaMalloc((void **)&dev[r], N * sizeof(float)));
        CHECK_CUDA(cudaMemcpy(dev[r], host[r], N * sizeof(float), cudaMemcpyHostToDevice));
    }
    ar_comm_t comm;
    CHECK_AR(ar_init(&comm, P, 0, AR_SUM));
    cudaStream_t stream;
    CHECK_CUDA(cudaStreamCreate(&stream));

    /* all-reduce, Sum, in place */
    CHECK_AR(ar_all_reduce(comm, (const void *const *)dev, (void *const *)dev, N, AR_F32,
                           AR_OP_DEFAULT, (ar_stream_t)stream));
    CHECK_CUDA(cudaStreamSynchronize(stream));
    for (int r = 0; r < P; ++r) {
        CHECK_CUDA(cudaMemcpy(out, dev[r], N * sizeof(float), cudaMemcpyDeviceToHost));
        for (int i = 0; i < N; ++i) {
            float want = host[0][i] + host[1][i] + host[2][i] + host[3][i];
            if (out[i] != want) {
                fprintf(stderr, "all-reduce: rank %d element %d: %g != %g\n", r, i, out[i], want);
                return 1;
            }
        }
    }

    /* one bucket (two tensors), Mean, fused SGD (lr 0.5, momentum 0.5) */
    float *w, *v;
    CHECK_CUDA(cudaMalloc((void **)&w, N * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void **)&v, N * sizeof(float)));
    CHECK_CUDA(cudaMemset(w, 0, N * sizeof(float)));
    CHECK_CUDA(cudaMemset(v, 0, N * sizeof(float)));
    size_t split = 4096, numel[2] = {split, N - split};
    void *ptrs[2 * P];
    float *masters[2] = {w, w + split}, *moms[2] = {v, v + split};
    for (int r = 0; r < P; ++r) {
        ptrs[r] = dev[r];
        ptrs[P + r] = dev[r] + split;
    }
    ar_bucket_t bucket = {2, ptrs, numel, AR_F32};
    ar_sgd_t sgd = {0.5f, 0.5f, masters, moms, 0};
    CHECK_AR(ar_bucket_all_reduce(comm, &bucket, AR_MEAN, &sgd, (ar_stream_t)stream));
    CHECK_AR(ar_get_async_error(comm));
    CHECK_CUDA(cudaMemcpy(out, w, N * sizeof(float), cudaMemcpyDeviceToHost));
    for (int i = 0; i < N; ++i) {
        /* every replica holds s (the Sum above): Mean = s, v = s, w = -0.5 s, all exact */
        float s = host[0][i] + host[1][i] + host[2][i] + host[3][i];
        if (out[i] != -0.5f * s) {
            fprintf(stderr, "bucket SGD: element %d: %g != %g\n", i, out[i], -0.5f * s);
            return 1;
        }
    }

    /* refusals happen on the host, before anything is enqueued */
    if (ar_all_reduce(comm, (const void *const *)dev, (void *const *)dev, N, (ar_dtype_t)9,
                      AR_SUM, NULL) != AR_ERR_INVALID_ARG)
        return 1;
    CHECK_AR(ar_destroy(comm));
    if (ar_destroy(comm) != AR_ERR_STATE)
        return 1;
    for (int r = 0; r < P; ++r)
        cudaFree(dev[r]);
    cudaFree(w);
    cudaFree(v);
    cudaStreamDestroy(stream);
    printf("c_client: ok\n");
    return 0;
}
