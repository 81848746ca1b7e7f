/*
 * The C ABI of include/rr.h used from plain C11 (gcc, no CUDA compiler, no
 * Python): device buffers from the CUDA runtime, every collective entry
 * point called once, results checked exactly on the host.
 *
 * fp32 allreduce inputs are small integers, so every partial sum is exact
 * and the expected result is the integer sum whatever the order.  Gathers
 * move tagged int32 values.  Exit status 0 and "abi_from_c ok" on success;
 * any mismatch or error prints its reason and exits 1.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "rr.h"

#define W 4
#define N 1000 /* elements per rank: not a multiple of the 16-byte vector */

static int fail_cuda(cudaError_t e, const char *what)
{
    fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
    return 1;
}

static int check(rr_status st, const char *what)
{
    if (st != RR_OK) {
        fprintf(stderr, "%s: %s (%s)\n", what, rr_status_string(st), rr_last_error());
        return 1;
    }
    return 0;
}

int main(void)
{
    cudaError_t e;
    float *bufs[W], *outs[W];
    int32_t *shards[W], *gathered, *lists[W];
    float host_in[W][N], host_out[N];
    int32_t host_shard[W][N], host_gathered[W * N];

    for (int r = 0; r < W; ++r) {
        for (int i = 0; i < N; ++i) {
            host_in[r][i] = (float)((i * 7 + r * 13) % 101 - 50);
            host_shard[r][i] = r * 100000 + i;
        }
        if ((e = cudaMalloc((void **)&bufs[r], N * sizeof(float))) != cudaSuccess) return fail_cuda(e, "cudaMalloc");
        if ((e = cudaMalloc((void **)&outs[r], N * sizeof(float))) != cudaSuccess) return fail_cuda(e, "cudaMalloc");
        if ((e = cudaMalloc((void **)&shards[r], N * sizeof(int32_t))) != cudaSuccess) return fail_cuda(e, "cudaMalloc");
        if ((e = cudaMalloc((void **)&lists[r], N * sizeof(int32_t))) != cudaSuccess) return fail_cuda(e, "cudaMalloc");
        if ((e = cudaMemcpy(bufs[r], host_in[r], N * sizeof(float), cudaMemcpyHostToDevice)) != cudaSuccess)
            return fail_cuda(e, "cudaMemcpy");
        if ((e = cudaMemcpy(shards[r], host_shard[r], N * sizeof(int32_t), cudaMemcpyHostToDevice)) != cudaSuccess)
            return fail_cuda(e, "cudaMemcpy");
    }
    if ((e = cudaMalloc((void **)&gathered, W * N * sizeof(int32_t))) != cudaSuccess) return fail_cuda(e, "cudaMalloc");

    rr_signal_pad *pad = NULL;
    if (check(rr_signal_pad_create(W, 0, 0, &pad), "rr_signal_pad_create")) return 1;

    /* two-shot, then one-shot: every output is the element-wise sum */
    const void *const *no_inputs = NULL;
    if (check(rr_allreduce_twoshot(no_inputs, (void *const *)bufs, (void *const *)outs, W, N, RR_FP32, 0, pad, 0),
              "rr_allreduce_twoshot"))
        return 1;
    if (check(rr_signal_pad_status(pad, 0), "status after two-shot")) return 1;
    static const char *const names[3] = {"two-shot", "one-shot", "allocation-free one-shot"};
    for (int pass = 0; pass < 3; ++pass) {
        if (pass == 1) {
            if ((e = cudaMemset(outs[W - 1], 0xff, N * sizeof(float))) != cudaSuccess) return fail_cuda(e, "cudaMemset");
            if (check(rr_allreduce_oneshot(no_inputs, (void *const *)bufs, (void *const *)outs, W, N, RR_FP32, 0, pad, 0),
                      "rr_allreduce_oneshot"))
                return 1;
            if (check(rr_signal_pad_status(pad, 0), "status after one-shot")) return 1;
        }
        if (pass == 2) {
            /* no pad: the library's static signal array */
            for (int q = 0; q < W; ++q)
                if ((e = cudaMemset(outs[q], 0xff, N * sizeof(float))) != cudaSuccess) return fail_cuda(e, "cudaMemset");
            if (check(rr_allreduce_oneshot_noalloc(no_inputs, (void *const *)bufs, (void *const *)outs, W, N, RR_FP32,
                                                   0, 0),
                      "rr_allreduce_oneshot_noalloc"))
                return 1;
            if (check(rr_allreduce_oneshot_noalloc_status(0), "status after the allocation-free one-shot")) return 1;
        }
        for (int q = 0; q < W; ++q) {
            if ((e = cudaMemcpy(host_out, outs[q], N * sizeof(float), cudaMemcpyDeviceToHost)) != cudaSuccess)
                return fail_cuda(e, "cudaMemcpy");
            for (int i = 0; i < N; ++i) {
                float want = 0.0f;
                for (int r = 0; r < W; ++r) want += host_in[r][i];
                if (host_out[i] != want) {
                    fprintf(stderr, "%s output %d element %d: %g, want %g\n", names[pass], q, i, host_out[i], want);
                    return 1;
                }
            }
        }
    }

    /* rank-major allgather into rank 2's output only */
    void *gouts[W] = {NULL, NULL, gathered, NULL};
    if (check(rr_allgather((const void *const *)shards, gouts, W, N, RR_INT32, pad, 0), "rr_allgather")) return 1;
    if (check(rr_signal_pad_status(pad, 0), "status after allgather")) return 1;
    if ((e = cudaMemcpy(host_gathered, gathered, sizeof host_gathered, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return fail_cuda(e, "cudaMemcpy");
    for (int r = 0; r < W; ++r)
        for (int i = 0; i < N; ++i)
            if (host_gathered[r * N + i] != host_shard[r][i]) {
                fprintf(stderr, "allgather element %d of rank %d: %d\n", i, r, host_gathered[r * N + i]);
                return 1;
            }

    /* param-contiguous: two params of 600 and 400 elements per shard */
    const int64_t splits[2] = {600, 400};
    if (check(rr_allgather_param_contiguous((const void *const *)shards, gouts, W, splits, 2, RR_INT32, pad, 0),
              "rr_allgather_param_contiguous"))
        return 1;
    if ((e = cudaMemcpy(host_gathered, gathered, sizeof host_gathered, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return fail_cuda(e, "cudaMemcpy");
    for (int s = 0, o = 0; s < 2; o += (int)splits[s], ++s)
        for (int r = 0; r < W; ++r)
            for (int i = 0; i < splits[s]; ++i)
                if (host_gathered[o * W + r * splits[s] + i] != host_shard[r][o + i]) {
                    fprintf(stderr, "param-contiguous: param %d rank %d element %d wrong\n", s, r, i);
                    return 1;
                }

    /* list output: rank 1's list only (W buffers), rank-major order */
    void *list_rows[W * W];
    memset(list_rows, 0, sizeof list_rows);
    for (int r = 0; r < W; ++r) list_rows[1 * W + r] = lists[r];
    if (check(rr_allgather_list((const void *const *)shards, list_rows, W, N, RR_INT32, pad, 0), "rr_allgather_list"))
        return 1;
    for (int r = 0; r < W; ++r) {
        if ((e = cudaMemcpy(host_gathered, lists[r], N * sizeof(int32_t), cudaMemcpyDeviceToHost)) != cudaSuccess)
            return fail_cuda(e, "cudaMemcpy");
        if (memcmp(host_gathered, host_shard[r], N * sizeof(int32_t)) != 0) {
            fprintf(stderr, "list entry %d differs from rank %d's shard\n", r, r);
            return 1;
        }
    }

    /* an argument error comes back synchronously, with a message */
    void *misaligned[W] = {(char *)gathered + 4, NULL, NULL, NULL};
    rr_status st = rr_allgather((const void *const *)shards, misaligned, W, N, RR_INT32, pad, 0);
    if (st != RR_ERR_ALIGNMENT || strlen(rr_last_error()) == 0) {
        fprintf(stderr, "misaligned output: got %s\n", rr_status_string(st));
        return 1;
    }
    int64_t gen = 0;
    if (check(rr_signal_pad_get_option(pad, RR_OPT_GENERATION, &gen), "get generation")) return 1;
    if (gen != 5) {
        fprintf(stderr, "generation %lld after 5 launched calls\n", (long long)gen);
        return 1;
    }
    if (check(rr_signal_pad_destroy(pad), "rr_signal_pad_destroy")) return 1;
    for (int r = 0; r < W; ++r) {
        cudaFree(bufs[r]);
        cudaFree(outs[r]);
        cudaFree(shards[r]);
        cudaFree(lists[r]);
    }
    cudaFree(gathered);
    printf("abi_from_c ok\n");
    return 0;
}
