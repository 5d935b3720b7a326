/* A plain C99 caller of the C ABI in include/ccl.h: no Python, no torch.
 *
 * It allocates p rank buffers with the CUDA runtime, fills rank r's element
 * e with the small integer ((r * 7 + e * 3) % 17) - 8 stored as float (sums
 * of such values are exact in any order), and checks on the host:
 *   - AllReduce (sum, ring) out of place: every rank holds the plain sum;
 *   - ReduceScatter (max, all-pairs) into rank r's own chunk, in place;
 *   - AllGather in place of the ReduceScatter result: every rank holds every
 *     chunk's maximum;
 *   - error statuses: n % p != 0 for ReduceScatter, a NULL rank pointer;
 *   - ccl_last_error() names the failure.
 * Exit status 0 when every check passes, 1 otherwise, 2 when no GPU is there.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "ccl.h"

#define P 5
#define N (P * 1003)

static float value(int r, int e) { return (float)(((r * 7 + e * 3) % 17) - 8); }

static int fails = 0;

static void check(int ok, const char *what)
{
    if (!ok) {
        fprintf(stderr, "FAIL: %s (%s)\n", what, ccl_last_error());
        ++fails;
    }
}

int main(void)
{
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
        fprintf(stderr, "no GPU\n");
        return 2;
    }
    float *host = (float *)malloc(sizeof(float) * N);
    float *in[P], *out[P];
    void *in_ptrs[P], *out_ptrs[P];
    for (int r = 0; r < P; ++r) {
        if (cudaMalloc((void **)&in[r], sizeof(float) * N) != cudaSuccess ||
            cudaMalloc((void **)&out[r], sizeof(float) * N) != cudaSuccess) {
            fprintf(stderr, "cudaMalloc failed\n");
            return 1;
        }
        for (int e = 0; e < N; ++e) host[e] = value(r, e);
        cudaMemcpy(in[r], host, sizeof(float) * N, cudaMemcpyHostToDevice);
        in_ptrs[r] = in[r];
        out_ptrs[r] = out[r];
    }
    cudaStream_t stream;
    cudaStreamCreate(&stream);

    /* AllReduce, sum, ring, out of place */
    ccl_comm_t comm = NULL;
    check(ccl_comm_create(&comm, P, in_ptrs) == CCL_OK, "ccl_comm_create");
    check(ccl_comm_set_outputs(comm, out_ptrs) == CCL_OK, "ccl_comm_set_outputs");
    check(ccl_allreduce(comm, CCL_SUM, CCL_F32, N, CCL_SCHED_RING, stream) == CCL_OK, "ccl_allreduce");
    cudaStreamSynchronize(stream);
    check(ccl_comm_check(comm) == CCL_OK, "ccl_comm_check");
    for (int r = 0; r < P; ++r) {
        cudaMemcpy(host, out[r], sizeof(float) * N, cudaMemcpyDeviceToHost);
        int ok = 1;
        for (int e = 0; e < N && ok; ++e) {
            float want = 0.0f;
            for (int k = 0; k < P; ++k) want += value(k, e);
            ok = host[e] == want;
        }
        check(ok, "AllReduce sum matches the plain sum on every rank");
    }
    /* ReduceScatter with n % p != 0 is refused */
    check(ccl_reduce_scatter(comm, CCL_SUM, CCL_F32, N - 1, CCL_SCHED_RING, stream) == CCL_ERR_INVALID_ARG,
          "ReduceScatter refuses n % p != 0");
    check(strlen(ccl_last_error()) > 0, "ccl_last_error names the failure");
    check(ccl_comm_destroy(comm) == CCL_OK, "ccl_comm_destroy");

    /* ReduceScatter (max, all-pairs) in place: rank r's chunk r of its own input */
    const int chunk = N / P;
    for (int r = 0; r < P; ++r) out_ptrs[r] = in[r] + (size_t)r * chunk;
    check(ccl_comm_create(&comm, P, in_ptrs) == CCL_OK, "ccl_comm_create (RS)");
    check(ccl_comm_set_outputs(comm, out_ptrs) == CCL_OK, "ccl_comm_set_outputs (RS)");
    check(ccl_reduce_scatter(comm, CCL_MAX, CCL_F32, N, CCL_SCHED_ALLPAIRS, stream) == CCL_OK, "ccl_reduce_scatter");
    check(ccl_comm_destroy(comm) == CCL_OK, "ccl_comm_destroy (RS)");
    /* AllGather in place: every rank receives every chunk */
    check(ccl_comm_create(&comm, P, in_ptrs) == CCL_OK, "ccl_comm_create (AG)");
    check(ccl_all_gather(comm, CCL_F32, N, stream) == CCL_OK, "ccl_all_gather");
    cudaStreamSynchronize(stream);
    check(ccl_comm_check(comm) == CCL_OK, "ccl_comm_check (AG)");
    for (int r = 0; r < P; ++r) {
        cudaMemcpy(host, in[r], sizeof(float) * N, cudaMemcpyDeviceToHost);
        int ok = 1;
        for (int e = 0; e < N && ok; ++e) {
            float want = value(0, e);
            for (int k = 1; k < P; ++k) want = value(k, e) > want ? value(k, e) : want;
            ok = host[e] == want;
        }
        check(ok, "ReduceScatter max then AllGather gives every rank the maximum");
    }
    check(ccl_comm_destroy(comm) == CCL_OK, "ccl_comm_destroy (AG)");

    /* a NULL rank pointer is refused */
    in_ptrs[2] = NULL;
    check(ccl_comm_create(&comm, P, in_ptrs) == CCL_ERR_INVALID_ARG && comm == NULL, "NULL rank pointer refused");

    for (int r = 0; r < P; ++r) {
        cudaFree(in[r]);
        cudaFree(out[r]);
    }
    cudaStreamDestroy(stream);
    free(host);
    printf("%s: %d failure(s)\n", fails ? "FAIL" : "ok", fails);
    return fails ? 1 : 0;
}
