/*
 * The library called from plain C, with nothing but the CUDA runtime: the
 * fused cross-entropy and the softmax forward on inputs read from a file.
 *
 *   ce_from_c <in.bin> <out.bin>
 *
 * in.bin:  int64 M, int64 V, then M*V fp32 logits (row-major), M int64 targets.
 * out.bin: float loss, int32 status of the calls, int32 gbce_last_error, then
 *          M*V fp32 gradients (d loss / d logits) and M*V fp32 softmax outputs.
 * Exit status 0 when every call returned GBCE_OK and the files were handled.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "gbce.h"

static int fail(const char *what)
{
    fprintf(stderr, "ce_from_c: %s\n", what);
    return 1;
}

int main(int argc, char **argv)
{
    if (argc != 3)
        return fail("usage: ce_from_c <in.bin> <out.bin>");
    FILE *in = fopen(argv[1], "rb");
    if (!in)
        return fail("cannot open the input");
    int64_t M = 0, V = 0;
    if (fread(&M, 8, 1, in) != 1 || fread(&V, 8, 1, in) != 1 || M < 1 || V < 1)
        return fail("bad header");
    const size_t n = (size_t)M * (size_t)V;
    float *logits = malloc(n * sizeof(float));
    float *grad = malloc(n * sizeof(float));
    float *soft = malloc(n * sizeof(float));
    int64_t *targets = malloc((size_t)M * sizeof(int64_t));
    if (!logits || !grad || !soft || !targets)
        return fail("out of host memory");
    if (fread(logits, sizeof(float), n, in) != n ||
        fread(targets, sizeof(int64_t), (size_t)M, in) != (size_t)M)
        return fail("short input");
    fclose(in);

    float *d_logits = NULL, *d_soft = NULL, *d_loss = NULL;
    int64_t *d_targets = NULL;
    cudaStream_t stream;
    if (cudaStreamCreate(&stream) != cudaSuccess ||
        cudaMalloc((void **)&d_logits, n * sizeof(float)) != cudaSuccess ||
        cudaMalloc((void **)&d_soft, n * sizeof(float)) != cudaSuccess ||
        cudaMalloc((void **)&d_loss, sizeof(float)) != cudaSuccess ||
        cudaMalloc((void **)&d_targets, (size_t)M * sizeof(int64_t)) != cudaSuccess)
        return fail("device allocation failed");
    if (cudaMemcpy(d_logits, logits, n * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(d_targets, targets, (size_t)M * sizeof(int64_t), cudaMemcpyHostToDevice) !=
            cudaSuccess)
        return fail("copy to the device failed");

    gbce_stream_t s = (gbce_stream_t)stream;
    /* the softmax of the logits first (out of place), then the fused CE in place */
    int rc = softmax_fwd(d_logits, V, d_soft, V, M, V, GBCE_F32, s);
    if (rc == GBCE_OK)
        rc = ce_fwd_bwd(d_logits, V, d_targets, d_loss, M, V, -100, GBCE_F32, s);
    const int flags = gbce_last_error(s);
    if (rc != GBCE_OK)
        fprintf(stderr, "ce_from_c: %s\n", gbce_status_string(rc));

    float loss = 0.f;
    if (cudaMemcpy(&loss, d_loss, sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(grad, d_logits, n * sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(soft, d_soft, n * sizeof(float), cudaMemcpyDeviceToHost) != cudaSuccess)
        return fail("copy from the device failed");

    FILE *out = fopen(argv[2], "wb");
    if (!out)
        return fail("cannot open the output");
    const int32_t status[2] = {rc, flags};
    if (fwrite(&loss, sizeof(float), 1, out) != 1 || fwrite(status, 4, 2, out) != 2 ||
        fwrite(grad, sizeof(float), n, out) != n || fwrite(soft, sizeof(float), n, out) != n)
        return fail("short output");
    fclose(out);

    cudaFree(d_logits);
    cudaFree(d_soft);
    cudaFree(d_loss);
    cudaFree(d_targets);
    cudaStreamDestroy(stream);
    free(logits);
    free(grad);
    free(soft);
    free(targets);
    return (rc == GBCE_OK && flags == GBCE_OK) ? 0 : 2;
}
