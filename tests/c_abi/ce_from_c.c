/*
 * The library called from plain C, with nothing but the CUDA runtime: the
 * fused cross-entropy (mean, and with reduction none, per-row losses and a
 * per-row gradient scale), the softmax forward and backward (the latter with
 * a status word of its own), and the plan query, on inputs read from a file.
 *
 *   ce_from_c <in.bin> <out.bin>
 *
 * in.bin:  int64 M, int64 V, then M*V fp32 logits (row-major), M int64 targets,
 *          M*V fp32 upstream gradients dy, M fp32 gradient scales s_r.
 * out.bin: float loss, int32 status of the calls, int32 gbce_last_error,
 *          int32 status word of the softmax backward call (softmax_bwd_ex),
 *          M*V fp32 gradients of the mean loss, M*V fp32 softmax outputs y,
 *          M*V fp32 softmax backward outputs dx (of y and dy),
 *          M*V fp32 gradients with reduction none scaled by s_r, M fp32 row
 *          losses, int32 CTAs per row of the plan, 32 bytes of its kernel name.
 * Exit status 0 when every call returned GBCE_OK and the files were handled.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "gbce.h"

static int fail(const char *what)
{
    fprintf(stderr, "ce_from_c: %s\n", what);
    return 1;
}

static int to_device(void **dst, const void *src, size_t bytes)
{
    if (cudaMalloc(dst, bytes) != cudaSuccess)
        return 1;
    return src && cudaMemcpy(*dst, src, bytes, cudaMemcpyHostToDevice) != cudaSuccess;
}

static int to_host(void *dst, const void *src, size_t bytes)
{
    return cudaMemcpy(dst, src, bytes, cudaMemcpyDeviceToHost) != cudaSuccess;
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
    const size_t n = (size_t)M * (size_t)V, mb = (size_t)M;
    float *logits = malloc(n * 4), *dy = malloc(n * 4), *scale = malloc(mb * 4);
    float *out = malloc(n * 4), *row_loss = malloc(mb * 4);
    int64_t *targets = malloc(mb * 8);
    if (!logits || !dy || !scale || !out || !row_loss || !targets)
        return fail("out of host memory");
    if (fread(logits, 4, n, in) != n || fread(targets, 8, mb, in) != mb ||
        fread(dy, 4, n, in) != n || fread(scale, 4, mb, in) != mb)
        return fail("short input");
    fclose(in);

    void *d_logits, *d_logits2, *d_soft, *d_dy, *d_scale, *d_loss, *d_row_loss, *d_targets;
    cudaStream_t stream;
    if (cudaStreamCreate(&stream) != cudaSuccess || to_device(&d_logits, logits, n * 4) ||
        to_device(&d_logits2, logits, n * 4) || to_device(&d_soft, NULL, n * 4) ||
        to_device(&d_dy, dy, n * 4) || to_device(&d_scale, scale, mb * 4) ||
        to_device(&d_loss, NULL, 4) || to_device(&d_row_loss, NULL, mb * 4) ||
        to_device(&d_targets, targets, mb * 8))
        return fail("device allocation or copy failed");

    gbce_stream_t s = (gbce_stream_t)stream;
    /* the softmax of the logits (out of place), its backward in place over dy,
       the fused CE in place (mean), then with reduction none on a second copy */
    int rc = softmax_fwd(d_logits, V, d_soft, V, M, V, GBCE_F32, s);
    unsigned int *d_status = NULL, call_status = 0xffffffffu;
    if (cudaMalloc((void **)&d_status, sizeof(unsigned int)) != cudaSuccess ||
        cudaMemset(d_status, 0, sizeof(unsigned int)) != cudaSuccess)
        return fail("device allocation failed");
    if (rc == GBCE_OK)  /* with a status word of the call's own */
        rc = softmax_bwd_ex(d_soft, V, d_dy, V, d_dy, V, M, V, GBCE_F32, d_status, s);
    if (rc == GBCE_OK)
        rc = ce_fwd_bwd(d_logits, V, d_targets, d_loss, M, V, -100, GBCE_F32, s);
    if (rc == GBCE_OK)
        rc = ce_fwd_bwd_ex(d_logits2, V, d_targets, NULL, d_row_loss, d_scale, M, V, -100,
                           GBCE_F32, GBCE_NONE, s);
    const int flags = gbce_last_error(s);
    if (cudaMemcpy(&call_status, d_status, sizeof(unsigned int), cudaMemcpyDeviceToHost) !=
        cudaSuccess)
        return fail("copy from the device failed");
    cudaFree(d_status);
    if (rc != GBCE_OK)
        fprintf(stderr, "ce_from_c: %s\n", gbce_status_string(rc));
    int ctas = 0;
    char name[32] = {0};
    const char *plan = gbce_plan(0, M, V, GBCE_F32, 1, &ctas);
    if (!plan)
        return fail("the plan query failed");
    strncpy(name, plan, sizeof name - 1);

    float loss = 0.f;
    FILE *o = fopen(argv[2], "wb");
    if (!o)
        return fail("cannot open the output");
    const int32_t status[3] = {rc, flags, (int32_t)call_status};
    int bad = to_host(&loss, d_loss, 4) || fwrite(&loss, 4, 1, o) != 1 ||
              fwrite(status, 4, 3, o) != 3;
    const void *blocks[4] = {d_logits, d_soft, d_dy, d_logits2};
    for (int b = 0; b < 4 && !bad; ++b)
        bad = to_host(out, blocks[b], n * 4) || fwrite(out, 4, n, o) != n;
    if (!bad)
        bad = to_host(row_loss, d_row_loss, mb * 4) || fwrite(row_loss, 4, mb, o) != mb ||
              fwrite(&ctas, 4, 1, o) != 1 || fwrite(name, 1, sizeof name, o) != sizeof name;
    fclose(o);
    if (bad)
        return fail("copy from the device or output failed");

    void *bufs[8] = {d_logits, d_logits2, d_soft, d_dy, d_scale, d_loss, d_row_loss, d_targets};
    for (int b = 0; b < 8; ++b)
        cudaFree(bufs[b]);
    cudaStreamDestroy(stream);
    free(logits);
    free(dy);
    free(scale);
    free(out);
    free(row_loss);
    free(targets);
    return (rc == GBCE_OK && flags == GBCE_OK) ? 0 : 2;
}
