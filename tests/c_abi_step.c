/*
 * The C ABI from plain C: device memory from cudaMalloc, no Python, no
 * torch.  All ranks' view, 3 ranks, fp16 grads and bf16 params, loss scale
 * 256, three steps through zero_step with a second state set bound (one
 * pass each), a +inf in rank 2's grads at step 2 (skipped: the scale
 * halves, t does not advance).  Inputs are read from and results written to
 * the binary files named on the command line; the test compares them with
 * the oracle.
 *
 *   c_abi_step <in.bin> <out.bin>
 *   in.bin:  numel (int64), then master0 (numel f32), then 3 steps x 3 ranks
 *            of numel fp16 grads (uint16)
 *   out.bin: the 3 step verdicts (int32 skipped each), the current master,
 *            m, v (P f32 each) and the params (P uint16)
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "zero.h"

#define WORLD 3
#define STEPS 3

static int check(int rc, const char *what)
{
    if (rc < 0) {
        fprintf(stderr, "%s: %s (%s)\n", what, zero_strerror(rc), zero_last_error());
        exit(1);
    }
    return rc;
}

static void cuda(cudaError_t e, const char *what)
{
    if (e != cudaSuccess) {
        fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
        exit(1);
    }
}

int main(int argc, char **argv)
{
    if (argc != 3) {
        fprintf(stderr, "usage: %s in.bin out.bin\n", argv[0]);
        return 2;
    }
    FILE *fi = fopen(argv[1], "rb");
    if (!fi) return 2;
    int64_t numel = 0;
    if (fread(&numel, 8, 1, fi) != 1) return 2;

    zero_ctx *ctx = NULL;
    check(zero_init(&ctx, numel, WORLD, 2, ZERO_F16, ZERO_BF16, -1, NULL, 0), "zero_init");
    const int64_t P = zero_ctx_state_elems(ctx);

    float *h_master = (float *)calloc((size_t)P, 4);
    uint16_t *h_grads = (uint16_t *)malloc((size_t)numel * 2 * WORLD * STEPS);
    if (fread(h_master, 4, (size_t)numel, fi) != (size_t)numel) return 2;
    if (fread(h_grads, 2, (size_t)numel * WORLD * STEPS, fi) != (size_t)numel * WORLD * STEPS)
        return 2;
    fclose(fi);

    float *d_state[6];
    for (int i = 0; i < 6; ++i) {
        cuda(cudaMalloc((void **)&d_state[i], (size_t)P * 4), "cudaMalloc state");
        cuda(cudaMemset(d_state[i], 0, (size_t)P * 4), "cudaMemset state");
    }
    cuda(cudaMemcpy(d_state[0], h_master, (size_t)P * 4, cudaMemcpyHostToDevice), "copy master");
    uint16_t *d_params;
    cuda(cudaMalloc((void **)&d_params, (size_t)P * 2), "cudaMalloc params");
    cuda(cudaMemset(d_params, 0, (size_t)P * 2), "cudaMemset params");
    uint64_t *d_words;                       /* the flag word and the current-set word */
    cuda(cudaMalloc((void **)&d_words, 16), "cudaMalloc words");
    cuda(cudaMemset(d_words, 0, 16), "cudaMemset words");
    void *d_grads[WORLD];
    for (int k = 0; k < WORLD; ++k)
        cuda(cudaMalloc(&d_grads[k], (size_t)numel * 2), "cudaMalloc grads");

    check(zero_bind(ctx, d_state[0], d_state[1], d_state[2], d_params, NULL, d_words), "bind");
    check(zero_bind_shadow(ctx, d_state[3], d_state[4], d_state[5], d_words + 1), "shadow");

    float scale = 256.0f;
    int64_t t = 0, good = 0;
    int32_t skipped_at[STEPS];
    for (int s = 0; s < STEPS; ++s) {
        for (int k = 0; k < WORLD; ++k)
            cuda(cudaMemcpy(d_grads[k], h_grads + ((size_t)s * WORLD + k) * (size_t)numel,
                            (size_t)numel * 2, cudaMemcpyHostToDevice), "copy grads");
        check(zero_step(ctx, (const void *const *)d_grads, WORLD, 1e-3, 0.9, 0.999, 1e-8, t + 1,
                        scale, NULL), "zero_step");
        int32_t nonfinite = 0, skipped = 0;
        check(zero_step_status(ctx, &nonfinite, &skipped), "status");
        skipped_at[s] = skipped;
        if (!skipped) ++t;
        scale = zero_scale_update(scale, skipped, &good, 2000);
    }
    int32_t which = 0;
    check(zero_current_state(ctx, &which), "current state");

    float *h_out = (float *)malloc((size_t)P * 4);
    uint16_t *h_params = (uint16_t *)malloc((size_t)P * 2);
    FILE *fo = fopen(argv[2], "wb");
    if (!fo) return 2;
    fwrite(skipped_at, 4, STEPS, fo);
    for (int i = 0; i < 3; ++i) {
        cuda(cudaMemcpy(h_out, d_state[which ? 3 + i : i], (size_t)P * 4, cudaMemcpyDeviceToHost),
             "copy state");
        fwrite(h_out, 4, (size_t)P, fo);
    }
    cuda(cudaMemcpy(h_params, d_params, (size_t)P * 2, cudaMemcpyDeviceToHost), "copy params");
    fwrite(h_params, 2, (size_t)P, fo);
    fclose(fo);
    zero_destroy(ctx);
    printf("c_abi_step: %d steps, skipped %d %d %d, final scale %g\n", STEPS, skipped_at[0],
           skipped_at[1], skipped_at[2], (double)scale);
    return 0;
}
