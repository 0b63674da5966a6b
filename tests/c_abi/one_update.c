/* one_update.c - a C99 program that drives the optimizer step through include/tl.h
 * with memory it allocates itself (cudaMalloc, one buffer per tensor), as a C caller
 * of the library would ("Mixed precision, loss scaling, gradient accumulation, and
 * activation checkpointing", section 4 "The interface": a logical update over
 * micro-batches with their valid-target counts).
 *
 *   one_update IN OUT
 *
 * IN (little-endian, written by the test): int64 ntensors, int64 numel[ntensors],
 * int64 k, int64 counts[k], int64 steps, float lr, beta1, beta2, eps, weight_decay,
 * max_norm; float master[P]; uint16 param[P] (bf16); then for every step and
 * micro-batch uint16 grads[P] (bf16), the tensors back to back in tensor order.
 * OUT: per step float norm, float coef, double sumsq, int64 t, int32 skipped,
 * int32 zero; then float master[P], m[P], v[P] and uint16 param[P].
 * Exit status 0 on success, 1 with a message on any failure. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "tl.h"

static void die(const char* what, int code) {
    fprintf(stderr, "one_update: %s failed (%d)\n", what, code);
    exit(1);
}

static void rd(void* p, size_t n, FILE* f) {
    if (n && fread(p, 1, n, f) != n) die("read", 0);
}

static void wr(const void* p, size_t n, FILE* f) {
    if (n && fwrite(p, 1, n, f) != n) die("write", 0);
}

#define CK(call) do { cudaError_t e_ = (call); if (e_ != cudaSuccess) die(#call, (int)e_); } while (0)
#define TL(call) do { int r_ = (call); if (r_ != TL_OK) die(#call, r_); } while (0)

int main(int argc, char** argv) {
    if (argc != 3) die("usage: one_update IN OUT", 0);
    FILE* in = fopen(argv[1], "rb");
    if (!in) die("open IN", 0);
    int64_t nt, k, steps;
    rd(&nt, 8, in);
    int64_t* numel = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nt > 0 ? nt : 1));
    rd(numel, sizeof(int64_t) * (size_t)nt, in);
    rd(&k, 8, in);
    int64_t* counts = (int64_t*)malloc(sizeof(int64_t) * (size_t)k);
    rd(counts, sizeof(int64_t) * (size_t)k, in);
    rd(&steps, 8, in);
    float h[6];
    rd(h, sizeof(h), in);
    tl_adamw_hp hp = {h[0], h[1], h[2], h[3], h[4]};
    const float max_norm = h[5];
    int64_t P = 0, N = 0;
    for (int64_t i = 0; i < nt; ++i) P += numel[i];
    for (int64_t i = 0; i < k; ++i) N += counts[i];
    float* hw = (float*)malloc(4 * (size_t)P);
    uint16_t* hpar = (uint16_t*)malloc(2 * (size_t)P);
    uint16_t* hg = (uint16_t*)malloc(2 * (size_t)P);
    rd(hw, 4 * (size_t)P, in);
    rd(hpar, 2 * (size_t)P, in);

    /* one device buffer per tensor and list */
    void** param = (void**)calloc((size_t)nt, sizeof(void*));
    float** master = (float**)calloc((size_t)nt, sizeof(float*));
    float** m = (float**)calloc((size_t)nt, sizeof(float*));
    float** v = (float**)calloc((size_t)nt, sizeof(float*));
    float** acc = (float**)calloc((size_t)nt, sizeof(float*));
    void** grads = (void**)calloc((size_t)(nt * k), sizeof(void*));
    int64_t off = 0;
    for (int64_t i = 0; i < nt; ++i) {
        const size_t n = (size_t)numel[i];
        CK(cudaMalloc(&param[i], 2 * n));
        CK(cudaMalloc((void**)&master[i], 4 * n));
        CK(cudaMalloc((void**)&m[i], 4 * n));
        CK(cudaMalloc((void**)&v[i], 4 * n));
        CK(cudaMalloc((void**)&acc[i], 4 * n));
        for (int64_t j = 0; j < k; ++j) CK(cudaMalloc(&grads[j * nt + i], 2 * n));
        CK(cudaMemcpy(master[i], hw + off, 4 * n, cudaMemcpyHostToDevice));
        CK(cudaMemcpy(param[i], hpar + off, 2 * n, cudaMemcpyHostToDevice));
        CK(cudaMemset(m[i], 0, 4 * n));
        CK(cudaMemset(v[i], 0, 4 * n));
        off += numel[i];
    }
    tl_config cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.param_dtype = TL_BF16;
    cfg.grad_dtype = TL_BF16;
    cfg.scaler_enabled = 0;
    cfg.init_scale = 1.0f;
    cfg.growth = 2.0f;
    cfg.backoff = 0.5f;
    cfg.interval = 2000;
    cfg.min_scale = 1.0f;
    cfg.max_scale = 1.0f;
    tl_ctx* ctx = NULL;
    TL(tl_create(&ctx, nt, numel, param, master, m, v, acc, &cfg, NULL));

    FILE* out = fopen(argv[2], "wb");
    if (!out) die("open OUT", 0);
    for (int64_t s = 0; s < steps; ++s) {
        for (int64_t j = 0; j < k; ++j) {
            rd(hg, 2 * (size_t)P, in);
            off = 0;
            for (int64_t i = 0; i < nt; ++i) {
                CK(cudaMemcpy(grads[j * nt + i], hg + off, 2 * (size_t)numel[i], cudaMemcpyHostToDevice));
                off += numel[i];
            }
        }
        /* the five calls of one logical update, all on the default stream */
        for (int64_t j = 0; j + 1 < k; ++j)
            TL(tl_accumulate(ctx, (const void* const*)(grads + j * nt), counts[j], N, j == 0 ? 1 : 0, NULL));
        TL(tl_unscale_check(ctx, (const void* const*)(grads + (k - 1) * nt), counts[k - 1], N, NULL));
        TL(tl_grad_norm(ctx, max_norm, NULL));
        TL(tl_clip_adamw_step(ctx, &hp, NULL));
        TL(tl_scaler_update(ctx, NULL));
        tl_status st;
        TL(tl_read_status(ctx, &st, NULL));
        const int32_t tail[2] = {st.skipped, 0};
        wr(&st.norm, 4, out);
        wr(&st.coef, 4, out);
        wr(&st.sumsq, 8, out);
        wr(&st.t, 8, out);
        wr(tail, 8, out);
    }
    float* const* lists[3] = {master, m, v};
    float* hf = (float*)malloc(4 * (size_t)P);
    for (int l = 0; l < 3; ++l) {
        off = 0;
        for (int64_t i = 0; i < nt; ++i) {
            CK(cudaMemcpy(hf + off, lists[l][i], 4 * (size_t)numel[i], cudaMemcpyDeviceToHost));
            off += numel[i];
        }
        wr(hf, 4 * (size_t)P, out);
    }
    off = 0;
    for (int64_t i = 0; i < nt; ++i) {
        CK(cudaMemcpy(hpar + off, param[i], 2 * (size_t)numel[i], cudaMemcpyDeviceToHost));
        off += numel[i];
    }
    wr(hpar, 2 * (size_t)P, out);
    fclose(out);
    fclose(in);
    TL(tl_destroy(ctx));
    for (int64_t i = 0; i < nt; ++i) {
        cudaFree(param[i]);
        cudaFree(master[i]);
        cudaFree(m[i]);
        cudaFree(v[i]);
        cudaFree(acc[i]);
        for (int64_t j = 0; j < k; ++j) cudaFree(grads[j * nt + i]);
    }
    free(hf); free(hw); free(hpar); free(hg); free(numel); free(counts);
    free(param); free(master); free(m); free(v); free(acc); free(grads);
    return 0;
}
