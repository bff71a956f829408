/*
 * One GRPO loss step through the C ABI of libgrpo, from plain C (no Python,
 * no torch): device memory from cudaMalloc, inputs made on the host from a
 * small linear congruential generator and copied over, then
 * grpo_group_advantages, grpo_build_mask, grpo_loss_fwd and
 * grpo_loss_fwd_bwd on one stream.  Then the same batch as two data-parallel
 * shards of one prompt group each (grpo_shard_counts, the counts summed on the
 * host, grpo_loss_fwd_bwd_shard).  Prints "ok <loss> <checksum>" and exits 0
 * when every call returns 0, the device status words read 0, the losses of
 * the two entry points are equal bit for bit, every gradient is finite, the
 * shards' dH rows equal the batch's bit for bit, and their loss shares and dW
 * add up to the batch's.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "grpo.h"

static uint32_t lcg_state = 12345u;
static float next_uniform(void) { /* in [-1, 1) */
    lcg_state = lcg_state * 1664525u + 1013904223u;
    return (float)((lcg_state >> 8) & 0xFFFFFF) / 8388608.0f - 1.0f;
}

static uint16_t to_bf16(float x) { /* round to nearest even (finite x) */
    uint32_t u;
    memcpy(&u, &x, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float from_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float x;
    memcpy(&x, &u, 4);
    return x;
}

#define CK(call)                                                                      \
    do {                                                                              \
        int rc_ = (int)(call);                                                        \
        if (rc_ != 0) {                                                               \
            fprintf(stderr, "%s failed: %d (%s)\n", #call, rc_, grpo_status_string(rc_)); \
            return 1;                                                                 \
        }                                                                             \
    } while (0)

#define CUDA(call)                                                                    \
    do {                                                                              \
        if ((call) != cudaSuccess) {                                                  \
            fprintf(stderr, "%s failed\n", #call);                                    \
            return 1;                                                                 \
        }                                                                             \
    } while (0)

int main(void) {
    const int n_groups = 2, G = 4, L = 96, d = 192, V = 1500;
    const int N = n_groups * G * L, n_seq = n_groups * G;
    grpo_shape shape;
    grpo_shape_init(&shape, n_groups, G, L, d, V, GRPO_BF16);
    shape.chunk_rows = 256;   /* several backward chunks */

    uint16_t* h_pol = malloc((size_t)N * d * 2);
    uint16_t* h_ref = malloc((size_t)N * d * 2);
    uint16_t* W = malloc((size_t)V * d * 2);
    int32_t* tokens = malloc((size_t)N * 4);
    int32_t* lengths = malloc((size_t)n_seq * 4);
    float* rewards = malloc((size_t)n_seq * 4);
    uint16_t* dH_host = malloc((size_t)N * d * 2);
    float* dW_host = malloc((size_t)V * d * 4);
    for (int64_t i = 0; i < (int64_t)N * d; ++i) {
        const float h = next_uniform();
        h_pol[i] = to_bf16(h);
        h_ref[i] = to_bf16(h + 0.05f * next_uniform());
    }
    for (int64_t i = 0; i < (int64_t)V * d; ++i) W[i] = to_bf16(0.05f * next_uniform());
    for (int i = 0; i < N; ++i) tokens[i] = (int32_t)((lcg_state = lcg_state * 1664525u + 1013904223u) >> 8) % V;
    for (int i = 0; i < n_seq; ++i) {
        lengths[i] = 10 + (int32_t)(((lcg_state = lcg_state * 1664525u + 1013904223u) >> 8) % (uint32_t)(L - 10));
        rewards[i] = (float)(i % 2) + 0.1f * next_uniform();
    }

    void *d_hp, *d_hr, *d_W, *d_tok, *d_len, *d_rew, *d_adv, *d_mask, *d_ws, *d_loss, *d_loss2, *d_dH, *d_dW;
    void *d_fi, *d_status;
    const size_t ws_bytes = grpo_workspace_bytes(&shape);
    if (ws_bytes == 0) {
        fprintf(stderr, "invalid shape\n");
        return 1;
    }
    CUDA(cudaMalloc(&d_hp, (size_t)N * d * 2));
    CUDA(cudaMalloc(&d_hr, (size_t)N * d * 2));
    CUDA(cudaMalloc(&d_W, (size_t)V * d * 2));
    CUDA(cudaMalloc(&d_tok, (size_t)N * 4));
    CUDA(cudaMalloc(&d_len, (size_t)n_seq * 4));
    CUDA(cudaMalloc(&d_rew, (size_t)n_seq * 4));
    CUDA(cudaMalloc(&d_adv, (size_t)n_seq * 4));
    CUDA(cudaMalloc(&d_mask, (size_t)N));
    CUDA(cudaMalloc(&d_ws, ws_bytes));
    CUDA(cudaMalloc(&d_loss, 4));
    CUDA(cudaMalloc(&d_loss2, 4));
    CUDA(cudaMalloc(&d_dH, (size_t)N * d * 2));
    CUDA(cudaMalloc(&d_dW, (size_t)V * d * 4));
    CUDA(cudaMalloc(&d_fi, 4));
    CUDA(cudaMalloc(&d_status, 4));
    CUDA(cudaMemcpy(d_hp, h_pol, (size_t)N * d * 2, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_hr, h_ref, (size_t)N * d * 2, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_W, W, (size_t)V * d * 2, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_tok, tokens, (size_t)N * 4, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_len, lengths, (size_t)n_seq * 4, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_rew, rewards, (size_t)n_seq * 4, cudaMemcpyHostToDevice));

    cudaStream_t st;
    CUDA(cudaStreamCreate(&st));
    grpo_stream_t gs = (grpo_stream_t)st;
    CK(grpo_group_advantages(d_rew, n_groups, G, shape.eps, shape.std_unbiased, d_adv, gs));
    CK(grpo_build_mask(d_len, &shape, d_mask, gs));
    CK(grpo_loss_fwd(d_hp, d_hr, d_W, d_tok, d_mask, d_adv, &shape, d_ws, ws_bytes, d_loss, NULL, d_status, gs));
    int32_t status = -1;
    CUDA(cudaStreamSynchronize(st));
    CUDA(cudaMemcpy(&status, d_status, 4, cudaMemcpyDeviceToHost));
    if (status != 0) {
        fprintf(stderr, "forward device status %d (%s)\n", status, grpo_status_string(status));
        return 1;
    }
    CK(grpo_loss_fwd_bwd(d_hp, d_hr, d_W, d_tok, d_mask, d_adv, &shape, 1.0f, d_ws, ws_bytes, d_loss2, d_dH, d_dW,
                         d_fi, NULL, d_status, gs));
    CUDA(cudaStreamSynchronize(st));
    float loss = 0.f, loss2 = 0.f;
    int32_t fi = -1;
    CUDA(cudaMemcpy(&status, d_status, 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(&loss, d_loss, 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(&loss2, d_loss2, 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(&fi, d_fi, 4, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(dH_host, d_dH, (size_t)N * d * 2, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(dW_host, d_dW, (size_t)V * d * 4, cudaMemcpyDeviceToHost));
    if (status != 0 || fi != 0) {
        fprintf(stderr, "backward device status %d, found_inf %d\n", status, fi);
        return 1;
    }
    if (memcmp(&loss, &loss2, 4) != 0) {
        fprintf(stderr, "losses differ: %.9g vs %.9g\n", loss, loss2);
        return 1;
    }
    /* the batch as two shards of one prompt group each (rows [r*N/2, (r+1)*N/2)) */
    {
        grpo_shape sh;
        grpo_shape_init(&sh, 1, G, L, d, V, GRPO_BF16);
        sh.chunk_rows = 256;
        const int Ns = G * L;
        const size_t ws_s = grpo_workspace_bytes(&sh);
        void *s_ws, *s_cnt[2], *s_gcnt, *s_loss[2], *s_dH[2], *s_dW[2], *s_fi;
        CUDA(cudaMalloc(&s_ws, ws_s));
        CUDA(cudaMalloc(&s_gcnt, 8));
        CUDA(cudaMalloc(&s_fi, 4));
        int32_t cnt[2][2], total[2] = {0, 0};
        for (int r = 0; r < 2; ++r) {
            CUDA(cudaMalloc(&s_cnt[r], 8));
            CUDA(cudaMalloc(&s_loss[r], 4));
            CUDA(cudaMalloc(&s_dH[r], (size_t)Ns * d * 2));
            CUDA(cudaMalloc(&s_dW[r], (size_t)V * d * 4));
            CK(grpo_shard_counts((const uint8_t*)d_mask + (size_t)r * Ns, &sh, s_cnt[r], gs));
        }
        CUDA(cudaStreamSynchronize(st));
        for (int r = 0; r < 2; ++r) {
            CUDA(cudaMemcpy(cnt[r], s_cnt[r], 8, cudaMemcpyDeviceToHost));
            total[0] += cnt[r][0];
            total[1] += cnt[r][1];
        }
        CUDA(cudaMemcpy(s_gcnt, total, 8, cudaMemcpyHostToDevice));   /* the host does the "all-reduce" */
        float share[2];
        for (int r = 0; r < 2; ++r) {
            const size_t ro = (size_t)r * Ns;
            CK(grpo_loss_fwd_bwd_shard((const char*)d_hp + ro * d * 2, (const char*)d_hr + ro * d * 2, d_W,
                                       (const int32_t*)d_tok + ro, (const uint8_t*)d_mask + ro,
                                       (const float*)d_adv + (size_t)r * G, &sh, s_gcnt, 1.0f, s_ws, ws_s, s_loss[r],
                                       s_dH[r], s_dW[r], s_fi, NULL, d_status, gs));
            CUDA(cudaStreamSynchronize(st));
            CUDA(cudaMemcpy(&status, d_status, 4, cudaMemcpyDeviceToHost));
            CUDA(cudaMemcpy(&share[r], s_loss[r], 4, cudaMemcpyDeviceToHost));
            if (status != 0) {
                fprintf(stderr, "shard %d device status %d\n", r, status);
                return 1;
            }
        }
        if (fabs((double)share[0] + share[1] - loss2) > 1e-6 * fabs(loss2)) {
            fprintf(stderr, "shard losses %.9g + %.9g != %.9g\n", share[0], share[1], loss2);
            return 1;
        }
        uint16_t* sdH = malloc((size_t)Ns * d * 2);
        float* sdW0 = malloc((size_t)V * d * 4);
        float* sdW1 = malloc((size_t)V * d * 4);
        for (int r = 0; r < 2; ++r) {
            CUDA(cudaMemcpy(sdH, s_dH[r], (size_t)Ns * d * 2, cudaMemcpyDeviceToHost));
            if (memcmp(sdH, dH_host + (size_t)r * Ns * d, (size_t)Ns * d * 2) != 0) {
                fprintf(stderr, "shard %d dH rows differ from the batch's\n", r);
                return 1;
            }
        }
        CUDA(cudaMemcpy(sdW0, s_dW[0], (size_t)V * d * 4, cudaMemcpyDeviceToHost));
        CUDA(cudaMemcpy(sdW1, s_dW[1], (size_t)V * d * 4, cudaMemcpyDeviceToHost));
        double top = 0.0, worst = 0.0;
        for (int64_t i = 0; i < (int64_t)V * d; ++i) {
            top = fmax(top, fabs(dW_host[i]));
            worst = fmax(worst, fabs((double)sdW0[i] + sdW1[i] - dW_host[i]));
        }
        if (!(worst <= 1e-5 * top)) {
            fprintf(stderr, "shard dW sum differs by %.3g (max %.3g)\n", worst, top);
            return 1;
        }
        free(sdH);
        free(sdW0);
        free(sdW1);
        for (int r = 0; r < 2; ++r) {
            cudaFree(s_cnt[r]);
            cudaFree(s_loss[r]);
            cudaFree(s_dH[r]);
            cudaFree(s_dW[r]);
        }
        cudaFree(s_ws);
        cudaFree(s_gcnt);
        cudaFree(s_fi);
    }
    double checksum = 0.0;
    for (int64_t i = 0; i < (int64_t)N * d; ++i) {
        const float x = from_bf16(dH_host[i]);
        if (!isfinite(x)) return 1;
        checksum += fabs(x);
    }
    for (int64_t i = 0; i < (int64_t)V * d; ++i) {
        if (!isfinite(dW_host[i])) return 1;
        checksum += fabs(dW_host[i]);
    }
    if (!(checksum > 0.0)) return 1;
    printf("ok %.9g %.9g\n", loss, checksum);
    return 0;
}
