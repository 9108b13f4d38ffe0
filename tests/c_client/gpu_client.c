/* A plain C99 client that runs one forward and backward on the GPU through
 * the C ABI alone: it allocates device memory with the CUDA runtime's C API,
 * creates its own stream and workspace, and calls ctx_attn_fwd and
 * ctx_attn_bwd.  The test that builds it supplies the inputs and checks the
 * outputs.
 *
 * usage: gpu_client IN OUT B S Hq Hkv D P causal
 *   IN:  q, k, v, dout as raw bf16, each dense [B,S,H,D] (H = Hq, Hkv, Hkv, Hq)
 *   OUT: out (bf16 [B,S,Hq,D]), lse (fp32 [B,Hq,S]), dq, dk, dv (bf16)
 * Exit status 0 on success; a failing step prints its status and exits 1. */
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "ctx_attn.h"

#define CUDA_OK(call)                                                          \
    do {                                                                       \
        cudaError_t e_ = (call);                                               \
        if (e_ != cudaSuccess) {                                               \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));        \
            return 1;                                                          \
        }                                                                      \
    } while (0)
#define CTX_OK_(call)                                                          \
    do {                                                                       \
        int rc_ = (call);                                                      \
        if (rc_ != CTX_OK) {                                                   \
            fprintf(stderr, "%s: %s (%d)\n", #call, ctx_status_string(rc_), rc_); \
            return 1;                                                          \
        }                                                                      \
    } while (0)

static ctx_tensor_t dense(void* p, int64_t B, int64_t S, int64_t H, int64_t D) {
    ctx_tensor_t t = {p, B, S, H, D, 0, 0, 0}; /* zero strides: dense in the call's layout */
    return t;
}

int main(int argc, char** argv) {
    if (argc != 10) {
        fprintf(stderr, "usage: %s IN OUT B S Hq Hkv D P causal\n", argv[0]);
        return 2;
    }
    const int64_t B = atol(argv[3]), S = atol(argv[4]), Hq = atol(argv[5]), Hkv = atol(argv[6]),
                  D = atol(argv[7]);
    const int P = atoi(argv[8]), causal = atoi(argv[9]);
    const size_t nq = (size_t)(B * S * Hq * D), nk = (size_t)(B * S * Hkv * D), nl = (size_t)(B * Hq * S);
    const size_t counts[4] = {nq, nk, nk, nq};

    /* inputs from the file into one host block */
    unsigned short* h_in = malloc(2 * (2 * nq + 2 * nk));
    FILE* f = fopen(argv[1], "rb");
    if (!h_in || !f || fread(h_in, 2, 2 * nq + 2 * nk, f) != 2 * nq + 2 * nk) {
        fprintf(stderr, "cannot read %s\n", argv[1]);
        return 1;
    }
    fclose(f);

    void* d_in[4];
    size_t at = 0;
    for (int i = 0; i < 4; ++i) {
        CUDA_OK(cudaMalloc(&d_in[i], 2 * counts[i]));
        CUDA_OK(cudaMemcpy(d_in[i], h_in + at, 2 * counts[i], cudaMemcpyHostToDevice));
        at += counts[i];
    }
    void *d_out, *d_dq, *d_dk, *d_dv, *d_ws;
    float* d_lse;
    CUDA_OK(cudaMalloc(&d_out, 2 * nq));
    CUDA_OK(cudaMalloc((void**)&d_lse, 4 * nl));
    CUDA_OK(cudaMalloc(&d_dq, 2 * nq));
    CUDA_OK(cudaMalloc(&d_dk, 2 * nk));
    CUDA_OK(cudaMalloc(&d_dv, 2 * nk));
    const size_t ws_bytes = ctx_attn_workspace_size((int)B, (int)S, (int)Hq, (int)Hkv, (int)D, P, 0);
    if (ws_bytes == 0) {
        fprintf(stderr, "invalid sizes\n");
        return 1;
    }
    CUDA_OK(cudaMalloc(&d_ws, ws_bytes));
    cudaStream_t stream;
    CUDA_OK(cudaStreamCreate(&stream));

    ctx_tensor_t q = dense(d_in[0], B, S, Hq, D), k = dense(d_in[1], B, S, Hkv, D),
                 v = dense(d_in[2], B, S, Hkv, D), dout = dense(d_in[3], B, S, Hq, D);
    ctx_tensor_t out = dense(d_out, B, S, Hq, D), dq = dense(d_dq, B, S, Hq, D),
                 dk = dense(d_dk, B, S, Hkv, D), dv = dense(d_dv, B, S, Hkv, D);
    CTX_OK_(ctx_attn_fwd(&q, &k, &v, P, NULL, CTX_LAYOUT_BSHD, causal, 0.0f, &out, d_lse, NULL, 0,
                         CTX_FLAG_NONE, stream));
    CTX_OK_(ctx_attn_bwd(&q, &k, &v, &out, d_lse, &dout, P, NULL, CTX_LAYOUT_BSHD, causal, 0.0f, &dq,
                         &dk, &dv, d_ws, ws_bytes, stream));
    CTX_OK_(ctx_get_device_status(stream)); /* synchronises; CTX_OK unless a wait ran out */

    /* outputs to the file */
    f = fopen(argv[2], "wb");
    if (!f) return 1;
    void* h = malloc(4 * nl > 2 * nq ? 4 * nl : 2 * nq);
    if (!h) return 1;
    const void* srcs[5] = {d_out, d_lse, d_dq, d_dk, d_dv};
    const size_t bytes[5] = {2 * nq, 4 * nl, 2 * nq, 2 * nk, 2 * nk};
    for (int i = 0; i < 5; ++i) {
        CUDA_OK(cudaMemcpy(h, srcs[i], bytes[i], cudaMemcpyDeviceToHost));
        if (fwrite(h, 1, bytes[i], f) != bytes[i]) return 1;
    }
    fclose(f);
    free(h);
    free(h_in);
    for (int i = 0; i < 4; ++i) cudaFree(d_in[i]);
    cudaFree(d_out); cudaFree(d_lse); cudaFree(d_dq); cudaFree(d_dk); cudaFree(d_dv); cudaFree(d_ws);
    cudaStreamDestroy(stream);
    printf("gpu client ok\n");
    return 0;
}
