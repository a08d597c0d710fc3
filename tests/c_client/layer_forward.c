/* A C program that uses the library through include/moe.h alone: it reads a layer's sizes, bf16 inputs and weights
 * from a file, packs the weights with moe_pack_router_weight / moe_pack_expert_weights, runs the forward of every
 * batch with moe_layer_forward_host from page-locked host memory, and writes the outputs to a file.
 *
 * Input file: int32 T, h, E, k, F, gating, capacity, num_ranks, n_batches; float32 alpha; then bf16 (as uint16)
 * x [n_batches][T][h], w_r [h][E], w_gate [E][F][h], w_up [E][F][h], w_down [E][h][F].
 * Output file: bf16 y [n_batches][T][h].
 * Usage: layer_forward IN OUT. Exit status 0 on success; a failing call prints its message and exits 1. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <stdint.h>
#include <cuda_runtime.h>
#include "moe.h"

#define CK_CUDA(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { \
    fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_)); return 1; } } while (0)
#define CK_MOE(x) do { int r_ = (x); if (r_ != MOE_OK) { \
    fprintf(stderr, "%s: status %d: %s\n", #x, r_, moe_last_error_string()); return 1; } } while (0)

static int read_all(FILE* f, void* dst, size_t bytes) { return fread(dst, 1, bytes, f) == bytes ? 0 : 1; }

/* host bf16 array -> new device buffer */
static int upload(FILE* f, size_t n, void** dev) {
    uint16_t* h = (uint16_t*)malloc(n * 2);
    if (!h || read_all(f, h, n * 2)) { free(h); fprintf(stderr, "short input\n"); return 1; }
    if (cudaMalloc(dev, n * 2) != cudaSuccess || cudaMemcpy(*dev, h, n * 2, cudaMemcpyHostToDevice) != cudaSuccess) {
        free(h);
        fprintf(stderr, "device upload failed\n");
        return 1;
    }
    free(h);
    return 0;
}

int main(int argc, char** argv) {
    if (argc != 3) { fprintf(stderr, "usage: %s IN OUT\n", argv[0]); return 2; }
    FILE* in = fopen(argv[1], "rb");
    if (!in) { perror(argv[1]); return 1; }
    int32_t hdr[9];
    float alpha;
    if (read_all(in, hdr, sizeof(hdr)) || read_all(in, &alpha, sizeof(alpha))) { fprintf(stderr, "short header\n"); return 1; }
    const int T = hdr[0], h = hdr[1], E = hdr[2], k = hdr[3], F = hdr[4], gating = hdr[5], capacity = hdr[6];
    const int num_ranks = hdr[7], nb = hdr[8];
    const size_t xbytes = (size_t)T * h * 2;

    /* page-locked host batches */
    void** x_host = (void**)calloc((size_t)nb, sizeof(void*));
    void** y_host = (void**)calloc((size_t)nb, sizeof(void*));
    if (!x_host || !y_host) return 1;
    for (int i = 0; i < nb; ++i) {
        CK_CUDA(cudaMallocHost(&x_host[i], xbytes));
        CK_CUDA(cudaMallocHost(&y_host[i], xbytes));
        if (read_all(in, x_host[i], xbytes)) { fprintf(stderr, "short x\n"); return 1; }
    }
    void *w_r, *w_gate, *w_up, *w_down;
    if (upload(in, (size_t)h * E, &w_r) || upload(in, (size_t)E * F * h, &w_gate) ||
        upload(in, (size_t)E * F * h, &w_up) || upload(in, (size_t)E * h * F, &w_down))
        return 1;
    fclose(in);

    cudaStream_t s;
    CK_CUDA(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
    void *w_r_packed, *packed;
    CK_CUDA(cudaMalloc(&w_r_packed, moe_router_packed_bytes(h, E, MOE_BF16)));
    CK_CUDA(cudaMalloc(&packed, moe_packed_weights_bytes(E, h, F, MOE_BF16)));
    CK_MOE(moe_pack_router_weight(w_r, h, E, MOE_BF16, w_r_packed, s));
    CK_MOE(moe_pack_expert_weights(w_gate, w_up, w_down, E, h, F, MOE_BF16, packed, s));

    moe_layer_desc d;
    memset(&d, 0, sizeof(d));
    d.T = T; d.h = h; d.E = E; d.k = k; d.F = F;
    d.dtype = MOE_BF16;
    d.gating = gating;
    d.alpha = alpha;
    d.capacity = capacity;
    d.num_ranks = num_ranks;
    d.w_r_packed = w_r_packed;
    d.bias = NULL;
    d.packed_w = packed;
    d.packed_shared = NULL;
    d.routing = MOE_ROUTING_TOKEN;
    d.payload = MOE_PAYLOAD_DTYPE;
    const size_t ws_bytes = moe_layer_host_workspace_size(&d);
    void* ws;
    CK_CUDA(cudaMalloc(&ws, ws_bytes));
    CK_MOE(moe_layer_forward_host(&d, nb, (const void* const*)x_host, (void* const*)y_host, ws, ws_bytes, s));
    CK_MOE(moe_check_device_error(s));       /* synchronises s: every y_host[i] is written */

    FILE* out = fopen(argv[2], "wb");
    if (!out) { perror(argv[2]); return 1; }
    for (int i = 0; i < nb; ++i)
        if (fwrite(y_host[i], 1, xbytes, out) != xbytes) { fprintf(stderr, "short write\n"); return 1; }
    fclose(out);
    printf("layer_forward: %d batches of %d tokens, %zu workspace bytes, %llu library launches\n", nb, T, ws_bytes,
           (unsigned long long)moe_launch_count());
    return 0;
}
