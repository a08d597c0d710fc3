// Sinkhorn routing: per-expert column scalings that make the routing matrix doubly stochastic.
//
// "Megatron-LM 分布式训练（六）", section "Router": the Sinkhorn option normalises the routing matrix by
// Sinkhorn iterations into a doubly stochastic one, which balances the experts without an aux loss.
// On K[t,e] = exp(L[t,e] - max_e L[t,e]) and from r = 1, every iteration sets
//   c_e = (T / E) / sum_t K[t,e] r_t        (columns sum to T / E)
//   r_t = 1 / sum_e K[t,e] c_e              (rows sum to 1)
// The top-k of diag(r) K diag(c) in a row is the top-k of L + log c (a row scaling keeps a row's order), so
// the result is the selection-only bias log c for MOE_GATING_SOFTMAX_SELBIAS.
//
// One launch per iteration (sk_iter_kernel), each a programmatic dependent of the one before: every block first
// derives c from the previous iteration's per-block partial column sums (the same fixed-order reduction in every
// block, eight loads in flight per thread), then, one warp per token, r_t from c and its own partial column sums of
// K r. A last one-block kernel writes log c.
#include <math.h>
#include <algorithm>
#include "common.cuh"

namespace moe {

constexpr int kSkWarps = 8;
constexpr int kSkThreads = kSkWarps * 32;

static int sk_grid(int T) { return std::max(1, std::min(cdiv(T, 4 * kSkWarps), 2 * num_sms())); }

// c_e = (T / E) / sum_b partial[b][e], computed identically by every block: S slices of blocks per expert in
// parallel (S * E <= kSkThreads, S a power of two), then a tree over the slices; fixed order.
__device__ __forceinline__ void sk_scalings(const float* __restrict__ partial, int G, int T, int E, float* s_red,
                                           float* s_c) {
    int S = 1;
    while (S * 2 * E <= kSkThreads) S *= 2;
    for (int e0 = 0; e0 < E; e0 += kSkThreads / S) {   // experts in groups of kSkThreads / S
        const int ne = min(E - e0, kSkThreads / S);
        const int tid = threadIdx.x, sl = tid / ne, ex = tid - sl * ne;
        float v = 0.f;
        if (sl < S)
            for (int b0 = sl; b0 < G; b0 += 8 * S) {       // eight loads in flight, added in block order
                float w[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) w[u] = b0 + u * S < G ? partial[(size_t)(b0 + u * S) * E + e0 + ex] : 0.f;
#pragma unroll
                for (int u = 0; u < 8; ++u) v += w[u];
            }
        s_red[tid] = v;
        for (int st = S / 2; st > 0; st >>= 1) {
            __syncthreads();
            if (sl < st) s_red[tid] += s_red[tid + st * ne];
        }
        __syncthreads();
        if (tid < ne) s_c[e0 + tid] = ((float)T / (float)E) / s_red[tid];
        __syncthreads();
    }
}

// One Sinkhorn iteration: from the previous iteration's partial column sums (null on the first iteration,
// where r = 1) derive c, then for every token r_t = 1 / sum_e K[t,e] c_e and the block's partial column sums
// of K[t,e] r_t in a fixed order.
template <int NPL>
__global__ void __launch_bounds__(kSkThreads)
sk_iter_kernel(const float* __restrict__ logits, int T, int E, const float* __restrict__ partial_in,
               float* __restrict__ partial_out) {
    extern __shared__ float sm[];
    float* s_c = sm;                                     // [E]
    float* s_red = sm + E;                               // [kSkThreads]
    float* s_part = s_red + kSkThreads;                  // [kSkWarps][E]
    const int G = gridDim.x;
    pdl_wait();                              // a programmatic dependent of the previous iteration (or the router)
    pdl_trigger();                           // the next iteration may launch; it waits for this one to complete
    if (partial_in) sk_scalings(partial_in, G, T, E, s_red, s_c);
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float acc[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) acc[i] = 0.f;
    for (int t = blockIdx.x * kSkWarps + warp; t < T; t += G * kSkWarps) {
        float L[NPL];
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            const int e = lane + 32 * i;
            L[i] = e < E ? logits[(size_t)t * E + e] : -INFINITY;
            m = fmaxf(m, L[i]);
        }
        m = warp_max(m);
        float K[NPL];
        float rs = 0.f;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            const int e = lane + 32 * i;
            K[i] = e < E ? expf(L[i] - m) : 0.f;
            if (partial_in && e < E) rs += K[i] * s_c[e];
        }
        const float r = partial_in ? 1.f / warp_sum(rs) : 1.f;
#pragma unroll
        for (int i = 0; i < NPL; ++i) acc[i] += K[i] * r;
    }
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E) s_part[warp * E + e] = acc[i];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float sum = 0.f;
        for (int w = 0; w < kSkWarps; ++w) sum += s_part[w * E + e];
        partial_out[(size_t)blockIdx.x * E + e] = sum;
    }
}

// sel_bias[e] = log c_e from the last iteration's partial column sums (one block).
__global__ void __launch_bounds__(kSkThreads)
sk_bias_kernel(const float* __restrict__ partial, int G, int T, int E, float* __restrict__ sel_bias) {
    extern __shared__ float sm[];
    float* s_c = sm;
    float* s_red = sm + E;
    sk_scalings(partial, G, T, E, s_red, s_c);
    for (int e = threadIdx.x; e < E; e += blockDim.x) sel_bias[e] = logf(s_c[e]);
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_sinkhorn_workspace_size(int T, int E) {
    if (T <= 0 || E <= 0) return 0;
    return 2 * align_up((size_t)2 * num_sms() * E * sizeof(float), 256);   // ping-pong partial column sums
}

extern "C" int moe_sinkhorn_bias(const float* logits, int T, int E, int n_iter, float* sel_bias, void* ws,
                                 size_t ws_bytes, void* stream) {
    MOE_REQUIRE(T >= 1 && E >= 1 && E <= 1024 && n_iter >= 1 && n_iter <= 1000, MOE_ERR_INVALID_ARG,
                "moe_sinkhorn_bias: T=%d E=%d n_iter=%d", T, E, n_iter);
    MOE_REQUIRE(logits && sel_bias, MOE_ERR_INVALID_ARG, "moe_sinkhorn_bias: null pointer");
    const size_t need = moe_sinkhorn_workspace_size(T, E);
    MOE_REQUIRE(ws && ws_bytes >= need, MOE_ERR_WORKSPACE, "moe_sinkhorn_bias: workspace %zu < %zu", ws_bytes, need);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int G = sk_grid(T);
    float* part[2] = {static_cast<float*>(ws),
                      reinterpret_cast<float*>(static_cast<char*>(ws) + need / 2)};
    const size_t smem = (size_t)(E + kSkThreads + kSkWarps * E) * sizeof(float);
    const int npl = cdiv(E, 32);
    for (int it = 0; it < n_iter; ++it) {
        const float* pin = it == 0 ? nullptr : part[(it + 1) & 1];
        float* pout = part[it & 1];
#define MOE_SK_LAUNCH(N)                                                                                 \
        cudaFuncSetAttribute(sk_iter_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);    \
        if (cudaError_t le = launch_pdl(sk_iter_kernel<N>, dim3(G), dim3(kSkThreads), smem, s, logits, T, E, pin, pout)) \
            return set_error(MOE_ERR_CUDA, "sk_iter_kernel: %s", cudaGetErrorString(le));
        if (npl <= 1) { MOE_SK_LAUNCH(1) }
        else if (npl <= 2) { MOE_SK_LAUNCH(2) }
        else if (npl <= 4) { MOE_SK_LAUNCH(4) }
        else if (npl <= 8) { MOE_SK_LAUNCH(8) }
        else if (npl <= 16) { MOE_SK_LAUNCH(16) }
        else { MOE_SK_LAUNCH(32) }
#undef MOE_SK_LAUNCH
        if (int rc = check_launch("sk_iter_kernel")) return rc;
    }
    sk_bias_kernel<<<1, kSkThreads, (size_t)(E + kSkThreads) * sizeof(float), s>>>(part[(n_iter - 1) & 1], G, T, E,
                                                                                  sel_bias);
    return check_launch("sk_bias_kernel");
}
