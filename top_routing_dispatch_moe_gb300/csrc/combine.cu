// Combine: un-permute the expert outputs and sum the k of each token weighted by their gates.
//
// "v6 长序列和 MoE", table row "combine" (back to the original position, k outputs weighted by gate and
// summed); "专家并行" (formulaic), forward pass (the top-2 weighted merge on the source GPU);
// "Megatron-LM 分布式训练（六）", data flow ("+ shared_experts", every token, gate 1).
//
// A gather, not a scatter: warps read a token's (at most k) expert rows with 16-byte loads, accumulate in fp32 in
// ascending j (after the shared expert's output), and write y once. No atomics, so the result is deterministic.
// HBM-bound: (kept assignments + T [+ T shared]) rows read, T rows written.
//
// The work is cut into items of one token and 512 columns (bf16; 256 for fp32), and a grid of exactly the warps
// that are resident at once loops over them, so that no short second wave of latency-bound warps ends the kernel
// (with one warp per token, about a tenth of the DeepSeek-V3-shaped layer's tokens were left to such a wave).
#include <algorithm>
#include "common.cuh"

namespace moe {

// 16-byte chunks per lane in one item (4 for k <= 2 would hold no more bytes in flight per SM: its registers
// would halve the resident warps).
__host__ __device__ constexpr int combine_chunks(int) { return 2; }

template <typename T, int KMAX>
__global__ void __launch_bounds__(256)
combine_kernel(const T* __restrict__ eout, const int32_t* __restrict__ dest_row, const float* __restrict__ gates,
               const T* __restrict__ shared_out, int T_, int h, int k, T* __restrict__ y) {
    constexpr int V = Vec16<T>::N;
    constexpr int U = combine_chunks(KMAX);       // 16-byte column chunks per lane per item
    constexpr int COLS = U * 32 * V;              // columns per item
    const int lane = threadIdx.x & 31;
    const int per_tok = (h + COLS - 1) / COLS;
    const long long items = (long long)T_ * per_tok;
    const long long nw = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long it = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items; it += nw) {
        const int t = (int)(it / per_tok);
        const int d0 = (int)(it - (long long)t * per_tok) * COLS + lane * V;
        const int myd = lane < k ? __ldg(dest_row + (size_t)t * k + lane) : -1;
        const float myg = lane < k ? __ldg(gates + (size_t)t * k + lane) : 0.f;
        int dj[KMAX];
        float gj[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            dj[j] = __shfl_sync(0xffffffffu, myd, j);
            gj[j] = __shfl_sync(0xffffffffu, myg, j);
        }
        float acc[U][V];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int d = d0 + u * 32 * V;
            if (shared_out && d < h) {
                Vec16<T> s = ld16_stream(shared_out + (size_t)t * h + d);
#pragma unroll
                for (int i = 0; i < V; ++i) acc[u][i] = s.get(i);
            } else {
#pragma unroll
                for (int i = 0; i < V; ++i) acc[u][i] = 0.f;
            }
        }
        // every load of the item before the first use: up to 8 rows x U chunks in flight per lane
        constexpr int JB = KMAX < 8 ? KMAX : 8;
#pragma unroll
        for (int j0 = 0; j0 < KMAX; j0 += JB) {
            if (j0 >= k) break;
            Vec16<T> v[JB][U];
#pragma unroll
            for (int jj = 0; jj < JB; ++jj)
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int j = j0 + jj, d = d0 + u * 32 * V;
                    if (j < KMAX && j < k && dj[j] >= 0 && d < h) v[jj][u] = ld16_stream(eout + (size_t)dj[j] * h + d);
                }
#pragma unroll
            for (int jj = 0; jj < JB; ++jj)
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int j = j0 + jj, d = d0 + u * 32 * V;
                    if (j < KMAX && j < k && dj[j] >= 0 && d < h) {
#pragma unroll
                        for (int i = 0; i < V; ++i) acc[u][i] = fmaf(gj[j], v[jj][u].get(i), acc[u][i]);
                    }
                }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int d = d0 + u * 32 * V;
            if (d < h) {
                Vec16<T> o;
#pragma unroll
                for (int i = 0; i < V; ++i) o.set(i, acc[u][i]);
                st16(y + (size_t)t * h + d, o);
            }
        }
    }
}

// Warps resident at once for an instantiation (blocks per SM x SMs x 8), at most one per item.
template <typename T, int KM>
static int combine_grid(int T_, int h) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_kernel<T, KM>, 256, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    const int cols = combine_chunks(KM) * 32 * Vec16<T>::N;
    const long long items = (long long)T_ * ((h + cols - 1) / cols);
    return (int)std::max(1LL, std::min((long long)per_sm * num_sms(), (items + 7) / 8));
}

}  // namespace moe

using namespace moe;

extern "C" int moe_combine(const void* eout, const int32_t* dest_row, const float* gates, const void* shared_out,
                           int T, int h, int k, int dtype, void* y, void* stream) {
    MOE_REQUIRE(dtype == MOE_F32 || dtype == MOE_BF16, MOE_ERR_UNSUPPORTED, "moe_combine: dtype %d", dtype);
    MOE_REQUIRE(T >= 0 && h > 0 && h % 8 == 0 && k >= 1 && k <= 16, MOE_ERR_INVALID_ARG,
                "moe_combine: T=%d h=%d k=%d", T, h, k);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(eout && dest_row && gates && y, MOE_ERR_INVALID_ARG, "moe_combine: null pointer");
    MOE_REQUIRE(aligned16(eout) && aligned16(shared_out) && aligned16(y), MOE_ERR_INVALID_ARG,
                "moe_combine: eout, shared_out and y must be 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const __nv_bfloat16* eb = static_cast<const __nv_bfloat16*>(eout);
    const __nv_bfloat16* sb = static_cast<const __nv_bfloat16*>(shared_out);
    __nv_bfloat16* yb = static_cast<__nv_bfloat16*>(y);
    const float* ef = static_cast<const float*>(eout);
    const float* sf = static_cast<const float*>(shared_out);
    float* yf = static_cast<float*>(y);
#define MOE_COMBINE(KM)                                                                                         \
    if (dtype == MOE_BF16)                                                                                      \
        combine_kernel<__nv_bfloat16, KM><<<combine_grid<__nv_bfloat16, KM>(T, h), 256, 0, s>>>(eb, dest_row, gates, sb, \
                                                                                          T, h, k, yb);        \
    else combine_kernel<float, KM><<<combine_grid<float, KM>(T, h), 256, 0, s>>>(ef, dest_row, gates, sf, T, h, k, yf);
    if (k <= 2) { MOE_COMBINE(2) }
    else if (k <= 4) { MOE_COMBINE(4) }
    else if (k <= 8) { MOE_COMBINE(8) }
    else { MOE_COMBINE(16) }
#undef MOE_COMBINE
    return check_launch("combine_kernel");
}
