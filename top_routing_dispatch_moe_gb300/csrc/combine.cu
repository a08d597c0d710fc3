// Combine: un-permute the expert outputs and sum the k of each token weighted by their gates.
//
// "v6 长序列和 MoE", table row "combine" (back to the original position, k outputs weighted by gate and
// summed); "专家并行" (formulaic), forward pass (the top-2 weighted merge on the source GPU);
// "Megatron-LM 分布式训练（六）", data flow ("+ shared_experts", every token, gate 1).
//
// A gather, not a scatter: one warp per token reads its (at most k) expert rows with 16-byte loads,
// accumulates in fp32 in ascending j (after the shared expert's output), and writes y once. No atomics,
// so the result is deterministic. HBM-bound: (kept assignments + T [+ T shared]) rows read, T rows written.
#include "common.cuh"

namespace moe {

template <typename T, int KMAX>
__global__ void __launch_bounds__(256)
combine_kernel(const T* __restrict__ eout, const int32_t* __restrict__ dest_row, const float* __restrict__ gates,
               const T* __restrict__ shared_out, int T_, int h, int k, T* __restrict__ y) {
    constexpr int V = Vec16<T>::N;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T_) return;
    const int myd = lane < k ? dest_row[(size_t)t * k + lane] : -1;
    const float myg = lane < k ? gates[(size_t)t * k + lane] : 0.f;
    int dj[KMAX];
    float gj[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        dj[j] = __shfl_sync(0xffffffffu, myd, j);
        gj[j] = __shfl_sync(0xffffffffu, myg, j);
    }
    constexpr int U = 2;                          // 16-byte column chunks per lane per pass
    for (int d0 = lane * V; d0 < h; d0 += U * 32 * V) {
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
        // issue every load of this pass before the first use: k rows x U chunks in flight per lane
#pragma unroll
        for (int j0 = 0; j0 < KMAX; j0 += 4) {
            if (j0 >= k) break;
            Vec16<T> v[4][U];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int j = j0 + jj, d = d0 + u * 32 * V;
                    if (j < KMAX && j < k && dj[j] >= 0 && d < h) v[jj][u] = ld16_stream(eout + (size_t)dj[j] * h + d);
                }
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
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
    const int grid = cdiv(T, 8);
    const __nv_bfloat16* eb = static_cast<const __nv_bfloat16*>(eout);
    const __nv_bfloat16* sb = static_cast<const __nv_bfloat16*>(shared_out);
    __nv_bfloat16* yb = static_cast<__nv_bfloat16*>(y);
    const float* ef = static_cast<const float*>(eout);
    const float* sf = static_cast<const float*>(shared_out);
    float* yf = static_cast<float*>(y);
#define MOE_COMBINE(KM)                                                                                         \
    if (dtype == MOE_BF16) combine_kernel<__nv_bfloat16, KM><<<grid, 256, 0, s>>>(eb, dest_row, gates, sb, T, h, k, yb); \
    else combine_kernel<float, KM><<<grid, 256, 0, s>>>(ef, dest_row, gates, sf, T, h, k, yf);
    if (k <= 2) { MOE_COMBINE(2) }
    else if (k <= 4) { MOE_COMBINE(4) }
    else if (k <= 8) { MOE_COMBINE(8) }
    else { MOE_COMBINE(16) }
#undef MOE_COMBINE
    return check_launch("combine_kernel");
}
