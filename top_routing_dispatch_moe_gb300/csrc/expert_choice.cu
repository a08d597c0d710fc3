// Expert-choice routing: every expert takes the C tokens it scores highest, then the same FFN machinery.
//
// "10.5 序列并行与专家并行", section 10.5.6 (load balancing), expert-choice bullet: the routing direction is
// reversed and each expert takes a fixed number of the highest-scoring tokens among all tokens, which
// balances the load by construction. Score = the per-token softmax over experts of the router logits; equal
// scores go to the lower token index; expert e's tokens fill rows e*C .. e*C + C - 1 in ascending token
// order; gate = the score.
//
// Kernels:
//   ec_prob_kernel     softmax over experts per token, written transposed (probT [E][T]) through a shared
//                      tile so that each expert's column is contiguous for the selection; slot[t][*] = -1;
//   ec_select_kernel   one block per expert: exact radix select (4 passes of 8 bits over the fp32 score
//                      bits, which order like the scores since scores are >= 0) finds the C-th largest
//                      score, then an ordered compaction in token order keeps every larger score and the
//                      first ties; writes tokens, gates and slot[t][e];
//   ec_gather_kernel   buf[e*C + j] = x[tokens[e][j]] (one warp per row) plus the tile schedule;
//   ec_combine_kernel  one warp per token: the experts that chose it, in ascending expert order (warp ballot),
//                      gate-weighted fp32 sum of their rows (+ shared expert), deterministic.
#include <math.h>
#include <algorithm>
#include "common.cuh"

namespace moe {

constexpr int kEcMaxE = 256;

__global__ void __launch_bounds__(256)
ec_prob_kernel(const float* __restrict__ logits, int T, int E, float* __restrict__ probT,
               int32_t* __restrict__ slot) {
    __shared__ float tile[32][kEcMaxE + 1];           // 32 tokens x E experts
    pdl_wait();                                       // a programmatic dependent: the router's logits from here on
    pdl_trigger();                                    // the selection may launch; it waits for this kernel
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t0 = blockIdx.x * 32;
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x)    // slot[t][e] = -1 (not chosen) for these tokens
        if (t0 + i / E < T) slot[(size_t)t0 * E + i] = -1;
    for (int tl = warp; tl < 32; tl += 8) {
        const int t = t0 + tl;
        if (t >= T) break;
        float m = -INFINITY;
        for (int e = lane; e < E; e += 32) m = fmaxf(m, logits[(size_t)t * E + e]);
        m = warp_max(m);
        float z = 0.f;
        for (int e = lane; e < E; e += 32) {
            const float v = expf(logits[(size_t)t * E + e] - m);
            tile[tl][e] = v;
            z += v;
        }
        z = warp_sum(z);
        const float inv = 1.f / z;
        for (int e = lane; e < E; e += 32) tile[tl][e] *= inv;
    }
    __syncthreads();
    for (int e = warp; e < E; e += 8) {
        const int t = t0 + lane;
        if (t < T) probT[(size_t)e * T + t] = tile[lane][e];
    }
}

__global__ void __launch_bounds__(1024)
ec_select_kernel(const float* __restrict__ probT, int T, int E, int C, int32_t* __restrict__ tokens,
                 float* __restrict__ gates, int32_t* __restrict__ slot) {
    __shared__ int s_hist[256];
    __shared__ int s_tmp[32];
    __shared__ uint32_t s_prefix;
    __shared__ int s_kth;
    pdl_wait();                                       // a programmatic dependent: probT and slot from here on
    const int e = blockIdx.x;
    const float* col = probT + (size_t)e * T;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) { s_prefix = 0u; s_kth = C; }
    // this thread's scores t = threadIdx.x + i blockDim.x, kept in registers across the passes when they fit
    constexpr int NV = 8;
    const bool cached = T <= NV * (int)blockDim.x;
    uint32_t kc[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int t = threadIdx.x + i * (int)blockDim.x;
        kc[i] = cached && t < T ? __float_as_uint(col[t]) : 0u;
    }
    uint32_t mask = 0u;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += blockDim.x) s_hist[i] = 0;
        __syncthreads();
        const uint32_t prefix = s_prefix;
        if (cached) {
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int t = threadIdx.x + i * (int)blockDim.x;
                if (t < T && (kc[i] & mask) == prefix) atomicAdd(&s_hist[(kc[i] >> shift) & 255u], 1);
            }
        } else {
            for (int t = threadIdx.x; t < T; t += blockDim.x) {
                const uint32_t key = __float_as_uint(col[t]);
                if ((key & mask) == prefix) atomicAdd(&s_hist[(key >> shift) & 255u], 1);
            }
        }
        __syncthreads();
        if (warp == 0) {
            // lane l owns digits 255 - 8l - 7 .. 255 - 8l (highest digits in lane 0)
            int own = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) own += s_hist[255 - 8 * lane - q];
            int incl = own;                         // inclusive prefix over lanes = count of digits >= the lane's lowest
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            const int kth = s_kth;
            const unsigned hit = __ballot_sync(0xffffffffu, incl >= kth);
            const int L = __ffs(hit) - 1;              // first lane whose range reaches the kth largest
            if (lane == L) {
                int cum = incl - own;                  // keys in digits above this lane's range
                int d = 255 - 8 * lane;
                for (int q = 0; q < 8; ++q, --d) {
                    if (cum + s_hist[d] >= kth) break;
                    cum += s_hist[d];
                }
                s_prefix = prefix | ((uint32_t)d << shift);
                s_kth = kth - cum;
            }
        }
        mask |= 255u << shift;
        __syncthreads();
    }
    const uint32_t K = s_prefix;                       // the C-th largest score's bits
    const int take_eq = s_kth;                         // how many scores equal to K are kept (lowest tokens)
    __shared__ int s_tot[2];
    int eq_run = 0, sel_run = 0;
    for (int base = 0; base < T; base += blockDim.x) {
        const int t = base + threadIdx.x;
        float p = 0.f;
        uint32_t key = 0u;
        if (t < T) { p = col[t]; key = __float_as_uint(p); }
        const int is_eq = (t < T && key == K) ? 1 : 0;
        const int eq_incl = block_inclusive_scan(is_eq, s_tmp);
        const int eq_rank = eq_run + eq_incl - is_eq;
        const int sel = (t < T && (key > K || (is_eq && eq_rank < take_eq))) ? 1 : 0;
        const int sel_incl = block_inclusive_scan(sel, s_tmp);
        const int pos = sel_run + sel_incl - 1;
        if (sel && pos < C) {                        // exactly C are selected; the bound keeps writes in range
            tokens[(size_t)e * C + pos] = t;
            gates[(size_t)e * C + pos] = p;
            slot[(size_t)t * E + e] = pos;
        }
        if (threadIdx.x == blockDim.x - 1) { s_tot[0] = eq_incl; s_tot[1] = sel_incl; }
        __syncthreads();
        eq_run += s_tot[0];
        sel_run += s_tot[1];
        __syncthreads();
    }
}

// buf[e*C + j] = x[tokens[e][j]]: one warp per row, 16-byte vectors.
template <typename T>
__global__ void __launch_bounds__(256)
ec_gather_kernel(const T* __restrict__ x, const int32_t* __restrict__ tokens, int T_, int rows, int h,
                 T* __restrict__ buf) {
    constexpr int V = Vec16<T>::N;
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (r >= rows) return;
    const int t = min(max(tokens[r], 0), T_ - 1);    // token ids come from the selection: always in range
    const T* src = x + (size_t)t * h;
    T* dst = buf + (size_t)r * h;
    constexpr int U = 4;
    for (int d0 = lane * V; d0 < h; d0 += U * 32 * V) {
        Vec16<T> v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (d0 + u * 32 * V < h) v[u] = ld16(src + d0 + u * 32 * V);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (d0 + u * 32 * V < h) st16(dst + d0 + u * 32 * V, v[u]);
    }
}

// Tile schedule of E groups of exactly C rows (group e at rows e*C).
__global__ void ec_sched_kernel(int E, int C, int32_t* sched) {
    const int tpe = (C + MOE_TILE_M - 1) / MOE_TILE_M;
    if (blockIdx.x == 0 && threadIdx.x == 0) { sched[0] = E * tpe; sched[1] = E; }
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e <= E; e += gridDim.x * blockDim.x)
        sched[kSchedHeader + e] = e * tpe;
    int4* tiles = reinterpret_cast<int4*>(sched + sched_tiles_offset(E));
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < E * tpe; i += gridDim.x * blockDim.x) {
        const int e = i / tpe, m = i - e * tpe;
        const int rb = e * C + m * MOE_TILE_M;
        tiles[i] = make_int4(e, rb, min(rb + MOE_TILE_M, (e + 1) * C), 0);
    }
}

// y[t] = shared_out[t] + sum over experts e that chose t (ascending e) of gate * eout[e*C + slot[t][e]].
template <typename T>
__global__ void __launch_bounds__(256)
ec_combine_kernel(const T* __restrict__ eout, const int32_t* __restrict__ slot, const float* __restrict__ gates,
                  const T* __restrict__ shared_out, int T_, int h, int E, int C, T* __restrict__ y) {
    constexpr int V = Vec16<T>::N;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T_) return;
    // the experts that chose t, 32 per ballot group, found once per token
    constexpr int G = kEcMaxE / 32;
    const int ngroups = (E + 31) / 32;
    int jl[G];
    float gl[G];
    unsigned ml[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const int e_l = 32 * g + lane;
        jl[g] = (g < ngroups && e_l < E) ? slot[(size_t)t * E + e_l] : -1;
        gl[g] = jl[g] >= 0 ? gates[(size_t)e_l * C + jl[g]] : 0.f;
        ml[g] = __ballot_sync(0xffffffffu, jl[g] >= 0);
    }
    // (row, gate) of the first kSel experts that chose t, ascending expert order, held by every lane
    constexpr int kSel = 16;
    int srow[kSel];
    float sg[kSel];
    int nsel = 0;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        unsigned m = ml[g];
        while (m) {
            const int src = __ffs(m) - 1;
            m &= m - 1;
            const int jj = __shfl_sync(0xffffffffu, jl[g], src);
            const float gg = __shfl_sync(0xffffffffu, gl[g], src);
            if (nsel < kSel) {
#pragma unroll
                for (int q = 0; q < kSel; ++q)
                    if (q == nsel) { srow[q] = (32 * g + src) * C + jj; sg[q] = gg; }
            }
            ++nsel;
        }
    }
    constexpr int U = 2;                            // column chunks per pass
    for (int d0b = 0; d0b < h; d0b += U * 32 * V) {  // warp-uniform trip count: shuffles below use all lanes
        float acc[U][V];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int d0 = d0b + u * 32 * V + lane * V;
            if (shared_out && d0 < h) {
                Vec16<T> sv = ld16_stream(shared_out + (size_t)t * h + d0);
#pragma unroll
                for (int i = 0; i < V; ++i) acc[u][i] = sv.get(i);
            } else {
#pragma unroll
                for (int i = 0; i < V; ++i) acc[u][i] = 0.f;
            }
        }
        // up to kSel rows from registers, four rows x U chunks in flight, in ascending expert order
#pragma unroll
        for (int q0 = 0; q0 < kSel; q0 += 4) {
            if (q0 >= nsel) break;
            Vec16<T> v[4][U];
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int d0 = d0b + u * 32 * V + lane * V;
                    if (d0 < h && q0 + qq < nsel) v[qq][u] = ld16_stream(eout + (size_t)srow[q0 + qq] * h + d0);
                }
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int d0 = d0b + u * 32 * V + lane * V;
                    if (d0 < h && q0 + qq < nsel) {
#pragma unroll
                        for (int i = 0; i < V; ++i) acc[u][i] = fmaf(sg[q0 + qq], v[qq][u].get(i), acc[u][i]);
                    }
                }
        }
        if (nsel > kSel) {                          // rare: more than kSel experts chose t; the rest in order
            int seen = 0;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                unsigned m = ml[g];
                while (m) {
                    const int src = __ffs(m) - 1;
                    m &= m - 1;
                    const int jj = __shfl_sync(0xffffffffu, jl[g], src);
                    const float gg = __shfl_sync(0xffffffffu, gl[g], src);
                    if (seen++ >= kSel) {
#pragma unroll
                        for (int u = 0; u < U; ++u) {
                            const int d0 = d0b + u * 32 * V + lane * V;
                            if (d0 < h) {
                                Vec16<T> v = ld16_stream(eout + ((size_t)(32 * g + src) * C + jj) * h + d0);
#pragma unroll
                                for (int i = 0; i < V; ++i) acc[u][i] = fmaf(gg, v.get(i), acc[u][i]);
                            }
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int d0 = d0b + u * 32 * V + lane * V;
            if (d0 < h) {
                Vec16<T> o;
#pragma unroll
                for (int i = 0; i < V; ++i) o.set(i, acc[u][i]);
                st16(y + (size_t)t * h + d0, o);
            }
        }
    }
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_expert_choice_workspace_size(int T, int E) {
    if (T < 0 || E <= 0) return 0;
    return align_up((size_t)T * E * sizeof(float), 256);
}

extern "C" int moe_expert_choice_route(const float* logits, int T, int E, int C, int32_t* tokens, float* gates,
                                       int32_t* slot, void* ws, size_t ws_bytes, void* stream) {
    MOE_REQUIRE(T >= 1 && E >= 1 && E <= kEcMaxE && C >= 1 && C <= T, MOE_ERR_INVALID_ARG,
                "moe_expert_choice_route: T=%d E=%d C=%d (need 1 <= C <= T, E <= %d)", T, E, C, kEcMaxE);
    MOE_REQUIRE(logits && tokens && gates && slot, MOE_ERR_INVALID_ARG, "moe_expert_choice_route: null pointer");
    const size_t need = moe_expert_choice_workspace_size(T, E);
    MOE_REQUIRE(ws && ws_bytes >= need, MOE_ERR_WORKSPACE, "moe_expert_choice_route: workspace %zu < %zu", ws_bytes,
                need);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* probT = static_cast<float*>(ws);
    const cudaError_t lp = launch_pdl(ec_prob_kernel, dim3(cdiv(T, 32)), dim3(256), 0, s, logits, T, E, probT, slot);
    if (int rc = check_launch(lp, "ec_prob_kernel")) return rc;
    const cudaError_t ls = launch_pdl(ec_select_kernel, dim3(E), dim3(1024), 0, s, (const float*)probT, T, E, C, tokens,
                                      gates, slot);
    return check_launch(ls, "ec_select_kernel");
}

extern "C" int moe_expert_choice_dispatch(const void* x, const int32_t* tokens, int T, int h, int E, int C, int dtype,
                                          void* buf, int32_t* tile_sched, void* stream) {
    MOE_REQUIRE(dtype == MOE_F32 || dtype == MOE_BF16, MOE_ERR_UNSUPPORTED, "moe_expert_choice_dispatch: dtype %d",
                dtype);
    MOE_REQUIRE(T >= 1 && h > 0 && h % 8 == 0 && E >= 1 && E <= kEcMaxE && C >= 1 && C <= T, MOE_ERR_INVALID_ARG,
                "moe_expert_choice_dispatch: T=%d h=%d E=%d C=%d", T, h, E, C);
    MOE_REQUIRE(x && tokens && buf && tile_sched, MOE_ERR_INVALID_ARG, "moe_expert_choice_dispatch: null pointer");
    MOE_REQUIRE(aligned16(x) && aligned16(buf) && aligned16(tile_sched), MOE_ERR_INVALID_ARG,
                "moe_expert_choice_dispatch: x, buf and tile_sched must be 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int rows = E * C;
    if (dtype == MOE_BF16)
        ec_gather_kernel<__nv_bfloat16><<<cdiv(rows, 8), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x), tokens,
                                                                       T, rows, h, static_cast<__nv_bfloat16*>(buf));
    else
        ec_gather_kernel<float><<<cdiv(rows, 8), 256, 0, s>>>(static_cast<const float*>(x), tokens, T, rows, h,
                                                               static_cast<float*>(buf));
    if (int rc = check_launch("ec_gather_kernel")) return rc;
    ec_sched_kernel<<<std::max(1, std::min(cdiv(rows, 128 * 256), 64)), 256, 0, s>>>(E, C, tile_sched);
    return check_launch("ec_sched_kernel");
}

extern "C" int moe_expert_choice_combine(const void* eout, const int32_t* slot, const float* gates,
                                         const void* shared_out, int T, int h, int E, int C, int dtype, void* y,
                                         void* stream) {
    MOE_REQUIRE(dtype == MOE_F32 || dtype == MOE_BF16, MOE_ERR_UNSUPPORTED, "moe_expert_choice_combine: dtype %d",
                dtype);
    MOE_REQUIRE(T >= 1 && h > 0 && h % 8 == 0 && E >= 1 && E <= kEcMaxE && C >= 1 && C <= T, MOE_ERR_INVALID_ARG,
                "moe_expert_choice_combine: T=%d h=%d E=%d C=%d", T, h, E, C);
    MOE_REQUIRE(eout && slot && gates && y, MOE_ERR_INVALID_ARG, "moe_expert_choice_combine: null pointer");
    MOE_REQUIRE(aligned16(eout) && aligned16(shared_out) && aligned16(y), MOE_ERR_INVALID_ARG,
                "moe_expert_choice_combine: eout, shared_out and y must be 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == MOE_BF16)
        ec_combine_kernel<__nv_bfloat16><<<cdiv(T, 8), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(eout), slot,
            gates, static_cast<const __nv_bfloat16*>(shared_out), T, h, E, C, static_cast<__nv_bfloat16*>(y));
    else
        ec_combine_kernel<float><<<cdiv(T, 8), 256, 0, s>>>(static_cast<const float*>(eout), slot, gates,
            static_cast<const float*>(shared_out), T, h, E, C, static_cast<float*>(y));
    return check_launch("ec_combine_kernel");
}
