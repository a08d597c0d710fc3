// Router: gating GEMM, top-k, gates, counts and the Switch aux-loss terms.
//
// "Megatron-LM 分布式训练（六）", section "Router": logits = hidden_states @ W_router, then top-k with
// softmax / sigmoid weights. "v6 长序列和 MoE", table rows "router" / "top-k" and the "Load balancing
// loss" bullet: aux = alpha * E * sum_i f_i P_i; DeepSeek-V3's bias is a selection-only term.
//
// Two ways to the logits, one gating epilogue:
//   E <= 32: fused kernel, W_r^T staged in shared memory (the whole router weight is at most a few hundred KB
//            and is read from L2 once per block), x streamed with 16-byte loads; bf16 on mma.sync tensor-core
//            instructions (16 tokens per block), fp32 on the CUDA cores (two tokens per warp).
//   E  > 32: logits GEMM [T,h] x [h,E] into fp32, then the gating kernel reads them back (L2-resident).
// The gating epilogue keeps the E logits of a token spread over the 32 lanes of a warp (lane l holds
// experts l, l+32, ...), takes k warp-wide argmax rounds (ties -> lower index), and accumulates per-block
// partial sums of P and per-block counts; a one-block finalize kernel adds the partials in a fixed order,
// so every output is deterministic.
#include <math.h>
#include <algorithm>
#include "common.cuh"
#include "ffn.cuh"

namespace moe {

constexpr int kRouterWarps = 8;
constexpr int kRouterMaxBlocks = 1024;
constexpr int kMaxK = 16;

struct GateOut {
    int32_t* ids;
    float* gates;
    float* logits;      // may be null
    float* partial_P;   // [grid][E]
    int32_t* partial_C; // [grid][E]
    unsigned* ticket;   // the finalize's arrival counter, zeroed by the gating kernel's block 0
};

// Order-preserving 32-bit key of a selection score: a larger score gives a larger key (-0 and +0 the same);
// key 0 marks a taken or absent slot (no finite or infinite score maps to it).
__device__ __forceinline__ unsigned score_key(float v) {
    const unsigned u = __float_as_uint(v == 0.f ? 0.f : v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The bias enters the logits in the plain and renormalised softmax modes; it is a selection-only term in the
// sigmoid mode and in the softmax mode with selection bias.
__host__ __device__ inline bool bias_in_logits(int gating) {
    return gating == MOE_GATING_SOFTMAX || gating == MOE_GATING_SOFTMAX_RENORM;
}

// Max / sum over the SEG lanes of this lane's segment (SEG = 32: the warp; 16: its half), a fixed butterfly order.
// For E <= 16 the lanes 16-31 of a whole-warp gating hold zeros, so the half-warp sums are the same bits.
template <int SEG>
__device__ __forceinline__ float seg_max(float v) {
#pragma unroll
    for (int o = SEG / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
template <int SEG>
__device__ __forceinline__ float seg_sum(float v) {
#pragma unroll
    for (int o = SEG / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
template <int SEG>
__device__ __forceinline__ unsigned seg_umax(unsigned v) {
    if constexpr (SEG == 32) {
        return __reduce_max_sync(0xffffffffu, v);
    } else {
#pragma unroll
        for (int o = SEG / 2; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
        return v;
    }
}
template <int SEG>
__device__ __forceinline__ unsigned seg_umin(unsigned v) {
    if constexpr (SEG == 32) {
        return __reduce_min_sync(0xffffffffu, v);
    } else {
#pragma unroll
        for (int o = SEG / 2; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
        return v;
    }
}

// Gating of one token whose NPL-per-lane logits are in L (expert of slot i = sl + 32 i, sl the lane's index in its
// segment of SEG lanes; with SEG = 16 each half-warp gates its own token, NPL = 1 and E <= 16). Every lane of the
// warp must call it (the reductions are shuffles); a segment with valid = false writes and accumulates nothing.
// Accumulates the token's router probabilities into Pacc and its choices into the shared histogram.
template <int NPL, int SEG = 32>
__device__ __forceinline__ void gate_token(float (&L)[NPL], int t, int E, int k, int gating, const float* bias,
                                           const GateOut& o, float (&Pacc)[NPL], int* s_hist, bool valid = true) {
    static_assert(SEG == 32 || (SEG == 16 && NPL == 1), "half-warp gating holds one expert per lane");
    const int lane = threadIdx.x & 31;
    const int sl = lane & (SEG - 1), seg0 = lane - sl;
    float score[NPL], prob[NPL];
    bool live[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) live[i] = valid && (sl + 32 * i) < E;

    if (gating == MOE_GATING_SIGMOID_BIAS_RENORM) {
        float s_sum = 0.f;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            float s = live[i] ? 1.f / (1.f + expf(-L[i])) : 0.f;
            prob[i] = s;                                   // sigmoid value, normalised below
            score[i] = live[i] ? s + (bias ? bias[sl + 32 * i] : 0.f) : -INFINITY;
            s_sum += s;
        }
        s_sum = seg_sum<SEG>(s_sum);
        float inv = 1.f / s_sum;
        if (valid) {
#pragma unroll
            for (int i = 0; i < NPL; ++i) Pacc[i] += prob[i] * inv;
        }
    } else {
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < NPL; ++i) if (live[i]) m = fmaxf(m, L[i]);
        m = seg_max<SEG>(m);
        float z = 0.f;
        const bool selbias = gating == MOE_GATING_SOFTMAX_SELBIAS && bias;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            prob[i] = live[i] ? expf(L[i] - m) : 0.f;
            z += prob[i];
            score[i] = live[i] ? L[i] + (selbias ? bias[sl + 32 * i] : 0.f) : -INFINITY;
        }
        z = seg_sum<SEG>(z);
        float inv = 1.f / z;
#pragma unroll
        for (int i = 0; i < NPL; ++i) prob[i] *= inv;
        if (valid) {
#pragma unroll
            for (int i = 0; i < NPL; ++i) Pacc[i] += prob[i];
        }
    }

    // k rounds of warp argmax on the selection score, on order-preserving keys: a warp max reduction finds the
    // largest key, a warp min reduction the smallest expert index holding it (equal scores: smaller index). Each lane
    // keeps its own largest remaining key (the lowest slot holding it) and that expert's probability, so a round
    // rescans the slots of the one lane that gave up its expert only.
    unsigned key[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) key[i] = live[i] ? score_key(score[i]) : 0u;
    unsigned lmax = key[0];
    int lslot = 0;
    float lprob = prob[0];
#pragma unroll
    for (int i = 1; i < NPL; ++i)
        if (key[i] > lmax) { lmax = key[i]; lslot = i; lprob = prob[i]; }
    int my_id = 0;                         // lane sl keeps choice j = sl (for the writes below)
    float my_p = 0.f;
    float psum = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
        if (j < k) {
            const unsigned m = seg_umax<SEG>(lmax);
            int bi = (int)seg_umin<SEG>(lmax == m ? (unsigned)(sl + 32 * lslot) : 0xffffffffu);
            if (bi >= E) bi = E - 1;          // only reachable with NaN scores: keeps every index in bounds
            const int owner = seg0 + (bi & 31);
            const float pv = __shfl_sync(0xffffffffu, lprob, owner);
            if (lane == owner) {               // this lane's expert is taken: its next largest key
#pragma unroll
                for (int i = 0; i < NPL; ++i)
                    if (i == lslot) key[i] = 0u;
                lmax = key[0];
                lslot = 0;
                lprob = prob[0];
#pragma unroll
                for (int i = 1; i < NPL; ++i)
                    if (key[i] > lmax) { lmax = key[i]; lslot = i; lprob = prob[i]; }
            }
            if (sl == j) {
                my_id = bi;
                my_p = pv;
            }
            psum += pv;
        }
    }
    const float norm = (gating == MOE_GATING_SOFTMAX || gating == MOE_GATING_SOFTMAX_SELBIAS) ? 1.f : 1.f / psum;
    if (valid && sl < k) {                 // the k choices in one store per output (k <= 16 <= SEG)
        o.ids[(size_t)t * k + sl] = my_id;
        o.gates[(size_t)t * k + sl] = my_p * norm;
        atomicAdd(&s_hist[my_id], 1);
    }
}

// Per-block partial sums of P and counts (fixed order over the block's warps).
template <int NPL>
__device__ __forceinline__ void flush_partials(float (&Pacc)[NPL], int E, float* s_P, int* s_hist,
                                               const GateOut& o) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        int e = lane + 32 * i;
        if (e < E) s_P[warp * E + e] = Pacc[i];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float s = 0.f;
        for (int w = 0; w < kRouterWarps; ++w) s += s_P[w * E + e];
        o.partial_P[(size_t)blockIdx.x * E + e] = s;
        o.partial_C[(size_t)blockIdx.x * E + e] = s_hist[e];
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) *o.ticket = 0u;     // the finalize runs after this kernel
}

// 16 bytes of elements -> fp32 (bf16: the value's bits are the high half of an fp32 word).
__device__ __forceinline__ void unpack16(const Vec16<float>& v, float (&f)[4]) {
    f[0] = v.v.x; f[1] = v.v.y; f[2] = v.v.z; f[3] = v.v.w;
}
__device__ __forceinline__ void unpack16(const Vec16<__nv_bfloat16>& v, float (&f)[8]) {
    const uint32_t w[4] = {v.v.x, v.v.y, v.v.z, v.v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Packed fp32 pairs: element 2i in the low word, 2i + 1 in the high word.
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(c) : "l"(a), "l"(b));
    return c;
}
__device__ __forceinline__ float pair_sum(unsigned long long p) {
    return __uint_as_float((uint32_t)p) + __uint_as_float((uint32_t)(p >> 32));
}
__device__ __forceinline__ void unpack_pairs(const Vec16<float>& v, unsigned long long (&p)[2]) {
    p[0] = ((unsigned long long)__float_as_uint(v.v.y) << 32) | __float_as_uint(v.v.x);
    p[1] = ((unsigned long long)__float_as_uint(v.v.w) << 32) | __float_as_uint(v.v.z);
}
__device__ __forceinline__ void unpack_pairs(const Vec16<__nv_bfloat16>& v, unsigned long long (&p)[4]) {
    const uint32_t w[4] = {v.v.x, v.v.y, v.v.z, v.v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        p[i] = ((unsigned long long)(w[i] & 0xffff0000u) << 32) | (unsigned long long)(w[i] << 16);
}

// ---------------------------------------------------------------------------------------------------
// E <= 32: fused logits + gating, W_r^T in shared memory (transposed while it is staged)
// ---------------------------------------------------------------------------------------------------
// W_r [h][E] (global) -> wT [E][h] (shared), so that a lane's 16-byte x chunk meets each expert's weights
// as one conflict-free 16-byte shared load. When an h-row of W_r is a whole number of 16-byte vectors, every
// thread keeps 8 vector loads in flight and scatters their elements; otherwise element by element.
template <typename T>
__device__ __forceinline__ void stage_router_weight(const T* __restrict__ w_r, int h, int E, T* __restrict__ wT) {
    constexpr int V = Vec16<T>::N;
    if ((E * (int)sizeof(T)) % 16 == 0) {
        const int RV = E / V;                                  // 16-byte vectors per h-row
        const int nvec = h * RV;
        constexpr int B = 4;
        for (int v0 = threadIdx.x; v0 < nvec; v0 += B * blockDim.x) {
            Vec16<T> r[B];
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int v = v0 + b * blockDim.x;
                if (v < nvec) r[b] = ld16(w_r + (size_t)v * V);
            }
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int v = v0 + b * blockDim.x;
                if (v < nvec) {
                    const int d = v / RV, e0 = (v - d * RV) * V;
                    const T* el = reinterpret_cast<const T*>(&r[b].v);
#pragma unroll
                    for (int i = 0; i < V; ++i) wT[(size_t)(e0 + i) * h + d] = el[i];
                }
            }
        }
    } else {
        for (int f = threadIdx.x; f < E * h; f += blockDim.x) {
            const int d = f / E;
            wT[(size_t)(f - d * E) * h + d] = w_r[f];
        }
    }
}

// U = 16-byte x chunks per token and lane in flight: 4 while the accumulators are small (E <= 8), else 2. Two
// blocks per SM for EMAX = 8; with 16 or 32 experts the two tokens' packed accumulators alone take 64 or 128
// registers, so one block per SM keeps them out of local memory.
template <typename T, int EMAX, int U>
__global__ void __launch_bounds__(kRouterWarps * 32, EMAX <= 8 ? 2 : 1)
router_small_kernel(const T* __restrict__ x, const T* __restrict__ w_r, const float* __restrict__ bias, int T_,
                    int h, int E, int k, int gating, GateOut o) {
    pdl_trigger();                            // the finalize may launch now (it waits for this kernel's partials)
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* wT = reinterpret_cast<T*>(smem_raw);                                     // [E][h]
    float* s_P = reinterpret_cast<float*>(smem_raw + (((size_t)E * h * sizeof(T) + 15) & ~(size_t)15));
    int* s_hist = reinterpret_cast<int*>(s_P + kRouterWarps * E);

    constexpr int V = Vec16<T>::N;
    stage_router_weight(w_r, h, E, wT);
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
    __syncthreads();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float Pacc[1] = {0.f};
    const bool use_bias_in_logits = bias && bias_in_logits(gating);
    const int nwarps = gridDim.x * kRouterWarps;
    // Two tokens per warp: every unpacked weight pair feeds both; accumulation in packed fp32 pairs
    // (even / odd element partial sums, added at the end).
    for (int t0 = 2 * (blockIdx.x * kRouterWarps + warp); t0 < T_; t0 += 2 * nwarps) {
        const bool has1 = t0 + 1 < T_;
        unsigned long long acc0[EMAX], acc1[EMAX];
#pragma unroll
        for (int e = 0; e < EMAX; ++e) { acc0[e] = 0ull; acc1[e] = 0ull; }
        const T* x0 = x + (size_t)t0 * h;
        const T* x1 = x + (size_t)(has1 ? t0 + 1 : t0) * h;
        for (int d0 = lane * V; d0 < h; d0 += U * 32 * V) {
            Vec16<T> va[U], vb[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int d = d0 + u * 32 * V;
                if (d < h) { va[u] = ld16_stream(x0 + d); vb[u] = ld16_stream(x1 + d); }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int d = d0 + u * 32 * V;
                if (d < h) {
                    unsigned long long xa[V / 2], xb[V / 2];
                    unpack_pairs(va[u], xa);
                    unpack_pairs(vb[u], xb);
#pragma unroll
                    for (int e = 0; e < EMAX; ++e) {
                        if (e < E) {
                            unsigned long long wp[V / 2];
                            unpack_pairs(*reinterpret_cast<const Vec16<T>*>(wT + (size_t)e * h + d), wp);
#pragma unroll
                            for (int i = 0; i < V / 2; ++i) {
                                acc0[e] = fma2(xa[i], wp[i], acc0[e]);
                                acc1[e] = fma2(xb[i], wp[i], acc1[e]);
                            }
                        }
                    }
                }
            }
        }
        float L0[1] = {-INFINITY}, L1[1] = {-INFINITY};
#pragma unroll
        for (int e = 0; e < EMAX; ++e) {
            if (e < E) {
                const float a = warp_sum(pair_sum(acc0[e])), b = warp_sum(pair_sum(acc1[e]));
                if (lane == e) { L0[0] = a; L1[0] = b; }
            }
        }
        if (lane < E && use_bias_in_logits) { L0[0] += bias[lane]; L1[0] += bias[lane]; }
        if (lane < E && o.logits) {
            o.logits[(size_t)t0 * E + lane] = L0[0];
            if (has1) o.logits[(size_t)(t0 + 1) * E + lane] = L1[0];
        }
        gate_token<1>(L0, t0, E, k, gating, bias, o, Pacc, s_hist);
        if (has1) gate_token<1>(L1, t0 + 1, E, k, gating, bias, o, Pacc, s_hist);
    }
    __syncthreads();
    flush_partials<1>(Pacc, E, s_P, s_hist, o);
}

// ---------------------------------------------------------------------------------------------------
// E <= 32, bf16: logits on mma.sync m16n8k16 (bf16 in, fp32 accumulate), fused with the gating
// ---------------------------------------------------------------------------------------------------
// The logits GEMM is HBM-bound (x is read once, 2 h E flop per 2 h bytes), so what matters is the number of
// instructions per byte: one mma.sync does 16 tokens x 8 experts x 16 of h. A block takes 16 tokens; its 8
// warps split h into contiguous slices of 32-column chunks, each warp accumulating its slice's partial
// logits, which are then added in a fixed warp order (deterministic).
// Within a 32-column chunk, lane (g = lane / 4, t = lane % 4) loads 16 contiguous bytes (columns 8t .. 8t+7)
// of token rows g and g + 8 and of W_r^T row g. The two k16 steps of the chunk take those columns in the order
// {8t, 8t+1 | 8t+2, 8t+3} and {8t+4, 8t+5 | 8t+6, 8t+7} as the fragment's {2t, 2t+1 | 2t+8, 2t+9}: A and B use
// the same permutation of k, so every column of the chunk is summed exactly once.
constexpr int kMmaTokens = 16;

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// W_r^T row stride in shared memory (elements): h rounded up to whole 32-column chunks, plus 64 bytes so that
// the 8 lanes of a 16-byte load phase (two W rows, four column groups) hit distinct banks.
__host__ __device__ inline int mma_wt_stride(int h) { return ((h + 31) / 32 * 32 * 2 + 127) / 128 * 64 + 32; }

// Token row t of x [T][h] into L2 (nothing for t outside [0, T)); the row is a multiple of 16 bytes.
__device__ __forceinline__ void prefetch_row_l2(const __nv_bfloat16* x, int T_, int h, int t) {
    if (t >= 0 && t < T_)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                     ::"l"(reinterpret_cast<uint64_t>(x + (size_t)t * h)), "r"((unsigned)(h * 2)) : "memory");
}

// The packed router weight's rows reach shared memory through the bulk-copy unit, completing on an mbarrier
// (addresses and sizes multiples of 16 bytes). A wait polls at most `limit` times, 32 ns apart.
__device__ __forceinline__ void bulk_row_to_shared(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, long long limit) {
    for (long long i = 0; i < limit; ++i) {
        uint32_t ok;
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
        if (ok) return true;
        __nanosleep(32);
    }
    return false;
}
constexpr long long kWeightDrainLimit = 1LL << 24;

template <int NB, int U>   // NB blocks of 8 experts (E <= 8 NB); 2 x U chunks of 32 columns in flight per warp
__global__ void __launch_bounds__(kRouterWarps * 32, 2)
router_mma_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ w_r,
                  const __nv_bfloat16* __restrict__ w_rT, const float* __restrict__ bias, int T_, int h, int E, int k,
                  int gating, GateOut o, unsigned* err, long long wait_limit) {
    pdl_trigger();                            // the finalize may launch now (it waits for this kernel's partials)
    // (an L2 prefetch of the block's first 16 token rows here was measured: the router weight's staging then
    // queued behind it, and the x loads ended no sooner)
    constexpr int EP = 8 * NB;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int stride = mma_wt_stride(h);
    __nv_bfloat16* wT = reinterpret_cast<__nv_bfloat16*>(smem_raw);                          // [EP][stride]
    float* red = reinterpret_cast<float*>(smem_raw + (size_t)EP * stride * 2);                // [warps][16][EP]
    float* s_P = red + kRouterWarps * kMmaTokens * EP;
    int* s_hist = reinterpret_cast<int*>(s_P + kRouterWarps * E);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int nchunks = (h + 31) / 32, cpw = (nchunks + kRouterWarps - 1) / kRouterWarps;
    const int c_begin = min(nchunks, warp * cpw), c_end = min(nchunks, c_begin + cpw);

    // This warp's slice of W_r [h][E] (rows d0 .. d1, one contiguous run of memory), transposed; rows e >= E
    // and columns d1 .. dz past h are zero. With E = EP every 16-byte vector lies in one W_r row, and each lane
    // keeps 8 vector loads in flight.
    const int d0 = c_begin * 32, d1 = min(h, c_end * 32), dz = c_end * 32;
    const __nv_bfloat16 zero = __float2bfloat16_rn(0.f);
    // (packed weight) the mbarrier on which its rows land, after the histogram
    const uint32_t wbar = (uint32_t)__cvta_generic_to_shared(s_hist + ((E + 1) & ~1));
    if (w_rT) {
        // the packed transpose W_r^T [E][h]: once every thread has its first x loads in flight, thread 0 has the
        // bulk-copy unit bring each expert's row into its padded shared row (below); rows e >= E are zero
        if (threadIdx.x == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(wbar) : "memory");
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        if (warp == 0)
            for (int f = lane; f < (EP - E) * h; f += 32) wT[(size_t)(E + f / h) * stride + f % h] = zero;
    } else if (E == EP) {
        const int nvec = (d1 - d0) * EP / 8;
        const uint4* src = reinterpret_cast<const uint4*>(w_r + (size_t)d0 * EP);
        constexpr int B = 8;
        for (int v0 = lane; v0 < nvec; v0 += 32 * B) {
            uint4 r[B];
#pragma unroll
            for (int b = 0; b < B; ++b)
                if (v0 + 32 * b < nvec) r[b] = __ldg(src + v0 + 32 * b);
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int v = v0 + 32 * b;
                if (v < nvec) {
                    const int d = d0 + (8 * v) / EP, e0 = (8 * v) % EP;
                    const __nv_bfloat16* el = reinterpret_cast<const __nv_bfloat16*>(&r[b]);
#pragma unroll
                    for (int i = 0; i < 8; ++i) wT[(size_t)(e0 + i) * stride + d] = el[i];
                }
            }
        }
    } else {
        for (int f = lane; f < (d1 - d0) * EP; f += 32) {
            const int d = d0 + f / EP, e = f % EP;
            wT[(size_t)e * stride + d] = e < E ? w_r[(size_t)d * E + e] : zero;
        }
    }
    for (int f = lane; f < (dz - d1) * EP; f += 32) wT[(size_t)(f % EP) * stride + d1 + f / EP] = zero;
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
    __syncthreads();

    float Pacc[1] = {0.f};
    const bool use_bias_in_logits = bias && bias_in_logits(gating);
    const int ntiles = (T_ + kMmaTokens - 1) / kMmaTokens;
    auto load = [&](uint4 (&xa)[U], uint4 (&xb)[U], const __nv_bfloat16* x0, const __nv_bfloat16* x1, int c0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int d = (c0 + u) * 32 + 8 * t;
            if (c0 + u < c_end && d < h) {
                xa[u] = __ldcs(reinterpret_cast<const uint4*>(x0 + d));
                xb[u] = __ldcs(reinterpret_cast<const uint4*>(x1 + d));
            } else {
                xa[u] = make_uint4(0, 0, 0, 0);
                xb[u] = make_uint4(0, 0, 0, 0);
            }
        }
    };
    auto compute = [&](float (&acc)[NB][4], const uint4 (&xa)[U], const uint4 (&xb)[U], int c0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (c0 + u < c_end) {
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                    const uint4 wv = *reinterpret_cast<const uint4*>(wT + (size_t)(8 * nb + g) * stride +
                                                                    (c0 + u) * 32 + 8 * t);
                    mma_bf16_16816(acc[nb], xa[u].x, xb[u].x, xa[u].y, xb[u].y, wv.x, wv.y);
                    mma_bf16_16816(acc[nb], xa[u].z, xb[u].z, xa[u].w, xb[u].w, wv.z, wv.w);
                }
            }
        }
    };
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int tok0 = tile * kMmaTokens;
        // the next tile of this block goes to L2 while this one is computed (the first one was prefetched at entry)
        if (threadIdx.x < kMmaTokens && tile + (int)gridDim.x < ntiles) prefetch_row_l2(x, T_, h, tok0 + (int)gridDim.x * kMmaTokens + threadIdx.x);
        const __nv_bfloat16* x0 = x + (size_t)min(tok0 + g, T_ - 1) * h;          // rows past T: any valid row,
        const __nv_bfloat16* x1 = x + (size_t)min(tok0 + g + 8, T_ - 1) * h;      // their logits are not used
        float acc[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
        // two register buffers of U chunks: the loads of one are in flight while the other is multiplied
        uint4 a0[U], b0[U], a1[U], b1[U];
        load(a0, b0, x0, x1, c_begin);
        if (w_rT && tile == (int)blockIdx.x) {
            if (threadIdx.x == 0) {
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(wbar),
                             "r"((unsigned)(E * h * 2)) : "memory");
                for (int e = 0; e < E; ++e)
                    bulk_row_to_shared((uint32_t)__cvta_generic_to_shared(wT + (size_t)e * stride),
                                       w_rT + (size_t)e * h, (uint32_t)(h * 2), wbar);
            }
            if (!bar_wait(wbar, 0, wait_limit)) {
                // the weight did not land in time: report it, and wait for the copy before going on (no copy may
                // land in the shared memory of an exited block); the results of this call are not to be used
                latch_device_error(err, kDevErrTimeout, 0x130u);
                if (!bar_wait(wbar, 0, kWeightDrainLimit)) latch_device_error(err, kDevErrTimeout, 0x131u);
            }
        }
        for (int c0 = c_begin; c0 < c_end; c0 += 2 * U) {
            load(a1, b1, x0, x1, c0 + U);
            compute(acc, a0, b0, c0);
            load(a0, b0, x0, x1, c0 + 2 * U);
            compute(acc, a1, b1, c0 + U);
        }
        // D fragment: rows g and g + 8 (tokens), columns 2t, 2t + 1 of each 8-expert block
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            float* r = red + (size_t)warp * kMmaTokens * EP + 8 * nb + 2 * t;
            r[g * EP] = acc[nb][0];
            r[g * EP + 1] = acc[nb][1];
            r[(g + 8) * EP] = acc[nb][2];
            r[(g + 8) * EP + 1] = acc[nb][3];
        }
        __syncthreads();
        // gating of the tile's 16 tokens: with E <= 16 warp w gates tokens 2w (lanes 0-15) and 2w + 1 (lanes
        // 16-31) at once, one expert per lane; otherwise the two one after the other, lane e holding expert e.
        // Lane e sums expert e's partial logits over the 8 warps' slices in slice order.
        if constexpr (EP <= 16) {
            const int j = 2 * warp + (lane >> 4), e = lane & 15;
            const int tok = tok0 + j;
            const bool tv = tok < T_;
            float L[1] = {-INFINITY};
            if (tv && e < E) {
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < kRouterWarps; ++w) v += red[((size_t)w * kMmaTokens + j) * EP + e];
                L[0] = v + (use_bias_in_logits ? bias[e] : 0.f);
                if (o.logits) o.logits[(size_t)tok * E + e] = L[0];
            }
            gate_token<1, 16>(L, tv ? tok : 0, E, k, gating, bias, o, Pacc, s_hist, tv);
        } else {
#pragma unroll
            for (int j = 2 * warp; j < 2 * warp + 2; ++j) {
                const int tok = tok0 + j;
                if (tok >= T_) break;
                float L[1] = {-INFINITY};
                if (lane < E) {
                    float v = 0.f;
#pragma unroll
                    for (int w = 0; w < kRouterWarps; ++w) v += red[((size_t)w * kMmaTokens + j) * EP + lane];
                    L[0] = v + (use_bias_in_logits ? bias[lane] : 0.f);
                    if (o.logits) o.logits[(size_t)tok * E + lane] = L[0];
                }
                gate_token<1>(L, tok, E, k, gating, bias, o, Pacc, s_hist);
            }
        }
        __syncthreads();                      // red is rewritten by the next tile
    }
    if constexpr (EP <= 16) Pacc[0] += __shfl_down_sync(0xffffffffu, Pacc[0], 16);   // expert e: lanes e and e + 16
    flush_partials<1>(Pacc, E, s_P, s_hist, o);
}

// ---------------------------------------------------------------------------------------------------
// E > 32: logits GEMM (fp32 accumulation, CUDA cores), then the gating kernel
// ---------------------------------------------------------------------------------------------------
// C[T,E] = x[T,h] @ W[h,E] (+ bias in softmax modes). 64x64 tiles, 16-deep K steps, 4x4 per thread. w_kmajor: w is
// the transpose W^T [E][h] (the packed router weight) instead of W [h][E].
template <typename T>
__global__ void __launch_bounds__(256)
router_logits_gemm(const T* __restrict__ x, const T* __restrict__ w, const float* __restrict__ bias, int T_, int h,
                   int E, float* __restrict__ out, int w_kmajor) {
    __shared__ float As[16][64 + 4];
    __shared__ float Bs[16][64 + 4];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < h; k0 += 16) {
        for (int i = threadIdx.x; i < 64 * 16; i += 256) {
            int r = i / 16, c = i % 16;                     // A: row r, k c
            int gm = m0 + r, gk = k0 + c;
            As[c][r] = (gm < T_ && gk < h) ? to_f32(x[(size_t)gm * h + gk]) : 0.f;
            int kr = i / 64, nc = i % 64;                   // B: k kr, col nc
            int bk = k0 + kr, bn = n0 + nc;
            Bs[kr][nc] = (bk < h && bn < E) ? to_f32(w_kmajor ? w[(size_t)bn * h + bk] : w[(size_t)bk * E + bn]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) { a[i] = As[kk][ty * 4 + i]; b[i] = Bs[kk][tx * 4 + i]; }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int gm = m0 + ty * 4 + i;
        if (gm >= T_) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int gn = n0 + tx * 4 + j;
            if (gn < E) out[(size_t)gm * E + gn] = acc[i][j] + (bias ? bias[gn] : 0.f);
        }
    }
}

// Gating on stored logits. The logits of token t are sum over q < nparts of logits[q part_stride + t E + e]
// (split-K partial products, added in part order) + lbias[e] (null: none); when o.logits is set the sums are
// written there.
template <int NPL>
__global__ void __launch_bounds__(kRouterWarps * 32)
router_gate_kernel(const float* __restrict__ logits, int nparts, size_t part_stride, const float* __restrict__ lbias,
                   const float* __restrict__ bias, int T_, int E, int k, int gating, GateOut o) {
    pdl_trigger();                            // the finalize may launch now (it waits for this kernel's partials)
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float* s_P = reinterpret_cast<float*>(smem_raw);
    int* s_hist = reinterpret_cast<int*>(s_P + kRouterWarps * E);
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float Pacc[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) Pacc[i] = 0.f;
    for (int t = blockIdx.x * kRouterWarps + warp; t < T_; t += gridDim.x * kRouterWarps) {
        float L[NPL];
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            int e = lane + 32 * i;
            L[i] = e < E ? logits[(size_t)t * E + e] : -INFINITY;
        }
        if (nparts > 1 || lbias) {
            int q = 1;
            for (; q + 3 < nparts; q += 4) {             // four parts' loads in flight, added in part order
                float v[4][NPL];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float* lq = logits + (q + u) * part_stride + (size_t)t * E;
#pragma unroll
                    for (int i = 0; i < NPL; ++i) {
                        int e = lane + 32 * i;
                        v[u][i] = e < E ? lq[e] : 0.f;
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int i = 0; i < NPL; ++i) L[i] += v[u][i];
            }
            for (; q < nparts; ++q) {
                const float* lq = logits + q * part_stride + (size_t)t * E;
#pragma unroll
                for (int i = 0; i < NPL; ++i) {
                    int e = lane + 32 * i;
                    if (e < E) L[i] += lq[e];
                }
            }
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
                int e = lane + 32 * i;
                if (e < E && lbias) L[i] += lbias[e];
            }
        }
        if (o.logits) {
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
                int e = lane + 32 * i;
                if (e < E) o.logits[(size_t)t * E + e] = L[i];
            }
        }
        gate_token<NPL>(L, t, E, k, gating, bias, o, Pacc, s_hist);
    }
    __syncthreads();
    flush_partials<NPL>(Pacc, E, s_P, s_hist, o);
}

// Counts, f, P and aux from the per-block partials of `grid` gating blocks. Each block takes chunks of
// kFinExperts experts (block b: chunks b, b + gridDim.x, ...). Thread (s, i) of its [kFinSlices][kFinExperts]
// arrangement sums the partials of gating blocks s, s + kFinSlices, ... of expert e0 + i (four loads in flight;
// a warp's loads read 8 consecutive experts of 4 rows); the 4 slices of a warp are added by a shuffle tree, then
// the 32 warps' sums by one warp (eight in warp order per lane, then a shuffle tree). Every block adds its experts' f_e P_e in expert order; with several blocks, the
// last one to arrive (counted on `ticket`, which the gating kernel zeroed) adds the blocks' sums in block order.
// No step depends on timing, so the results are the same on every run.
constexpr int kFinExperts = 8;
constexpr int kFinThreads = 1024;
constexpr int kFinSlices = kFinThreads / kFinExperts;
__global__ void __launch_bounds__(kFinThreads, 1)
router_finalize(const float* __restrict__ partial_P, const int32_t* __restrict__ partial_C, int grid, int T_, int E,
                int k, float alpha, int32_t* counts, float* f, float* P, float* aux, float* term_part,
                unsigned* ticket) {
    pdl_wait();                               // the gating kernel's partials and its zeroed ticket
    constexpr int NW = kFinThreads / 32;
    __shared__ float s_p[NW][kFinExperts];
    __shared__ int s_c[NW][kFinExperts];
    __shared__ float s_t[kFinExperts];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int sl = tid / kFinExperts, i = tid % kFinExperts;
    float term = 0.f;                                    // thread 0: this block's sum of f_e P_e
    for (int e0 = blockIdx.x * kFinExperts; e0 < E; e0 += gridDim.x * kFinExperts) {
        const int e = e0 + i;
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
        int cs[4] = {0, 0, 0, 0};
        if (e < E) {
            int b = sl;
            for (; b + 3 * kFinSlices < grid; b += 4 * kFinSlices) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    ps[u] += partial_P[(size_t)(b + u * kFinSlices) * E + e];
                    cs[u] += partial_C[(size_t)(b + u * kFinSlices) * E + e];
                }
            }
            for (; b < grid; b += kFinSlices) {
                ps[0] += partial_P[(size_t)b * E + e];
                cs[0] += partial_C[(size_t)b * E + e];
            }
        }
        float tp = (ps[0] + ps[1]) + (ps[2] + ps[3]);
        int tc = cs[0] + cs[1] + cs[2] + cs[3];
#pragma unroll
        for (int o = 16; o >= kFinExperts; o >>= 1) {      // the warp's slices of expert i: lanes i, i + 8, ...
            tp += __shfl_down_sync(0xffffffffu, tp, o);
            tc += __shfl_down_sync(0xffffffffu, tc, o);
        }
        if (lane < kFinExperts) {
            s_p[warp][lane] = tp;
            s_c[warp][lane] = tc;
        }
        __syncthreads();
        if (warp == 0) {          // lane (q, i): warps 8q .. 8q + 7 of expert i in order, then a shuffle tree over q
            constexpr int WQ = NW / (32 / kFinExperts);
            const int q = lane / kFinExperts;
            float sp = 0.f;
            int sc = 0;
#pragma unroll
            for (int w = 0; w < WQ; ++w) {
                sp += s_p[q * WQ + w][i];
                sc += s_c[q * WQ + w][i];
            }
#pragma unroll
            for (int o = 16; o >= kFinExperts; o >>= 1) {
                sp += __shfl_down_sync(0xffffffffu, sp, o);
                sc += __shfl_down_sync(0xffffffffu, sc, o);
            }
            if (lane < kFinExperts && e < E) {
                const float Pe = T_ > 0 ? sp / (float)T_ : 0.f;
                const float fe = T_ > 0 ? (float)sc / ((float)k * (float)T_) : 0.f;
                counts[e] = sc;
                f[e] = fe;
                P[e] = Pe;
                s_t[lane] = fe * Pe;
            }
        }
        __syncthreads();
        if (tid == 0)
            for (int j = 0; j < min(kFinExperts, E - e0); ++j) term += s_t[j];
        __syncthreads();                                 // s_p, s_c and s_t are rewritten by the next chunk
    }
    if (tid != 0) return;
    if (gridDim.x == 1) { aux[0] = alpha * (float)E * term; return; }
    term_part[blockIdx.x] = term;
    __threadfence();
    if (atomicAdd(ticket, 1u) != gridDim.x - 1) return;
    __threadfence();
    float sum = 0.f;
    for (unsigned b = 0; b < gridDim.x; ++b) sum += __ldcg(term_part + b);
    aux[0] = alpha * (float)E * sum;
}

// W_r [h, E] -> W_rT [E, h]: the K-major operand of the tensor-core logits GEMM. 32 x 32 shared-memory tiles.
template <typename T>
__global__ void __launch_bounds__(256)
router_transpose_kernel(const T* __restrict__ w, int h, int E, T* __restrict__ wT) {
    __shared__ T tile[32][33];
    const int e0 = blockIdx.x * 32, d0 = blockIdx.y * 32;
    for (int r = threadIdx.y; r < 32; r += 8) {
        const int d = d0 + r, e = e0 + threadIdx.x;
        if (d < h && e < E) tile[r][threadIdx.x] = w[(size_t)d * E + e];
    }
    __syncthreads();
    for (int r = threadIdx.y; r < 32; r += 8) {
        const int e = e0 + r, d = d0 + threadIdx.x;
        if (e < E && d < h) wT[(size_t)e * h + d] = tile[threadIdx.x][r];
    }
}

// ---------------------------------------------------------------------------------------------------
// host
// ---------------------------------------------------------------------------------------------------
// Upper bound of the blocks of any router launch (sizes the partial-sum workspace).
static int router_grid(int T) { return std::max(1, std::min(cdiv(T, kRouterWarps), kRouterMaxBlocks)); }
// The gating kernel on stored logits: a few tokens per warp, as many blocks as are resident at once (its per-token
// latency chain needs the warps), at most router_grid(T) (the size of the per-block partials in the workspace).
template <int N>
static int gate_grid(int T, size_t smem) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, router_gate_kernel<N>, kRouterWarps * 32, smem) !=
            cudaSuccess || per_sm < 1)
        per_sm = 1;
    return std::max(1, std::min(router_grid(T), per_sm * num_sms()));
}
// The fused small-E kernel stages the router weight into every block and takes two tokens per warp; its register
// budget allows two blocks per SM for E <= 8, one otherwise.
static int router_small_grid(int T, int E) {
    return std::max(1, std::min(cdiv(T, 2 * kRouterWarps), (E <= 8 ? 2 : 1) * num_sms()));
}

static size_t small_smem_bytes(int h, int E, int el) {
    return align_up((size_t)E * h * el, 16) + (size_t)kRouterWarps * E * sizeof(float) + (size_t)E * sizeof(int);
}
// 8-expert blocks of the bf16 fused kernel instantiated for E (1, 2 or 4): sizes its shared memory and picks
// the launch, so the two always agree.
static int mma_blocks(int E) { return E <= 8 ? 1 : E <= 16 ? 2 : 4; }
// The bf16 fused kernel on mma.sync: W_r^T padded to 8-expert blocks, the per-warp partial logits, P, counts.
static size_t mma_smem_bytes(int h, int E) {
    const int EP = 8 * mma_blocks(E);
    return (size_t)EP * mma_wt_stride(h) * 2 + (size_t)kRouterWarps * kMmaTokens * EP * sizeof(float) +
           (size_t)kRouterWarps * E * sizeof(float) + (size_t)E * sizeof(int) + 16;   // + the weight's mbarrier
}
static int router_mma_grid(int T) { return std::max(1, std::min(cdiv(T, kMmaTokens), 2 * num_sms())); }
static bool use_small_path(int h, int E, int el) {
    return E <= 32 && (el == 2 ? mma_smem_bytes(h, E) : small_smem_bytes(h, E, el)) <= 200 * 1024;
}

// The logits GEMM runs on the tcgen05 tensor cores for bf16 with E > 32 (E % 4 == 0 keeps the fp32 row
// stores 16-byte aligned); otherwise on the CUDA cores.
static bool use_tc_logits(int E, int dtype, bool small) { return !small && dtype == MOE_BF16 && E % 4 == 0; }

// Split of the tensor-core logits GEMM's contraction: with fewer 128 x 256 output tiles than SMs, the K range is
// cut into S chunks of kchunk columns (a multiple of 64, every chunk non-empty), S <= 16, so that about one tile
// of one chunk lands on each SM. S = 1: no split.
struct RouterSplit { int S, kchunk; };
static RouterSplit router_split(int T, int h, int E, bool tc) {
    if (!tc || T <= 0) return {1, h};
    RouterSplit r{1, h};
    tc_splitk_plan(T, E, h, &r.S, &r.kchunk);
    return r;
}

struct RouterWs {
    float* partial_P; int32_t* partial_C; float* logits; void* w_rT; int32_t* sched; float* parts;
    unsigned* ticket; float* term_part; size_t bytes;
};

// Blocks of the finalize: one per kFinExperts experts when gating blocks zeroed its arrival counter (T > 0).
static int finalize_grid(int T, int E) { return T > 0 ? cdiv(E, kFinExperts) : 1; }

static RouterWs router_ws_layout(void* ws, int T, int h, int E, int el, bool small, bool need_logits, bool tc,
                                 int split) {
    RouterWs w{};
    const int G = router_grid(T);
    size_t off = 0;
    char* base = static_cast<char*>(ws);
    w.partial_P = reinterpret_cast<float*>(base + off); off = align_up(off + (size_t)G * E * 4, 256);
    w.partial_C = reinterpret_cast<int32_t*>(base + off); off = align_up(off + (size_t)G * E * 4, 256);
    w.ticket = reinterpret_cast<unsigned*>(base + off); off = align_up(off + 4, 256);
    w.term_part = reinterpret_cast<float*>(base + off); off = align_up(off + (size_t)cdiv(E, kFinExperts) * 4, 256);
    w.logits = nullptr;
    if (need_logits) { w.logits = reinterpret_cast<float*>(base + off); off = align_up(off + (size_t)T * E * 4, 256); }
    w.w_rT = nullptr;
    w.sched = nullptr;
    if (tc) {                                // transposed weight: the tensor-core GEMM's K-major operand
        w.w_rT = base + off; off = align_up(off + (size_t)E * h * el, 256);
    }
    if (tc) { w.sched = reinterpret_cast<int32_t*>(base + off); off = align_up(off + sched_words(T, 1) * 4, 256); }
    w.parts = nullptr;
    if (split > 1) { w.parts = reinterpret_cast<float*>(base + off); off = align_up(off + (size_t)split * T * E * 4, 256); }
    w.bytes = off;
    return w;
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_router_workspace_size(int T, int h, int E, int k, int dtype) {
    (void)k;
    if (T < 0 || h <= 0 || E <= 0) return 0;
    const int el = dtype == MOE_F32 ? 4 : 2;
    const bool small = use_small_path(h, E, el);
    const bool tc = use_tc_logits(E, dtype, small);
    return router_ws_layout(nullptr, T, h, E, el, small, !small, tc, router_split(T, h, E, tc).S).bytes;
}

// The router on w_r [h][E], or (bf16, w_r null) on the packed transpose w_rT [E][h] of moe_pack_router_weight,
// which spares the tensor-core path its per-call transpose and the fused small-E kernel its scattered staging.
static int router_run(const void* x, const void* w_r, const void* w_rT, const float* bias, int T, int h, int E, int k,
                      int dtype, int gating, float alpha, float* logits, int32_t* topk_ids, float* gates,
                      int32_t* counts, float* f, float* P, float* aux, void* ws, size_t ws_bytes, void* stream) {
    MOE_REQUIRE(dtype == MOE_F32 || dtype == MOE_BF16, MOE_ERR_UNSUPPORTED, "moe_router: dtype %d", dtype);
    MOE_REQUIRE(gating >= MOE_GATING_SOFTMAX && gating <= MOE_GATING_SOFTMAX_SELBIAS, MOE_ERR_UNSUPPORTED,
                "moe_router: gating mode %d", gating);
    MOE_REQUIRE(T >= 0 && h > 0 && h % 8 == 0, MOE_ERR_INVALID_ARG, "moe_router: T=%d h=%d (need T>=0, h%%8==0)", T, h);
    MOE_REQUIRE(E >= 1 && E <= 1024 && k >= 1 && k <= E && k <= kMaxK, MOE_ERR_INVALID_ARG,
                "moe_router: E=%d k=%d (need 1<=k<=min(E,16), E<=1024)", E, k);
    MOE_REQUIRE((w_r || w_rT) && counts && f && P && aux && (T == 0 || (x && topk_ids && gates)), MOE_ERR_INVALID_ARG,
                "moe_router: null pointer");
    MOE_REQUIRE(aligned16(x) && aligned16(w_r) && aligned16(w_rT) && aligned16(logits), MOE_ERR_INVALID_ARG,
                "moe_router: x, w_r and logits must be 16-byte aligned");
    const int el = dtype == MOE_F32 ? 4 : 2;
    const bool small = use_small_path(h, E, el);
    const bool tc = use_tc_logits(E, dtype, small);
    const RouterSplit sp = router_split(T, h, E, tc);
    RouterWs w = router_ws_layout(ws, T, h, E, el, small, !small && logits == nullptr && sp.S == 1, tc, sp.S);
    MOE_REQUIRE(ws_bytes >= w.bytes && (w.bytes == 0 || ws), MOE_ERR_WORKSPACE,
                "moe_router: workspace %zu < %zu bytes", ws_bytes, w.bytes);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int G = !small ? 1 : dtype == MOE_BF16 ? router_mma_grid(T) : router_small_grid(T, E);   // !small: set at launch
    GateOut o{topk_ids, gates, logits, w.partial_P, w.partial_C, w.ticket};
    if (T > 0) {
        if (small && dtype == MOE_BF16) {
            const size_t smem = mma_smem_bytes(h, E);
            unsigned* err = device_error_word();
            MOE_REQUIRE(err, MOE_ERR_CUDA, "moe_router: device error word unavailable");
            const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
            const __nv_bfloat16* wb = static_cast<const __nv_bfloat16*>(w_r);
            const __nv_bfloat16* wtb = static_cast<const __nv_bfloat16*>(w_rT);
#define MOE_MMA_LAUNCH(NB, UU)                                                                                \
            cudaFuncSetAttribute(router_mma_kernel<NB, UU>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
            router_mma_kernel<NB, UU><<<G, kRouterWarps * 32, smem, s>>>(xb, wb, wtb, bias, T, h, E, k, gating, o, err, \
                                                                      wait_limit());
            switch (mma_blocks(E)) {
                case 1: { MOE_MMA_LAUNCH(1, 4) } break;
                case 2: { MOE_MMA_LAUNCH(2, 4) } break;
                default: { MOE_MMA_LAUNCH(4, 2) } break;
            }
#undef MOE_MMA_LAUNCH
            if (int rc = check_launch("router_mma_kernel")) return rc;
        } else if (small) {
            const size_t smem = small_smem_bytes(h, E, el);
#define MOE_SMALL_LAUNCH(EM, UU)                                                                              \
            cudaFuncSetAttribute(router_small_kernel<float, EM, UU>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                 (int)smem);                                                                  \
            router_small_kernel<float, EM, UU><<<G, kRouterWarps * 32, smem, s>>>(static_cast<const float*>(x), \
                static_cast<const float*>(w_r), bias, T, h, E, k, gating, o);
            if (E <= 8) { MOE_SMALL_LAUNCH(8, 2) }
            else if (E <= 16) { MOE_SMALL_LAUNCH(16, 2) }
            else { MOE_SMALL_LAUNCH(32, 2) }
#undef MOE_SMALL_LAUNCH
            if (int rc = check_launch("router_small_kernel")) return rc;
        } else {
            float* lg = sp.S > 1 ? w.parts : logits ? logits : w.logits;
            const float* lbias = bias_in_logits(gating) ? bias : nullptr;
            if (tc) {
                const void* wt = w_rT;
                if (!wt) {                           // not packed: transpose into the workspace on every call
                    router_transpose_kernel<__nv_bfloat16><<<dim3(cdiv(E, 32), cdiv(h, 32)), dim3(32, 8), 0, s>>>(
                        static_cast<const __nv_bfloat16*>(w_r), h, E, static_cast<__nv_bfloat16*>(w.w_rT));
                    if (int rc = check_launch("router_transpose_kernel")) return rc;
                    wt = w.w_rT;
                }
                if (sp.S > 1) {
                    if (int rc = tc_gemm_f32_splitk(x, T, h, 0, wt, E, h, 0, h, sp.S, sp.kchunk, lg, s)) return rc;
                } else {
                    if (int rc = launch_dense_sched(T, w.sched, s)) return rc;
                    if (int rc = tc_router_logits(x, wt, lbias, T, h, E, w.sched, lg, s)) return rc;
                }
            } else {
                dim3 grid(cdiv(E, 64), cdiv(T, 64));
                if (dtype == MOE_BF16)
                    router_logits_gemm<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x),
                        static_cast<const __nv_bfloat16*>(w_r ? w_r : w_rT), lbias, T, h, E, lg, w_r ? 0 : 1);
                else
                    router_logits_gemm<float><<<grid, 256, 0, s>>>(static_cast<const float*>(x),
                        static_cast<const float*>(w_r), lbias, T, h, E, lg, 0);
                if (int rc = check_launch("router_logits_gemm")) return rc;
            }
            const size_t smem = (size_t)kRouterWarps * E * sizeof(float) + (size_t)E * sizeof(int);
            const int npl = cdiv(E, 32);
            // unsplit: the GEMM wrote the final logits (bias included); split: the gate adds the parts and the bias
            o.logits = sp.S > 1 ? logits : nullptr;
            const float* gbias = sp.S > 1 ? lbias : nullptr;
            const size_t pstride = (size_t)T * E;
#define MOE_GATE_LAUNCH(N)                                                                              \
            cudaFuncSetAttribute(router_gate_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
            G = gate_grid<N>(T, smem);                                                                         \
            router_gate_kernel<N><<<G, kRouterWarps * 32, smem, s>>>(lg, sp.S, pstride, gbias, bias, T, E, k, gating, o);
            if (npl <= 2) { MOE_GATE_LAUNCH(2) }
            else if (npl <= 4) { MOE_GATE_LAUNCH(4) }
            else if (npl <= 8) { MOE_GATE_LAUNCH(8) }
            else if (npl <= 16) { MOE_GATE_LAUNCH(16) }
            else { MOE_GATE_LAUNCH(32) }
#undef MOE_GATE_LAUNCH
            if (int rc = check_launch("router_gate_kernel")) return rc;
        }
    }
    const cudaError_t le = launch_pdl(router_finalize, dim3(finalize_grid(T, E)), dim3(kFinThreads), 0, s,
                                      (const float*)w.partial_P, (const int32_t*)w.partial_C, T > 0 ? G : 0, T, E, k,
                                      alpha, counts, f, P, aux, w.term_part, w.ticket);
    return check_launch(le, "router_finalize");
}

extern "C" int moe_router(const void* x, const void* w_r, const float* bias, int T, int h, int E, int k, int dtype,
                          int gating, float alpha, float* logits, int32_t* topk_ids, float* gates, int32_t* counts,
                          float* f, float* P, float* aux, void* ws, size_t ws_bytes, void* stream) {
    return router_run(x, w_r, nullptr, bias, T, h, E, k, dtype, gating, alpha, logits, topk_ids, gates, counts, f, P,
                      aux, ws, ws_bytes, stream);
}

extern "C" size_t moe_router_packed_bytes(int h, int E, int dtype) {
    if (h <= 0 || E <= 0) return 0;
    return align_up((size_t)h * E * (dtype == MOE_F32 ? 4 : 2), 256);
}

extern "C" int moe_pack_router_weight(const void* w_r, int h, int E, int dtype, void* packed, void* stream) {
    MOE_REQUIRE(dtype == MOE_F32 || dtype == MOE_BF16, MOE_ERR_UNSUPPORTED, "moe_pack_router_weight: dtype %d", dtype);
    MOE_REQUIRE(h > 0 && h % 8 == 0 && E >= 1 && E <= 1024, MOE_ERR_INVALID_ARG, "moe_pack_router_weight: h=%d E=%d", h,
                E);
    MOE_REQUIRE(w_r && packed && aligned16(w_r) && aligned16(packed), MOE_ERR_INVALID_ARG,
                "moe_pack_router_weight: null or misaligned pointer");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == MOE_F32) {                  // the fp32 kernels read w_r as it is
        const cudaError_t e = cudaMemcpyAsync(packed, w_r, (size_t)h * E * 4, cudaMemcpyDeviceToDevice, s);
        MOE_REQUIRE(e == cudaSuccess, MOE_ERR_CUDA, "moe_pack_router_weight: %s", cudaGetErrorString(e));
        return MOE_OK;
    }
    router_transpose_kernel<__nv_bfloat16><<<dim3(cdiv(E, 32), cdiv(h, 32)), dim3(32, 8), 0, s>>>(
        static_cast<const __nv_bfloat16*>(w_r), h, E, static_cast<__nv_bfloat16*>(packed));
    return check_launch("router_transpose_kernel");
}

extern "C" int moe_router_packed(const void* x, const void* w_packed, const float* bias, int T, int h, int E, int k,
                                 int dtype, int gating, float alpha, float* logits, int32_t* topk_ids, float* gates,
                                 int32_t* counts, float* f, float* P, float* aux, void* ws, size_t ws_bytes,
                                 void* stream) {
    if (dtype == MOE_F32)
        return router_run(x, w_packed, nullptr, bias, T, h, E, k, dtype, gating, alpha, logits, topk_ids, gates, counts,
                          f, P, aux, ws, ws_bytes, stream);
    return router_run(x, nullptr, w_packed, bias, T, h, E, k, dtype, gating, alpha, logits, topk_ids, gates, counts, f,
                      P, aux, ws, ws_bytes, stream);
}

extern "C" size_t moe_router_from_logits_workspace_size(int T, int E) {
    if (T < 0 || E <= 0) return 0;
    return router_ws_layout(nullptr, T, 8, E, 4, false, false, false, 1).bytes;
}

extern "C" int moe_router_from_logits(const float* logits, const float* bias, int T, int E, int k, int gating,
                                      float alpha, int32_t* topk_ids, float* gates, int32_t* counts, float* f,
                                      float* P, float* aux, void* ws, size_t ws_bytes, void* stream) {
    MOE_REQUIRE(gating >= MOE_GATING_SOFTMAX && gating <= MOE_GATING_SOFTMAX_SELBIAS, MOE_ERR_UNSUPPORTED,
                "moe_router_from_logits: gating mode %d", gating);
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= 1024 && k >= 1 && k <= E && k <= kMaxK, MOE_ERR_INVALID_ARG,
                "moe_router_from_logits: T=%d E=%d k=%d", T, E, k);
    MOE_REQUIRE(counts && f && P && aux && (T == 0 || (logits && topk_ids && gates)), MOE_ERR_INVALID_ARG,
                "moe_router_from_logits: null pointer");
    const size_t need = moe_router_from_logits_workspace_size(T, E);
    MOE_REQUIRE(ws && ws_bytes >= need, MOE_ERR_WORKSPACE, "moe_router_from_logits: workspace %zu < %zu", ws_bytes,
                need);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int G = 1;                               // set at launch, <= router_grid(T), which sizes the workspace
    const RouterWs w = router_ws_layout(ws, T, 8, E, 4, false, false, false, 1);
    GateOut o{topk_ids, gates, nullptr, w.partial_P, w.partial_C, w.ticket};
    if (T > 0) {
        const size_t smem = (size_t)kRouterWarps * E * sizeof(float) + (size_t)E * sizeof(int);
        const int npl = cdiv(E, 32);
#define MOE_GATE_LAUNCH2(N)                                                                             \
        cudaFuncSetAttribute(router_gate_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
        G = gate_grid<N>(T, smem);                                                                         \
        router_gate_kernel<N><<<G, kRouterWarps * 32, smem, s>>>(logits, 1, 0, nullptr, bias, T, E, k, gating, o);
        if (npl <= 2) { MOE_GATE_LAUNCH2(2) }
        else if (npl <= 4) { MOE_GATE_LAUNCH2(4) }
        else if (npl <= 8) { MOE_GATE_LAUNCH2(8) }
        else if (npl <= 16) { MOE_GATE_LAUNCH2(16) }
        else { MOE_GATE_LAUNCH2(32) }
#undef MOE_GATE_LAUNCH2
        if (int rc = check_launch("router_gate_kernel")) return rc;
    }
    const cudaError_t le = launch_pdl(router_finalize, dim3(finalize_grid(T, E)), dim3(kFinThreads), 0, s,
                                      (const float*)o.partial_P, (const int32_t*)o.partial_C, T > 0 ? G : 0, T, E, k,
                                      alpha, counts, f, P, aux, w.term_part, w.ticket);
    return check_launch(le, "router_finalize");
}
