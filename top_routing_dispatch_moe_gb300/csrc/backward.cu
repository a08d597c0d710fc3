// Backward of the routing side of the layer: combine, router (gates and aux loss), router weight, dispatch.
//
// "专家并行" (formulaic), section "BWD（反向传播）" and the overlap notes: the gradients go back along the
// routing path to the experts, and each expert computes its own weight gradients. The pages give no formulas;
// this is the chain rule through the forward (combine.cu, router.cu, dispatch.cu) with the top-k selection,
// the counts and the capacity drops held constant. Every reduction runs in a fixed order (no atomics), so
// every output is deterministic.
#include <math.h>
#include <algorithm>
#include "ffn.cuh"

namespace moe {

constexpr int kBwdWarps = 8;

// ---------------------------------------------------------------------------------------------------
// combine backward: y[t] = sum_kept gate[t,j] eout[dest_row[t,j]]
// ---------------------------------------------------------------------------------------------------
// One warp per dispatched row r (token t = src_token[r], slot j = src_slot[r]): d_eout[r] = gate[t,j] dy[t]
// (pad rows: zero) and d_gates[t,j] = <dy[t], eout[r]> in fp32 (lane-strided partial sums, then a fixed
// butterfly). Pairs that were dropped get d_gates = 0 from a second grid-stride pass.
template <typename T>
__global__ void __launch_bounds__(kBwdWarps * 32)
combine_bwd_kernel(const T* __restrict__ dy, const T* __restrict__ eout, const int32_t* __restrict__ src_token,
                   const int32_t* __restrict__ src_slot, const int32_t* __restrict__ dest_row,
                   const float* __restrict__ gates, int T_, int h, int k, int rows, T* __restrict__ d_eout,
                   float* __restrict__ d_gates) {
    constexpr int V = Vec16<T>::N;
    const int lane = threadIdx.x & 31;
    const int nwarps = gridDim.x * kBwdWarps;
    for (int r = blockIdx.x * kBwdWarps + (threadIdx.x >> 5); r < rows; r += nwarps) {
        const int t = src_token[r];
        T* out = d_eout + (size_t)r * h;
        if (t < 0) {
            Vec16<T> z;
#pragma unroll
            for (int i = 0; i < V; ++i) z.set(i, 0.f);
            for (int d = lane * V; d < h; d += 32 * V) st16(out + d, z);
            continue;
        }
        const int j = src_slot[r];
        const float g = gates[(size_t)t * k + j];
        const T* dyr = dy + (size_t)t * h;
        const T* er = eout + (size_t)r * h;
        float dot = 0.f;
        for (int d = lane * V; d < h; d += 32 * V) {
            const Vec16<T> a = ld16(dyr + d), b = ld16_stream(er + d);
            Vec16<T> o;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                const float av = a.get(i);
                dot = fmaf(av, b.get(i), dot);
                o.set(i, g * av);
            }
            st16(out + d, o);
        }
        dot = warp_sum(dot);
        if (lane == 0) d_gates[(size_t)t * k + j] = dot;
    }
    const int tid = blockIdx.x * blockDim.x + threadIdx.x;
    for (int i = tid; i < T_ * k; i += gridDim.x * blockDim.x)
        if (dest_row[i] < 0) d_gates[i] = 0.f;
}

// ---------------------------------------------------------------------------------------------------
// router backward: d_logits from the gate gradients and the aux loss
// ---------------------------------------------------------------------------------------------------
// One warp per token, lane l holding experts l, l + 32, ... (NPL per lane). With c_e = d_aux alpha E f_e / T
// (the gradient of aux with respect to each token's router probability of e):
//   softmax (and softmax with a selection-only bias): dp_e = sum_j [ids_j = e] d_g_j + c_e
//   softmax_renorm: dp_e = sum_j [ids_j = e] (d_g_j - sum_i d_g_i g_i) / S + c_e, S = sum_j p[ids_j]
//   then dL = p (dp - <dp, p>)
//   sigmoid: ds_e = sum_j [ids_j = e] (d_g_j - sum_i d_g_i g_i) / S + (c_e - <c, q>) / sum(s), q = s / sum(s),
//   S = sum_j s[ids_j]; then dL = ds s (1 - s).
// Per-block partial sums of dL (the bias gradient in the softmax modes) in a fixed warp order.
template <int NPL>
__global__ void __launch_bounds__(kBwdWarps * 32)
router_bwd_kernel(const float* __restrict__ logits, const int32_t* __restrict__ ids, const float* __restrict__ gates,
                  const float* __restrict__ d_gates, const float* __restrict__ f, int T_, int E, int k, int gating,
                  float alpha, float d_aux, float* __restrict__ d_logits, float* __restrict__ partial_db) {
    extern __shared__ float s_db[];                       // [kBwdWarps][E]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float c[NPL], acc[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
        const int e = lane + 32 * i;
        c[i] = e < E ? d_aux * alpha * (float)E * f[e] / (float)T_ : 0.f;
        acc[i] = 0.f;
    }
    const bool sig = gating == MOE_GATING_SIGMOID_BIAS_RENORM;
    const bool renorm = gating == MOE_GATING_SOFTMAX_RENORM || sig;
    for (int t = blockIdx.x * kBwdWarps + warp; t < T_; t += gridDim.x * kBwdWarps) {
        float L[NPL], p[NPL];
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            const int e = lane + 32 * i;
            L[i] = e < E ? logits[(size_t)t * E + e] : 0.f;
        }
        float denom = 0.f;                                    // softmax: sum exp; sigmoid: sum s
        if (sig) {
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
                p[i] = (lane + 32 * i) < E ? 1.f / (1.f + expf(-L[i])) : 0.f;
                denom += p[i];
            }
            denom = warp_sum(denom);
        } else {
            float m = -INFINITY;
#pragma unroll
            for (int i = 0; i < NPL; ++i) if ((lane + 32 * i) < E) m = fmaxf(m, L[i]);
            m = warp_max(m);
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
                p[i] = (lane + 32 * i) < E ? expf(L[i] - m) : 0.f;
                denom += p[i];
            }
            denom = warp_sum(denom);
            const float inv = 1.f / denom;
#pragma unroll
            for (int i = 0; i < NPL; ++i) p[i] *= inv;
        }
        // the k chosen experts: their gate gradients, and (renormalised modes) S and sum_i d_g_i g_i
        float gsum = 0.f, S = 0.f;
        float dsel[NPL];
#pragma unroll
        for (int i = 0; i < NPL; ++i) dsel[i] = 0.f;
        for (int j = 0; j < k; ++j) {
            const int e = ids[(size_t)t * k + j];
            const float dg = d_gates[(size_t)t * k + j];
            gsum += dg * gates[(size_t)t * k + j];
            float pe = 0.f;
#pragma unroll
            for (int i = 0; i < NPL; ++i) if (i == (e >> 5)) pe = p[i];
            S += __shfl_sync(0xffffffffu, pe, e & 31);
#pragma unroll
            for (int i = 0; i < NPL; ++i) if (lane + 32 * i == e) dsel[i] += dg;
        }
        // dsel: sum_j [ids_j = e] d_g_j (the plain softmax gates' gradient per expert)
        float dL[NPL];
        if (sig) {
            float cq = 0.f;
#pragma unroll
            for (int i = 0; i < NPL; ++i) cq += c[i] * p[i];
            cq = warp_sum(cq) / denom;                             // <c, q>
            const float invS = 1.f / S, invD = 1.f / denom;
#pragma unroll
            for (int i = 0; i < NPL; ++i) dL[i] = 0.f;
            // chosen entries: (d_g - gsum) / S; the same expert appears at most once among the k
            for (int j = 0; j < k; ++j) {
                const int e = ids[(size_t)t * k + j];
                const float dg = d_gates[(size_t)t * k + j];
#pragma unroll
                for (int i = 0; i < NPL; ++i) if (lane + 32 * i == e) dL[i] += (dg - gsum) * invS;
            }
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
                const float ds = dL[i] + (c[i] - cq) * invD;
                dL[i] = (lane + 32 * i) < E ? ds * p[i] * (1.f - p[i]) : 0.f;
            }
        } else {
            float dp[NPL];
            if (renorm) {
                const float invS = 1.f / S;
#pragma unroll
                for (int i = 0; i < NPL; ++i) dp[i] = 0.f;
                for (int j = 0; j < k; ++j) {
                    const int e = ids[(size_t)t * k + j];
                    const float dg = d_gates[(size_t)t * k + j];
#pragma unroll
                    for (int i = 0; i < NPL; ++i) if (lane + 32 * i == e) dp[i] += (dg - gsum) * invS;
                }
            } else {
#pragma unroll
                for (int i = 0; i < NPL; ++i) dp[i] = dsel[i];
            }
            float dot = 0.f;
#pragma unroll
            for (int i = 0; i < NPL; ++i) {
                dp[i] += c[i];
                dot += dp[i] * p[i];
            }
            dot = warp_sum(dot);
#pragma unroll
            for (int i = 0; i < NPL; ++i) dL[i] = (lane + 32 * i) < E ? p[i] * (dp[i] - dot) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E) d_logits[(size_t)t * E + e] = dL[i];
            acc[i] += dL[i];
        }
    }
    if (partial_db) {
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
            const int e = lane + 32 * i;
            if (e < E) s_db[warp * E + e] = acc[i];
        }
        __syncthreads();
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            float s = 0.f;
            for (int w = 0; w < kBwdWarps; ++w) s += s_db[w * E + e];
            partial_db[(size_t)blockIdx.x * E + e] = s;
        }
    }
}

// out[e] = sum over b < G of partial[b][e], in block order (one thread per e).
__global__ void column_sum_kernel(const float* __restrict__ partial, int G, int E, float* __restrict__ out) {
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < E; e += gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int b = 0; b < G; ++b) s += partial[(size_t)b * E + e];
        out[e] = s;
    }
}

// ---------------------------------------------------------------------------------------------------
// Tensor-core path of the two router-weight products (bf16 x and W_r, E >= 64): d_logits is fp32, so each
// value v is written as three bf16 pieces v = p0 + p1 + p2 + r (p0 = bf16(v), p1 = bf16(v - p0),
// p2 = bf16(v - p0 - p1); |r| <= 2^-24 |v|), and the product with a bf16 operand runs as one GEMM over
// three times the reduction length (bf16 x bf16 products are exact in the fp32 accumulator). The result is
// the fp32 product up to the accumulation order, as on the CUDA cores.
// ---------------------------------------------------------------------------------------------------
__device__ __forceinline__ void split3(float v, __nv_bfloat16 (&q)[3]) {
    q[0] = __float2bfloat16_rn(v);
    float r = v - __bfloat162float(q[0]);
    q[1] = __float2bfloat16_rn(r);
    r -= __bfloat162float(q[1]);
    q[2] = __float2bfloat16_rn(r);
}

// dL [T][E] fp32 -> out [T][3 Ep] bf16: piece q of dL[t][e] at column q Ep + e, zero for e >= E.
__global__ void split3_rows_kernel(const float* __restrict__ dL, int T_, int E, int Ep, __nv_bfloat16* __restrict__ out) {
    const long long n = (long long)T_ * Ep;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(i / Ep), e = (int)(i - (long long)t * Ep);
        __nv_bfloat16 q[3];
        split3(e < E ? dL[(size_t)t * E + e] : 0.f, q);
        __nv_bfloat16* row = out + (size_t)t * 3 * Ep;
        row[e] = q[0];
        row[Ep + e] = q[1];
        row[2 * Ep + e] = q[2];
    }
}

// dL [T][E] fp32 -> out [E][3 Tp] bf16: piece q of dL[t][e] at out[e][q Tp + t], zero for t >= T (32 x 32 tiles).
__global__ void __launch_bounds__(256)
split3_cols_kernel(const float* __restrict__ dL, int T_, int E, int Tp, __nv_bfloat16* __restrict__ out) {
    __shared__ float tile[32][33];
    const int e0 = blockIdx.x * 32, t0 = blockIdx.y * 32;
    for (int r = threadIdx.y; r < 32; r += 8) {
        const int t = t0 + r, e = e0 + threadIdx.x;
        tile[r][threadIdx.x] = (t < T_ && e < E) ? dL[(size_t)t * E + e] : 0.f;
    }
    __syncthreads();
    for (int r = threadIdx.y; r < 32; r += 8) {
        const int e = e0 + r, t = t0 + threadIdx.x;
        if (e < E && t < Tp) {
            __nv_bfloat16 q[3];
            split3(tile[threadIdx.x][r], q);
            __nv_bfloat16* row = out + (size_t)e * 3 * Tp;
            row[t] = q[0];
            row[Tp + t] = q[1];
            row[2 * Tp + t] = q[2];
        }
    }
}

// x [R][C] -> xT [C][ldd]: xT[c][r] = x[r][c] for r < R, zero for R <= r < ldd (64 x 64 tiles).
template <typename T>
__global__ void __launch_bounds__(256)
transpose_pad_kernel(const T* __restrict__ x, int R, int C, int ldd, T* __restrict__ xT) {
    __shared__ T tile[64][65];
    const int c0 = blockIdx.x * 64, r0 = blockIdx.y * 64;
    for (int i = threadIdx.y; i < 64; i += blockDim.y) {
        const int r = r0 + i, c = c0 + threadIdx.x;
        tile[i][threadIdx.x] = (r < R && c < C) ? x[(size_t)r * C + c] : T(0.f);
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 64; i += blockDim.y) {
        const int c = c0 + i, r = r0 + threadIdx.x;
        if (c < C && r < ldd) xT[(size_t)c * ldd + r] = tile[threadIdx.x][i];
    }
}

// The tensor-core path applies to bf16 with E >= 64 experts (E % 8 == 0, h % 8 == 0).
static bool tc_router_bwd(int h, int E, int dtype) { return dtype == MOE_BF16 && E >= 64 && E % 8 == 0 && h % 8 == 0; }
static int round64(int v) { return (v + 63) / 64 * 64; }

// ---------------------------------------------------------------------------------------------------
// router weight gradient: dW_r[d][e] = sum_t x[t][d] dL[t][e]
// ---------------------------------------------------------------------------------------------------
// Block (column block of 256 d, token slice s): one thread per column d, experts in groups of 32 whose dL
// values for 64 tokens at a time sit in shared memory (read as broadcasts). Partial sums per slice, then a
// fixed-order sum over the slices.
constexpr int kWgCols = 256, kWgTok = 64;

template <typename T>
__global__ void __launch_bounds__(kWgCols)
router_wgrad_kernel(const T* __restrict__ x, const float* __restrict__ dL, int T_, int h, int E, int tslice,
                    float* __restrict__ partial) {
    __shared__ float s_dl[kWgTok][32];
    const int d = blockIdx.x * kWgCols + threadIdx.x;
    const int s = blockIdx.y;
    const int t0 = s * tslice, t1 = min(T_, t0 + tslice);
    for (int e0 = 0; e0 < E; e0 += 32) {
        float acc[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = 0.f;
        for (int tt = t0; tt < t1; tt += kWgTok) {
            __syncthreads();
            for (int i = threadIdx.x; i < kWgTok * 32; i += blockDim.x) {
                const int ti = i >> 5, ej = i & 31;
                s_dl[ti][ej] = (tt + ti < t1 && e0 + ej < E) ? dL[(size_t)(tt + ti) * E + e0 + ej] : 0.f;
            }
            __syncthreads();
            const int n = min(kWgTok, t1 - tt);
            for (int i = 0; i < n; ++i) {
                const float xv = d < h ? to_f32(x[(size_t)(tt + i) * h + d]) : 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[j] = fmaf(xv, s_dl[i][j], acc[j]);
            }
        }
        if (d < h)
            for (int j = 0; j < 32 && e0 + j < E; ++j) partial[((size_t)s * h + d) * E + e0 + j] = acc[j];
    }
}

// ---------------------------------------------------------------------------------------------------
// dispatch backward: dx[t] = extra[t] + sum_kept d_buf[dest_row[t,j]] + sum_e dL[t,e] W_r[:, e]
// ---------------------------------------------------------------------------------------------------
// One warp per token, 16-byte column chunks per lane, fp32 accumulation in a fixed order (extra, then the
// kept rows in ascending j, then the experts in ascending e); W_r^T [E][h] (transposed per call into the
// workspace) gives coalesced 16-byte reads of the router term.
template <typename T>
__global__ void __launch_bounds__(256)
wr_transpose_kernel(const T* __restrict__ w, int h, int E, T* __restrict__ wT) {
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

template <typename T, int KMAX>
__global__ void __launch_bounds__(256)
dispatch_bwd_kernel(const T* __restrict__ d_buf, const int32_t* __restrict__ dest_row, const float* __restrict__ dL,
                    const T* __restrict__ w_rT, const float* __restrict__ rterm, const T* __restrict__ extra, int T_,
                    int h, int k, int E, T* __restrict__ dx) {
    constexpr int V = Vec16<T>::N;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T_) return;
    const int myd = lane < k ? dest_row[(size_t)t * k + lane] : -1;
    int dj[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) dj[j] = __shfl_sync(0xffffffffu, myd, j);
    const float* dlt = dL ? dL + (size_t)t * E : nullptr;
    for (int d = lane * V; d < h; d += 32 * V) {
        float acc[V];
        if (extra) {
            const Vec16<T> v = ld16(extra + (size_t)t * h + d);
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] = v.get(i);
        } else {
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            if (j < k && dj[j] >= 0) {
                const Vec16<T> v = ld16_stream(d_buf + (size_t)dj[j] * h + d);
#pragma unroll
                for (int i = 0; i < V; ++i) acc[i] += v.get(i);
            }
        }
        if (rterm) {                         // the router term, summed over e by the tensor cores
            const float* rt = rterm + (size_t)t * h + d;
#pragma unroll
            for (int i = 0; i < V; i += 4) {
                const float4 v = *reinterpret_cast<const float4*>(rt + i);
                acc[i] += v.x; acc[i + 1] += v.y; acc[i + 2] += v.z; acc[i + 3] += v.w;
            }
        } else if (dlt) {
            for (int e = 0; e < E; ++e) {
                const float de = __ldg(dlt + e);
                const Vec16<T> w = ld16(w_rT + (size_t)e * h + d);
#pragma unroll
                for (int i = 0; i < V; ++i) acc[i] = fmaf(de, w.get(i), acc[i]);
            }
        }
        Vec16<T> o;
#pragma unroll
        for (int i = 0; i < V; ++i) o.set(i, acc[i]);
        st16(dx + (size_t)t * h + d, o);
    }
}

// Router weight gradient on the tensor cores: xT [h][Tp] (Tp = T rounded up to 64), the d_logits pieces
// [E][3 Tp], the split-K parts [S][h][E] (S > 1).
struct RwgTc { int Tp, S, kchunk; size_t xT_off, dl_off, parts_off, bytes; };
static RwgTc rwg_tc_layout(int T, int h, int E) {
    RwgTc L{};
    L.Tp = round64(std::max(T, 1));
    tc_splitk_plan(h, E, 3 * L.Tp, &L.S, &L.kchunk);
    L.xT_off = 0;
    L.dl_off = align_up((size_t)h * L.Tp * 2, 256);
    L.parts_off = L.dl_off + align_up((size_t)E * 3 * L.Tp * 2, 256);
    L.bytes = L.parts_off + (L.S > 1 ? align_up((size_t)L.S * h * E * 4, 256) : 0);
    return L;
}
// Dispatch backward on the tensor cores: the d_logits pieces [T][3 Ep] (Ep = E rounded up to 64), then the
// router term [T][h] fp32.
struct DbTc { int Ep; size_t dl_off, rterm_off, bytes; };
static DbTc db_tc_layout(int T, int h, int E) {
    DbTc L{};
    L.Ep = round64(E);
    L.dl_off = 0;
    L.rterm_off = align_up((size_t)T * 3 * L.Ep * 2, 256);
    L.bytes = L.rterm_off + align_up((size_t)T * h * 4, 256);
    return L;
}

static int bwd_router_grid(int T) { return std::max(1, std::min(cdiv(T, kBwdWarps), 2 * num_sms())); }
static int wgrad_slices(int T, int h) {
    const int cb = cdiv(h, kWgCols);
    return std::max(1, std::min(std::min(cdiv(T, kWgTok), 64), cdiv(2 * num_sms(), cb)));
}

}  // namespace moe

using namespace moe;

extern "C" int moe_combine_backward(const void* dy, const void* eout, const int32_t* src_token, const int32_t* src_slot,
                                    const int32_t* dest_row, const float* gates, int T, int h, int k, int rows,
                                    int dtype, void* d_eout, float* d_gates, void* stream) {
    MOE_REQUIRE(dtype == MOE_F32 || dtype == MOE_BF16, MOE_ERR_UNSUPPORTED, "moe_combine_backward: dtype %d", dtype);
    MOE_REQUIRE(T >= 0 && rows >= 0 && h > 0 && h % 8 == 0 && k >= 1 && k <= 32, MOE_ERR_INVALID_ARG,
                "moe_combine_backward: T=%d rows=%d h=%d k=%d", T, rows, h, k);
    if (T == 0 && rows == 0) return MOE_OK;
    MOE_REQUIRE(dy && eout && src_token && src_slot && dest_row && gates && d_eout && d_gates, MOE_ERR_INVALID_ARG,
                "moe_combine_backward: null pointer");
    MOE_REQUIRE(aligned16(dy) && aligned16(eout) && aligned16(d_eout), MOE_ERR_INVALID_ARG,
                "moe_combine_backward: dy, eout and d_eout must be 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int grid = std::max(1, std::min(cdiv(std::max(rows, 1), kBwdWarps), 4 * num_sms()));
    if (dtype == MOE_BF16)
        combine_bwd_kernel<__nv_bfloat16><<<grid, kBwdWarps * 32, 0, s>>>(
            static_cast<const __nv_bfloat16*>(dy), static_cast<const __nv_bfloat16*>(eout), src_token, src_slot, dest_row,
            gates, T, h, k, rows, static_cast<__nv_bfloat16*>(d_eout), d_gates);
    else
        combine_bwd_kernel<float><<<grid, kBwdWarps * 32, 0, s>>>(
            static_cast<const float*>(dy), static_cast<const float*>(eout), src_token, src_slot, dest_row, gates, T, h, k,
            rows, static_cast<float*>(d_eout), d_gates);
    return check_launch("combine_bwd_kernel");
}

extern "C" size_t moe_router_backward_workspace_size(int T, int E) {
    if (T < 0 || E <= 0) return 0;
    return align_up((size_t)bwd_router_grid(T) * E * sizeof(float), 256);
}

extern "C" int moe_router_backward(const float* logits, const int32_t* topk_ids, const float* gates,
                                   const float* d_gates, const float* f, int T, int E, int k, int gating, float alpha,
                                   float d_aux, float* d_logits, float* d_bias, void* ws, size_t ws_bytes,
                                   void* stream) {
    MOE_REQUIRE(gating >= MOE_GATING_SOFTMAX && gating <= MOE_GATING_SOFTMAX_SELBIAS, MOE_ERR_UNSUPPORTED,
                "moe_router_backward: gating mode %d", gating);
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= 1024 && k >= 1 && k <= E, MOE_ERR_INVALID_ARG,
                "moe_router_backward: T=%d E=%d k=%d", T, E, k);
    MOE_REQUIRE(T == 0 || (logits && topk_ids && gates && d_gates && f && d_logits), MOE_ERR_INVALID_ARG,
                "moe_router_backward: null pointer");
    const size_t need = moe_router_backward_workspace_size(T, E);
    MOE_REQUIRE(!d_bias || (ws && ws_bytes >= need), MOE_ERR_WORKSPACE, "moe_router_backward: workspace %zu < %zu",
                ws_bytes, need);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        if (d_bias && cudaMemsetAsync(d_bias, 0, (size_t)E * sizeof(float), s) != cudaSuccess)
            return set_error(MOE_ERR_CUDA, "moe_router_backward: memset failed");
        return MOE_OK;
    }
    const int G = bwd_router_grid(T);
    float* part = d_bias ? static_cast<float*>(ws) : nullptr;
    const size_t smem = (size_t)kBwdWarps * E * sizeof(float);
    const int npl = cdiv(E, 32);
#define MOE_RB_LAUNCH(N)                                                                                   \
    cudaFuncSetAttribute(router_bwd_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);    \
    router_bwd_kernel<N><<<G, kBwdWarps * 32, smem, s>>>(logits, topk_ids, gates, d_gates, f, T, E, k, gating, \
                                                         alpha, d_aux, d_logits, part);
    if (npl <= 1) { MOE_RB_LAUNCH(1) }
    else if (npl <= 2) { MOE_RB_LAUNCH(2) }
    else if (npl <= 4) { MOE_RB_LAUNCH(4) }
    else if (npl <= 8) { MOE_RB_LAUNCH(8) }
    else if (npl <= 16) { MOE_RB_LAUNCH(16) }
    else { MOE_RB_LAUNCH(32) }
#undef MOE_RB_LAUNCH
    if (int rc = check_launch("router_bwd_kernel")) return rc;
    if (!d_bias) return MOE_OK;
    column_sum_kernel<<<cdiv(E, 256), 256, 0, s>>>(part, G, E, d_bias);
    return check_launch("column_sum_kernel");
}

extern "C" size_t moe_router_weight_grad_workspace_size(int T, int h, int E) {
    if (T < 0 || h <= 0 || E <= 0) return 0;
    const size_t simt = align_up((size_t)wgrad_slices(std::max(T, 1), h) * h * E * sizeof(float), 256);
    return tc_router_bwd(h, E, MOE_BF16) ? std::max(simt, rwg_tc_layout(T, h, E).bytes) : simt;
}

extern "C" int moe_router_weight_grad(const void* x, const float* d_logits, int T, int h, int E, int dtype, float* dW_r,
                                      void* ws, size_t ws_bytes, void* stream) {
    MOE_REQUIRE(dtype == MOE_F32 || dtype == MOE_BF16, MOE_ERR_UNSUPPORTED, "moe_router_weight_grad: dtype %d", dtype);
    MOE_REQUIRE(T >= 0 && h > 0 && E >= 1 && E <= 1024, MOE_ERR_INVALID_ARG, "moe_router_weight_grad: T=%d h=%d E=%d",
                T, h, E);
    MOE_REQUIRE(dW_r && (T == 0 || (x && d_logits)), MOE_ERR_INVALID_ARG, "moe_router_weight_grad: null pointer");
    const size_t need = moe_router_weight_grad_workspace_size(T, h, E);
    MOE_REQUIRE(ws && ws_bytes >= need, MOE_ERR_WORKSPACE, "moe_router_weight_grad: workspace %zu < %zu", ws_bytes, need);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        if (cudaMemsetAsync(dW_r, 0, (size_t)h * E * sizeof(float), s) != cudaSuccess)
            return set_error(MOE_ERR_CUDA, "moe_router_weight_grad: memset failed");
        return MOE_OK;
    }
    if (tc_router_bwd(h, E, dtype)) {
        // dW_r = xT [h][Tp] times the pieces [E][3 Tp] over k < 3 Tp (x's column k mod Tp)
        const RwgTc L = rwg_tc_layout(T, h, E);
        char* base = static_cast<char*>(ws);
        __nv_bfloat16* xT = reinterpret_cast<__nv_bfloat16*>(base + L.xT_off);
        __nv_bfloat16* dlp = reinterpret_cast<__nv_bfloat16*>(base + L.dl_off);
        transpose_pad_kernel<__nv_bfloat16><<<dim3(cdiv(h, 64), L.Tp / 64), dim3(64, 4), 0, s>>>(
            static_cast<const __nv_bfloat16*>(x), T, h, L.Tp, xT);
        if (int rc = check_launch("transpose_pad_kernel")) return rc;
        split3_cols_kernel<<<dim3(cdiv(E, 32), L.Tp / 32), dim3(32, 8), 0, s>>>(d_logits, T, E, L.Tp, dlp);
        if (int rc = check_launch("split3_cols_kernel")) return rc;
        float* parts = L.S > 1 ? reinterpret_cast<float*>(base + L.parts_off) : dW_r;
        if (int rc = tc_gemm_f32_splitk(xT, h, L.Tp, L.Tp, dlp, E, 3 * L.Tp, 0, 3 * L.Tp, L.S, L.kchunk, parts, s))
            return rc;
        if (L.S == 1) return MOE_OK;
        column_sum_kernel<<<cdiv(h * E, 256), 256, 0, s>>>(parts, L.S, h * E, dW_r);
        return check_launch("column_sum_kernel");
    }
    const int S = wgrad_slices(T, h);
    const int tslice = cdiv(T, S);
    float* part = static_cast<float*>(ws);
    const dim3 grid(cdiv(h, kWgCols), S);
    if (dtype == MOE_BF16)
        router_wgrad_kernel<__nv_bfloat16><<<grid, kWgCols, 0, s>>>(static_cast<const __nv_bfloat16*>(x), d_logits, T,
                                                                    h, E, tslice, part);
    else
        router_wgrad_kernel<float><<<grid, kWgCols, 0, s>>>(static_cast<const float*>(x), d_logits, T, h, E, tslice,
                                                            part);
    if (int rc = check_launch("router_wgrad_kernel")) return rc;
    column_sum_kernel<<<cdiv(h * E, 256), 256, 0, s>>>(part, S, h * E, dW_r);
    return check_launch("column_sum_kernel");
}

extern "C" size_t moe_dispatch_backward_workspace_size(int T, int h, int E, int dtype) {
    if (T < 0 || h <= 0 || E <= 0) return 0;
    if (tc_router_bwd(h, E, dtype)) return db_tc_layout(T, h, E).bytes;
    return align_up((size_t)h * E * (dtype == MOE_F32 ? 4 : 2), 256);
}

extern "C" int moe_dispatch_backward(const void* d_buf, const int32_t* dest_row, const float* d_logits, const void* w_r,
                                     const void* dx_extra, int T, int h, int k, int E, int dtype, void* dx, void* ws,
                                     size_t ws_bytes, void* stream) {
    MOE_REQUIRE(dtype == MOE_F32 || dtype == MOE_BF16, MOE_ERR_UNSUPPORTED, "moe_dispatch_backward: dtype %d", dtype);
    MOE_REQUIRE(T >= 0 && h > 0 && h % 8 == 0 && k >= 1 && k <= 32 && E >= 1, MOE_ERR_INVALID_ARG,
                "moe_dispatch_backward: T=%d h=%d k=%d E=%d", T, h, k, E);
    if (T == 0) return MOE_OK;
    MOE_REQUIRE(d_buf && dest_row && dx && (!d_logits || w_r), MOE_ERR_INVALID_ARG, "moe_dispatch_backward: null pointer");
    MOE_REQUIRE(aligned16(d_buf) && aligned16(dx) && aligned16(dx_extra), MOE_ERR_INVALID_ARG,
                "moe_dispatch_backward: d_buf, dx and dx_extra must be 16-byte aligned");
    const size_t need = d_logits ? moe_dispatch_backward_workspace_size(T, h, E, dtype) : 0;
    MOE_REQUIRE(need == 0 || (ws && ws_bytes >= need && aligned16(ws)), MOE_ERR_WORKSPACE,
                "moe_dispatch_backward: workspace %zu < %zu", ws_bytes, need);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const dim3 tgrid(cdiv(E, 32), cdiv(h, 32)), tblock(32, 8);
    const int grid = cdiv(T, 8);
    const float* rterm = nullptr;
    if (d_logits && tc_router_bwd(h, E, dtype)) {
        // router term [T][h] = pieces [T][3 Ep] times W_r [h][E] over k < 3 Ep (W_r's column k mod Ep)
        const DbTc L = db_tc_layout(T, h, E);
        char* base = static_cast<char*>(ws);
        __nv_bfloat16* dlp = reinterpret_cast<__nv_bfloat16*>(base + L.dl_off);
        float* rt = reinterpret_cast<float*>(base + L.rterm_off);
        const long long n = (long long)T * L.Ep;
        split3_rows_kernel<<<(int)std::min<long long>(cdiv(n, 256), 8LL * num_sms()), 256, 0, s>>>(d_logits, T, E,
                                                                                                  L.Ep, dlp);
        if (int rc = check_launch("split3_rows_kernel")) return rc;
        if (int rc = tc_gemm_f32_splitk(dlp, T, 3 * L.Ep, 0, w_r, h, E, L.Ep, 3 * L.Ep, 1, 3 * L.Ep, rt, s)) return rc;
        rterm = rt;
        d_logits = nullptr;
    }
#define MOE_DB_LAUNCH(TY, KM)                                                                                   \
    dispatch_bwd_kernel<TY, KM><<<grid, 256, 0, s>>>(static_cast<const TY*>(d_buf), dest_row, d_logits,           \
        static_cast<const TY*>(ws), rterm, static_cast<const TY*>(dx_extra), T, h, k, E, static_cast<TY*>(dx));
    if (dtype == MOE_BF16) {
        if (d_logits) {
            wr_transpose_kernel<__nv_bfloat16><<<tgrid, tblock, 0, s>>>(static_cast<const __nv_bfloat16*>(w_r), h, E,
                                                                        static_cast<__nv_bfloat16*>(ws));
            if (int rc = check_launch("wr_transpose_kernel")) return rc;
        }
        if (k <= 2) { MOE_DB_LAUNCH(__nv_bfloat16, 2) }
        else if (k <= 8) { MOE_DB_LAUNCH(__nv_bfloat16, 8) }
        else { MOE_DB_LAUNCH(__nv_bfloat16, 32) }
    } else {
        if (d_logits) {
            wr_transpose_kernel<float><<<tgrid, tblock, 0, s>>>(static_cast<const float*>(w_r), h, E,
                                                                static_cast<float*>(ws));
            if (int rc = check_launch("wr_transpose_kernel")) return rc;
        }
        if (k <= 2) { MOE_DB_LAUNCH(float, 2) }
        else if (k <= 8) { MOE_DB_LAUNCH(float, 8) }
        else { MOE_DB_LAUNCH(float, 32) }
    }
#undef MOE_DB_LAUNCH
    return check_launch("dispatch_bwd_kernel");
}
