// Backward of the grouped SwiGLU expert FFN: C-ABI entry points, the weight-gradient operand transposes.
//
// "专家并行" (formulaic), section "BWD（反向传播）": each GPU first computes the gradients of its own experts'
// weights. The chain rule through the forward (ffn_tc.cu) with g = x W_gate^T, u = x W_up^T, a = silu(g) u:
//   d_act = d_eout W_down;  d_g = d_act u s (1 + g (1 - s)), d_u = d_act silu(g)  (s the logistic of g);
//   d_buf = d_g W_gate + d_u W_up;  dW_down = d_eout^T act;  dW_gate = d_g^T buf;  dW_up = d_u^T buf.
// All GEMMs run on the tcgen05 grouped kernels. The weight gradients contract over each expert's rows: those
// rows are transposed into K-major column segments, one per expert, each padded with zeros to a multiple of 64
// columns, so the GEMM's K loop of expert e covers exactly its rows.
#include <algorithm>
#include "ffn.cuh"

namespace moe {

constexpr int kSegAlign = 64;

// seg[0] = 0, seg[e + 1] = seg[e] + kept[e] rounded up to 64 (one warp, 32 experts per step).
__global__ void seg_offsets_kernel(const int32_t* __restrict__ kept, int E, int32_t* __restrict__ seg) {
    const int lane = threadIdx.x;
    int carry = 0;
    if (lane == 0) seg[0] = 0;
    for (int base = 0; base < E; base += 32) {
        const int e = base + lane;
        int v = e < E ? (kept[e] + kSegAlign - 1) / kSegAlign * kSegAlign : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += t;
        }
        if (e < E) seg[e + 1] = carry + v;
        carry += __shfl_sync(0xffffffffu, v, 31);
    }
}

// dst [C][ktot]: column k of expert e's segment [seg[e], seg[e+1]) holds row offsets[e] + (k - seg[e]) of
// src [rows][C] while k - seg[e] < kept[e], zero after it. bf16, C % 8 == 0. One 64 (k) x 64 (c) tile per block,
// 16-byte accesses on both sides: the tile is read as rows of 8 16-byte vectors and written as dst rows of 8
// 16-byte vectors (a warp stores four whole 128-byte lines). In shared memory element (k, c) sits in row k at
// 16-byte chunk (c / 8) ^ (k / 8): a store phase's eight vectors of one row land in distinct chunks, and the
// eight k-rows 8 apart that one column read touches land in distinct banks. A 64-column tile of dst lies in
// one expert's segment (segments are 64-aligned).
__global__ void __launch_bounds__(256)
segment_transpose_kernel(const __nv_bfloat16* __restrict__ src, int C, const int32_t* __restrict__ offsets,
                         const int32_t* __restrict__ kept, const int32_t* __restrict__ seg, int E, long long ktot,
                         __nv_bfloat16* __restrict__ dst) {
    __shared__ __align__(16) uint16_t tile[64 * 64];
    const int k0 = blockIdx.x * 64;
    if (k0 >= seg[E]) return;                 // the grid covers the largest possible ktot
    int lo = 0, hi = E - 1;                   // last e with seg[e] <= k0
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (seg[mid] <= k0) lo = mid; else hi = mid - 1;
    }
    const int e = lo, local0 = k0 - seg[e], n = kept[e], r0 = offsets[e];
    const int c0 = blockIdx.y * 64;
    const int t = threadIdx.x;
#pragma unroll
    for (int p = 0; p < 2; ++p) {             // 64 rows x 8 vectors
        const int k = (t >> 3) + 32 * p, v = t & 7, c = c0 + 8 * v;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (local0 + k < n && c < C) val = __ldcs(reinterpret_cast<const uint4*>(src + (size_t)(r0 + local0 + k) * C + c));
        *reinterpret_cast<uint4*>(tile + k * 64 + 8 * (v ^ (k >> 3))) = val;
    }
    __syncthreads();
#pragma unroll
    for (int p = 0; p < 2; ++p) {             // 64 dst rows (c) x 8 vectors of 8 k
        const int cc = (t >> 3) + 32 * p, w = t & 7;
        if (c0 + cc >= C) continue;
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            const int ka = 8 * w + j, kb = ka + 1;
            const uint32_t a = tile[ka * 64 + 8 * ((cc >> 3) ^ (ka >> 3)) + (cc & 7)];
            const uint32_t b = tile[kb * 64 + 8 * ((cc >> 3) ^ (kb >> 3)) + (cc & 7)];
            o[j >> 1] = a | (b << 16);
        }
        *reinterpret_cast<uint4*>(dst + (size_t)(c0 + cc) * ktot + k0 + 8 * w) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// d_gu from the saved pre-activations, over the live rows of the tile schedule: with g, u of feature f at
// columns (f / 128) 256 + f % 128 and that + 128 of gu [rows][2 Fp], s = logistic(g) and da = d_act[row][f]
// (0 for f >= F): d_g = da u s (1 + g (1 - s)), d_u = da g s, written to the same columns of d_gu. Work unit =
// (tile, 64 column vectors of 8 features); four rows of 64 vector lanes per block pass.
__global__ void __launch_bounds__(256)
swiglu_bwd_kernel(const __nv_bfloat16* __restrict__ gu, const __nv_bfloat16* __restrict__ d_act,
                  const int32_t* __restrict__ sched, int E, int F, int Fp, __nv_bfloat16* __restrict__ d_gu) {
    const int ntiles = sched[0];
    const int4* tiles = reinterpret_cast<const int4*>(sched + sched_tiles_offset(E));
    const int nv = Fp / 8, cch = (nv + 63) / 64;
    const long long units = (long long)ntiles * cch;
    const size_t ld = 2 * (size_t)Fp;
    for (long long w = blockIdx.x; w < units; w += gridDim.x) {
        const int m = (int)(w / cch), c = (int)(w - (long long)m * cch);
        const int4 t = tiles[m];
        const int v = c * 64 + (threadIdx.x & 63);
        if (v >= nv) continue;
        const int f = v * 8;
        const size_t col = (size_t)(f >> 7) * 256 + (f & 127);
        for (int r = t.y + (threadIdx.x >> 6); r < t.z; r += 4) {
            const Vec16<__nv_bfloat16> g = ld16(gu + (size_t)r * ld + col), u = ld16(gu + (size_t)r * ld + col + 128);
            Vec16<__nv_bfloat16> da;
            if (f < F) da = ld16(d_act + (size_t)r * F + f);
            else da.v = make_uint4(0, 0, 0, 0);
            Vec16<__nv_bfloat16> og, ou;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float gv = g.get(i), uv = u.get(i), a = da.get(i);
                const float sg = 1.f / (1.f + expf(-gv));
                og.set(i, a * uv * sg * (1.f + gv * (1.f - sg)));
                ou.set(i, a * gv * sg);
            }
            st16(d_gu + (size_t)r * ld + col, og);
            st16(d_gu + (size_t)r * ld + col + 128, ou);
        }
    }
}

// Column extent of the transposed operands: every expert's rows rounded up to 64, at most rows + 63 E.
static long long grads_ktot(int rows, int E) {
    return ((long long)rows + (long long)(kSegAlign - 1) * E + kSegAlign - 1) / kSegAlign * kSegAlign;
}

struct GradsWs { int32_t* seg; void* d_eout_t; void* act_t; void* d_gu_t; void* buf_t; long long ktot; size_t bytes; };

static GradsWs grads_ws_layout(void* ws, int E, int h, int F, int rows) {
    GradsWs w{};
    const int Fp = (F + 127) / 128 * 128;
    w.ktot = grads_ktot(rows, E);
    char* base = static_cast<char*>(ws);
    size_t off = 0;
    w.seg = reinterpret_cast<int32_t*>(base + off); off = align_up(off + (size_t)(E + 1) * 4, 256);
    w.d_eout_t = base + off; off = align_up(off + (size_t)h * w.ktot * 2, 256);
    w.act_t = base + off;    off = align_up(off + (size_t)F * w.ktot * 2, 256);
    w.d_gu_t = base + off;   off = align_up(off + (size_t)2 * Fp * w.ktot * 2, 256);
    w.buf_t = base + off;    off = align_up(off + (size_t)h * w.ktot * 2, 256);
    w.bytes = off;
    return w;
}

static int bwd_ffn_check(const char* fn, int E, int h, int F, int rows, int dtype) {
    MOE_REQUIRE(dtype == MOE_BF16, MOE_ERR_UNSUPPORTED, "%s: bf16 only (the tensor-core path)", fn);
    MOE_REQUIRE(E >= 1 && E <= 1024 && h > 0 && F > 0 && h % 8 == 0 && F % 8 == 0 && rows >= 0, MOE_ERR_INVALID_ARG,
                "%s: E=%d h=%d F=%d rows=%d (need h%%8==0, F%%8==0)", fn, E, h, F, rows);
    return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" int moe_expert_down_backward(const void* d_eout, const int32_t* tile_sched, const void* packed_bwd, int E,
                                        int h, int F, int rows, int dtype, void* d_act, void* stream) {
    if (int rc = bwd_ffn_check("moe_expert_down_backward", E, h, F, rows, dtype)) return rc;
    if (rows == 0) return MOE_OK;
    MOE_REQUIRE(d_eout && tile_sched && packed_bwd && d_act, MOE_ERR_INVALID_ARG, "moe_expert_down_backward: null pointer");
    MOE_REQUIRE(aligned16(d_eout) && aligned16(tile_sched) && aligned16(packed_bwd) && aligned16(d_act),
                MOE_ERR_INVALID_ARG, "moe_expert_down_backward: pointers must be 16-byte aligned");
    return ffn_tc_down_backward(d_eout, tile_sched, packed_bwd, E, h, F, rows, d_act, static_cast<cudaStream_t>(stream));
}

extern "C" int moe_expert_up_gate_backward(const void* buf, const void* d_act, const int32_t* tile_sched,
                                           const void* packed_w, const void* packed_bwd, int E, int h, int F, int rows,
                                           int dtype, void* d_gu, void* d_buf, void* stream) {
    if (int rc = bwd_ffn_check("moe_expert_up_gate_backward", E, h, F, rows, dtype)) return rc;
    if (rows == 0) return MOE_OK;
    MOE_REQUIRE(buf && d_act && tile_sched && packed_w && packed_bwd && d_gu && d_buf, MOE_ERR_INVALID_ARG,
                "moe_expert_up_gate_backward: null pointer");
    MOE_REQUIRE(aligned16(buf) && aligned16(d_act) && aligned16(tile_sched) && aligned16(packed_w) &&
                    aligned16(packed_bwd) && aligned16(d_gu) && aligned16(d_buf),
                MOE_ERR_INVALID_ARG, "moe_expert_up_gate_backward: pointers must be 16-byte aligned");
    return ffn_tc_up_gate_backward(buf, d_act, tile_sched, packed_w, packed_bwd, E, h, F, rows, d_gu, d_buf,
                                   static_cast<cudaStream_t>(stream));
}

extern "C" int moe_expert_up_gate_backward_saved(const void* gu, const void* d_act, const int32_t* tile_sched,
                                                 const void* packed_bwd, int E, int h, int F, int rows, int dtype,
                                                 void* d_gu, void* d_buf, void* stream) {
    if (int rc = bwd_ffn_check("moe_expert_up_gate_backward_saved", E, h, F, rows, dtype)) return rc;
    if (rows == 0) return MOE_OK;
    MOE_REQUIRE(gu && d_act && tile_sched && packed_bwd && d_gu && d_buf, MOE_ERR_INVALID_ARG,
                "moe_expert_up_gate_backward_saved: null pointer");
    MOE_REQUIRE(aligned16(gu) && aligned16(d_act) && aligned16(tile_sched) && aligned16(packed_bwd) && aligned16(d_gu) &&
                    aligned16(d_buf),
                MOE_ERR_INVALID_ARG, "moe_expert_up_gate_backward_saved: pointers must be 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int Fp = (F + 127) / 128 * 128;
    swiglu_bwd_kernel<<<4 * num_sms(), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(gu),
                                                    static_cast<const __nv_bfloat16*>(d_act), tile_sched, E, F, Fp,
                                                    static_cast<__nv_bfloat16*>(d_gu));
    if (int rc = check_launch("swiglu_bwd_kernel")) return rc;
    return ffn_tc_dbuf(d_gu, tile_sched, packed_bwd, E, h, F, rows, d_buf, s);
}

extern "C" size_t moe_expert_weight_grads_workspace_size(int E, int h, int F, int rows, int dtype) {
    if (E <= 0 || h <= 0 || F <= 0 || rows < 0 || dtype != MOE_BF16) return 0;
    return grads_ws_layout(nullptr, E, h, F, rows).bytes;
}

extern "C" int moe_expert_weight_grads(const void* buf, const void* act, const void* d_gu, const void* d_eout,
                                       const int32_t* offsets, const int32_t* kept_counts, int E, int h, int F, int rows,
                                       int dtype, float* dW_gate, float* dW_up, float* dW_down, void* ws,
                                       size_t ws_bytes, void* stream) {
    if (int rc = bwd_ffn_check("moe_expert_weight_grads", E, h, F, rows, dtype)) return rc;
    MOE_REQUIRE(offsets && kept_counts && dW_gate && dW_up && dW_down &&
                    (rows == 0 || (buf && act && d_gu && d_eout)),
                MOE_ERR_INVALID_ARG, "moe_expert_weight_grads: null pointer");
    MOE_REQUIRE(aligned16(dW_gate) && aligned16(dW_up) && aligned16(dW_down) && aligned16(ws) && aligned16(buf) &&
                    aligned16(act) && aligned16(d_gu) && aligned16(d_eout),
                MOE_ERR_INVALID_ARG, "moe_expert_weight_grads: pointers must be 16-byte aligned");
    const GradsWs w = grads_ws_layout(ws, E, h, F, rows);
    MOE_REQUIRE(ws && ws_bytes >= w.bytes, MOE_ERR_WORKSPACE, "moe_expert_weight_grads: workspace %zu < %zu", ws_bytes,
                w.bytes);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int Fp = (F + 127) / 128 * 128;
    seg_offsets_kernel<<<1, 32, 0, s>>>(kept_counts, E, w.seg);
    if (int rc = check_launch("seg_offsets_kernel")) return rc;
    using B = __nv_bfloat16;
    const int kt = (int)(w.ktot / 64);
    struct { const void* src; int C; void* dst; } tr[4] = {
        {d_eout, h, w.d_eout_t}, {act, F, w.act_t}, {d_gu, 2 * Fp, w.d_gu_t}, {buf, h, w.buf_t}};
    for (auto& t : tr) {
        segment_transpose_kernel<<<dim3(kt, cdiv(t.C, 64)), 256, 0, s>>>(
            static_cast<const B*>(t.src), t.C, offsets, kept_counts, w.seg, E, w.ktot, static_cast<B*>(t.dst));
        if (int rc = check_launch("segment_transpose_kernel")) return rc;
    }
    // dW_down[e] [h][F] = d_eout_e^T act_e ; dW_gate / dW_up [E][F][h] from d_gu_e^T buf_e (packed rows)
    if (int rc = ffn_tc_weight_grad(w.d_eout_t, w.act_t, w.ktot, w.seg, E, h, F, 0, F, dW_down, nullptr, s)) return rc;
    return ffn_tc_weight_grad(w.d_gu_t, w.buf_t, w.ktot, w.seg, E, 2 * Fp, h, 1, F, dW_gate, dW_up, s);
}
