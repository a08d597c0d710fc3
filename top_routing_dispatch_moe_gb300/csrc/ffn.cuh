// Grouped SwiGLU expert FFN: shared declarations.
#pragma once
#include "common.cuh"

namespace moe {

struct PackedLayout {
    int Fp;                 // F rounded up to 128
    size_t up_gate_off;     // bytes: [E][Fp/128][256][h]
    size_t down_off;        // bytes: [E][h][F]
    size_t total_bytes;
};

inline PackedLayout packed_layout(int E, int h, int F, int el) {
    PackedLayout L;
    L.Fp = (F + 127) / 128 * 128;
    L.up_gate_off = 0;
    L.down_off = align_up((size_t)E * 2 * L.Fp * h * el, 256);
    L.total_bytes = L.down_off + (size_t)E * h * F * el;
    return L;
}

// Backward packing: W_down^T [E][F][h], then W_gu^T [E][h][2Fp] (columns in the forward's packed order) from the
// next 256-byte boundary.
struct PackedBwdLayout {
    int Fp;
    size_t down_t_off;
    size_t gu_t_off;
    size_t total_bytes;
};

inline PackedBwdLayout packed_bwd_layout(int E, int h, int F, int el) {
    PackedBwdLayout L;
    L.Fp = (F + 127) / 128 * 128;
    L.down_t_off = 0;
    L.gu_t_off = align_up((size_t)E * F * h * el, 256);
    L.total_bytes = L.gu_t_off + (size_t)E * h * 2 * L.Fp * el;
    return L;
}

// CUDA-core path (fp32; the reference-precision path of the library).
int ffn_simt_up_gate(const void* buf, const int32_t* sched, const void* packed, int E, int h, int F, int rows, int dtype,
                     void* act, cudaStream_t s);
int ffn_simt_down(const void* act, const int32_t* sched, const void* packed, int E, int h, int F, int rows, int dtype,
                  void* eout, cudaStream_t s);

// tcgen05 tensor-core path (bf16 operands, fp32 accumulation in tensor memory). With T_sh > 0 the same launch
// also runs the shared expert (packed_sh, one expert) on its T_sh dense rows: x_sh -> act_sh, act_sh -> out_sh.
// gu / gu_sh (may be null): also store the pre-activations g and u of the routed / shared rows, [rows][2 Fp] in
// the packed gate/up column order (the layout of d_gu).
int ffn_tc_up_gate(const void* buf, const int32_t* sched, const void* packed, int E, int h, int F, int rows, void* act,
                   cudaStream_t s, const void* x_sh = nullptr, int T_sh = 0, const void* packed_sh = nullptr,
                   void* act_sh = nullptr, void* gu = nullptr, void* gu_sh = nullptr);
int ffn_tc_down(const void* act, const int32_t* sched, const void* packed, int E, int h, int F, int rows, void* eout,
                cudaStream_t s, const void* act_sh = nullptr, int T_sh = 0, const void* packed_sh = nullptr,
                void* out_sh = nullptr);

// The down GEMM with the combine fused into its epilogue: eout (and out_sh) as ffn_tc_down, plus
// y [T][h] = out_sh[t] (when T_sh > 0) + sum over kept j ascending of gates[t][j] eout[dest_row[t][j]], bit-identical
// to moe_combine. arrivals [T][cdiv(h, 256)] int32: zero on entry, zero again once the launch has completed.
int ffn_tc_down_combine(const void* act, const int32_t* sched, const void* packed, int E, int h, int F, int rows,
                        void* eout, cudaStream_t s, const void* act_sh, int T_sh, const void* packed_sh, void* out_sh,
                        const int32_t* src_token, const int32_t* dest_row, const float* gates, int T, int k, void* y,
                        int32_t* arrivals);

// Up/gate GEMM on the FP8 send buffer (e4m3 codes + per-row, per-128-column scales), dequantised in the prologue.
int ffn_tc_up_gate_fp8(const uint8_t* buf8, const float* scales, const int32_t* sched, const void* packed, int E, int h,
                       int F, int rows, void* act, cudaStream_t s);
// Backward on the tensor cores (bf16): down dgrad; up/gate recompute with the SwiGLU backward epilogue, then
// the up/gate dgrad; the experts' weight gradients from K-major transposed operands.
int ffn_tc_down_backward(const void* d_eout, const int32_t* sched, const void* packed_bwd, int E, int h, int F,
                         int rows, void* d_act, cudaStream_t s);
int ffn_tc_up_gate_backward(const void* buf, const void* d_act, const int32_t* sched, const void* packed,
                            const void* packed_bwd, int E, int h, int F, int rows, void* d_gu, void* d_buf,
                            cudaStream_t s);
// d_buf [rows][h] = d_gu [rows][2 Fp] times the packed gate/up weights (the second step of the up/gate backward).
int ffn_tc_dbuf(const void* d_gu, const int32_t* sched, const void* packed_bwd, int E, int h, int F, int rows,
                void* d_buf, cudaStream_t s);
int ffn_tc_weight_grad(const void* At, const void* Bt, long long ktot, const int32_t* seg, int E, int M, int N, int gu,
                       int F, float* out, float* out2, cudaStream_t s);

// Router logits on the tensor cores (bf16 x and transposed router weight, fp32 logits + bias).
int tc_router_logits(const void* x, const void* w_rT, const float* bias, int T, int h, int E, const int32_t* sched,
                     float* logits, cudaStream_t s);
// parts [S][M][N] fp32 (N % 4 == 0), part q = A[:, k in Q] B[:, k in Q]^T over the reduction indices
// Q = [q kchunk, min(K, (q + 1) kchunk)) (kchunk a multiple of 64, every part non-empty); A [M][a_cols] and
// B [N][b_cols] bf16 with contiguous columns (a_cols, b_cols multiples of 8; columns past them read as zero),
// reduction index k at column k mod a_kmod of A and k mod b_kmod of B (kmod 0: k itself; else a multiple of 64).
// The caller adds the parts (in order) when S > 1.
int tc_gemm_f32_splitk(const void* a, int M, int a_cols, int a_kmod, const void* b, int N, int b_cols, int b_kmod, int K,
                       int S, int kchunk, float* parts, cudaStream_t s);
// Split of an [M] x [N] x K product: S parts of kchunk columns so that the 128 x 256 output tiles of all parts
// cover about one per SM (S <= 16; S = 1 when the tiles alone fill the SMs).
void tc_splitk_plan(int M, int N, int K, int* S, int* kchunk);
// Dense tile schedule of `rows` rows (one group), launched on `s`.
int launch_dense_sched(int rows, int32_t* sched, cudaStream_t s);

}  // namespace moe
