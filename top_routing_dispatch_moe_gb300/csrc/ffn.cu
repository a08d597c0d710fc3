// C-ABI entry points of the grouped SwiGLU expert FFN ("Megatron-LM 分布式训练（六）", data flow: the
// experts run as one GroupedGEMM; "v6 长序列和 MoE", table row "expert": each expert's FFN h -> F -> h).
// bf16 goes to the tcgen05 tensor-core kernels, fp32 to the CUDA-core kernels.
#include "ffn.cuh"

using namespace moe;

static int ffn_check(const char* fn, const void* in, const int32_t* sched, const void* packed, int E, int h, int F,
                     int rows, int dtype, const void* out) {
    MOE_REQUIRE(dtype == MOE_F32 || dtype == MOE_BF16, MOE_ERR_UNSUPPORTED, "%s: dtype %d", fn, dtype);
    MOE_REQUIRE(E >= 1 && E <= 1024 && h > 0 && F > 0 && h % 8 == 0 && F % 8 == 0 && rows >= 0, MOE_ERR_INVALID_ARG,
                "%s: E=%d h=%d F=%d rows=%d (need h%%8==0, F%%8==0)", fn, E, h, F, rows);
    MOE_REQUIRE(rows == 0 || (in && sched && packed && out), MOE_ERR_INVALID_ARG, "%s: null pointer", fn);
    MOE_REQUIRE(aligned16(in) && aligned16(sched) && aligned16(packed) && aligned16(out), MOE_ERR_INVALID_ARG,
                "%s: pointers must be 16-byte aligned", fn);
    return MOE_OK;
}

extern "C" int moe_expert_up_gate(const void* buf, const int32_t* tile_sched, const void* packed_w, int E, int h, int F,
                                  int rows, int dtype, void* act, void* stream) {
    if (int rc = ffn_check("moe_expert_up_gate", buf, tile_sched, packed_w, E, h, F, rows, dtype, act)) return rc;
    if (rows == 0) return MOE_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == MOE_BF16) return ffn_tc_up_gate(buf, tile_sched, packed_w, E, h, F, rows, act, s);
    return ffn_simt_up_gate(buf, tile_sched, packed_w, E, h, F, rows, dtype, act, s);
}

extern "C" int moe_expert_down(const void* act, const int32_t* tile_sched, const void* packed_w, int E, int h, int F,
                               int rows, int dtype, void* eout, void* stream) {
    if (int rc = ffn_check("moe_expert_down", act, tile_sched, packed_w, E, h, F, rows, dtype, eout)) return rc;
    if (rows == 0) return MOE_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == MOE_BF16) return ffn_tc_down(act, tile_sched, packed_w, E, h, F, rows, eout, s);
    return ffn_simt_down(act, tile_sched, packed_w, E, h, F, rows, dtype, eout, s);
}

static int shared_check(const char* fn, const int32_t* sched, const void* in_sh, int T, const void* packed_sh,
                        const void* out_sh, int dtype) {
    MOE_REQUIRE(dtype == MOE_BF16, MOE_ERR_UNSUPPORTED, "%s: bf16 only (fp32: one call per group)", fn);
    MOE_REQUIRE(T >= 0, MOE_ERR_INVALID_ARG, "%s: T=%d", fn, T);
    MOE_REQUIRE(sched && (T == 0 || (in_sh && packed_sh && out_sh)), MOE_ERR_INVALID_ARG, "%s: null pointer", fn);
    MOE_REQUIRE(aligned16(in_sh) && aligned16(packed_sh) && aligned16(out_sh), MOE_ERR_INVALID_ARG,
                "%s: pointers must be 16-byte aligned", fn);
    return MOE_OK;
}

extern "C" int moe_expert_up_gate_shared(const void* buf, const int32_t* tile_sched, const void* packed_w, int E, int h,
                                         int F, int rows, const void* x, int T, const void* packed_shared,
                                         void* act_shared, int dtype, void* act, void* stream) {
    if (int rc = ffn_check("moe_expert_up_gate_shared", buf, tile_sched, packed_w, E, h, F, rows, dtype, act)) return rc;
    if (int rc = shared_check("moe_expert_up_gate_shared", tile_sched, x, T, packed_shared, act_shared, dtype)) return rc;
    if (rows == 0 && T == 0) return MOE_OK;
    return ffn_tc_up_gate(buf, tile_sched, packed_w, E, h, F, rows, act, static_cast<cudaStream_t>(stream), x, T,
                          packed_shared, act_shared);
}

extern "C" int moe_expert_up_gate_save(const void* buf, const int32_t* tile_sched, const void* packed_w, int E, int h,
                                       int F, int rows, const void* x, int T, const void* packed_shared,
                                       void* act_shared, void* gu_shared, int dtype, void* act, void* gu,
                                       void* stream) {
    if (int rc = ffn_check("moe_expert_up_gate_save", buf, tile_sched, packed_w, E, h, F, rows, dtype, act)) return rc;
    MOE_REQUIRE(dtype == MOE_BF16, MOE_ERR_UNSUPPORTED, "moe_expert_up_gate_save: bf16 only");
    MOE_REQUIRE((rows == 0 || gu) && aligned16(gu), MOE_ERR_INVALID_ARG,
                "moe_expert_up_gate_save: gu null or not 16-byte aligned");
    if (packed_shared) {
        if (int rc = shared_check("moe_expert_up_gate_save", tile_sched, x, T, packed_shared, act_shared, dtype))
            return rc;
        MOE_REQUIRE((T == 0 || gu_shared) && aligned16(gu_shared), MOE_ERR_INVALID_ARG,
                    "moe_expert_up_gate_save: gu_shared null or not 16-byte aligned");
    } else {
        T = 0;
    }
    if (rows == 0 && T == 0) return MOE_OK;
    return ffn_tc_up_gate(buf, tile_sched, packed_w, E, h, F, rows, act, static_cast<cudaStream_t>(stream),
                          T ? x : nullptr, T, T ? packed_shared : nullptr, T ? act_shared : nullptr, gu,
                          T ? gu_shared : nullptr);
}

extern "C" int moe_expert_down_shared(const void* act, const int32_t* tile_sched, const void* packed_w, int E, int h,
                                      int F, int rows, const void* act_shared, int T, const void* packed_shared,
                                      void* out_shared, int dtype, void* eout, void* stream) {
    if (int rc = ffn_check("moe_expert_down_shared", act, tile_sched, packed_w, E, h, F, rows, dtype, eout)) return rc;
    if (int rc = shared_check("moe_expert_down_shared", tile_sched, act_shared, T, packed_shared, out_shared, dtype))
        return rc;
    if (rows == 0 && T == 0) return MOE_OK;
    return ffn_tc_down(act, tile_sched, packed_w, E, h, F, rows, eout, static_cast<cudaStream_t>(stream), act_shared, T,
                       packed_shared, out_shared);
}

extern "C" size_t moe_combine_arrivals_bytes(int T, int h) {
    if (T < 0 || h <= 0) return 0;
    return align_up((size_t)T * cdiv(h, 256) * sizeof(int32_t), 256);
}

extern "C" int moe_expert_down_combine(const void* act, const int32_t* tile_sched, const void* packed_w, int E, int h,
                                       int F, int rows, const int32_t* src_token, const int32_t* dest_row,
                                       const float* gates, int T, int k, const void* act_shared,
                                       const void* packed_shared, int dtype, void* eout, void* out_shared, void* y,
                                       int32_t* arrivals, void* stream) {
    const char* fn = "moe_expert_down_combine";
    if (int rc = ffn_check(fn, act, tile_sched, packed_w, E, h, F, rows, dtype, eout)) return rc;
    MOE_REQUIRE(dtype == MOE_BF16, MOE_ERR_UNSUPPORTED, "%s: bf16 only (fp32: moe_expert_down, then moe_combine)", fn);
    MOE_REQUIRE(T >= 0 && k >= 1 && k <= 16 && k <= E, MOE_ERR_INVALID_ARG, "%s: T=%d k=%d E=%d", fn, T, k, E);
    const bool has_sh = act_shared != nullptr;
    MOE_REQUIRE(has_sh == (packed_shared != nullptr) && has_sh == (out_shared != nullptr), MOE_ERR_INVALID_ARG,
                "%s: act_shared, packed_shared and out_shared must be all NULL or all set", fn);
    if (has_sh) {
        if (int rc = shared_check(fn, tile_sched, act_shared, T, packed_shared, out_shared, dtype)) return rc;
    }
    MOE_REQUIRE(T == 0 || (dest_row && gates && y && arrivals), MOE_ERR_INVALID_ARG, "%s: null pointer", fn);
    MOE_REQUIRE(rows == 0 || src_token, MOE_ERR_INVALID_ARG, "%s: null src_token", fn);
    MOE_REQUIRE(aligned16(y), MOE_ERR_INVALID_ARG, "%s: y must be 16-byte aligned", fn);
    if (T == 0) return MOE_OK;                 // no token: nothing to combine, and no routed row either
    return ffn_tc_down_combine(act, tile_sched, packed_w, E, h, F, rows, eout, static_cast<cudaStream_t>(stream),
                               has_sh ? act_shared : nullptr, has_sh ? T : 0, packed_shared, out_shared, src_token,
                               dest_row, gates, T, k, y, arrivals);
}

extern "C" int moe_expert_up_gate_fp8(const uint8_t* buf8, const float* scales, const int32_t* tile_sched,
                                      const void* packed_w, int E, int h, int F, int rows, void* act, void* stream) {
    MOE_REQUIRE(E >= 1 && E <= 1024 && h > 0 && h % 128 == 0 && F > 0 && F % 8 == 0 && rows >= 0, MOE_ERR_INVALID_ARG,
                "moe_expert_up_gate_fp8: E=%d h=%d F=%d rows=%d (need h%%128==0, F%%8==0)", E, h, F, rows);
    if (rows == 0) return MOE_OK;
    MOE_REQUIRE(buf8 && scales && tile_sched && packed_w && act, MOE_ERR_INVALID_ARG, "moe_expert_up_gate_fp8: null pointer");
    MOE_REQUIRE(aligned16(buf8) && aligned16(tile_sched) && aligned16(packed_w) && aligned16(act), MOE_ERR_INVALID_ARG,
                "moe_expert_up_gate_fp8: pointers must be 16-byte aligned");
    return ffn_tc_up_gate_fp8(buf8, scales, tile_sched, packed_w, E, h, F, rows, act, static_cast<cudaStream_t>(stream));
}

extern "C" size_t moe_expert_ffn_workspace_size(int rows, int F, int dtype) {
    if (rows < 0 || F <= 0) return 0;
    return align_up((size_t)rows * F * (dtype == MOE_F32 ? 4 : 2), 256);
}

extern "C" int moe_expert_ffn(const void* buf, const int32_t* tile_sched, const void* packed_w, int E, int h, int F,
                              int rows, int dtype, void* eout, void* ws, size_t ws_bytes, void* stream) {
    if (int rc = ffn_check("moe_expert_ffn", buf, tile_sched, packed_w, E, h, F, rows, dtype, eout)) return rc;
    const size_t need = moe_expert_ffn_workspace_size(rows, F, dtype);
    MOE_REQUIRE(ws_bytes >= need && (need == 0 || ws), MOE_ERR_WORKSPACE, "moe_expert_ffn: workspace %zu < %zu",
                ws_bytes, need);
    MOE_REQUIRE(aligned16(ws), MOE_ERR_INVALID_ARG, "moe_expert_ffn: workspace must be 16-byte aligned");
    if (int rc = moe_expert_up_gate(buf, tile_sched, packed_w, E, h, F, rows, dtype, ws, stream)) return rc;
    return moe_expert_down(ws, tile_sched, packed_w, E, h, F, rows, dtype, eout, stream);
}
