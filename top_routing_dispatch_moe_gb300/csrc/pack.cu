// One-time repack of the SwiGLU expert weights for the grouped GEMM.
//
// "v6 长序列和 MoE", section "MoE": a SwiGLU FFN holds three h x F matrices (gate, up, down).
//
// Packed layout (elements of the working dtype):
//   region 1, up/gate operand, [E][Fp/128][256][h] with Fp = F rounded up to 128: block b of expert e
//     holds gate rows f = 128 b .. 128 b + 127 in its first 128 rows and the up rows of the same f in the
//     next 128 (rows with f >= F are zero). One 256-wide GEMM tile therefore produces the gate and the up
//     projection of the same 128 columns of F, and its epilogue applies silu(g) * u without another pass.
//   region 2, down operand, [E][h][F]: W_down as given (K-major for the second GEMM), starting at the
//     first 256-byte boundary after region 1.
#include "common.cuh"
#include "ffn.cuh"

namespace moe {

template <typename T>
__global__ void pack_kernel(const T* __restrict__ wg, const T* __restrict__ wu, const T* __restrict__ wd, int E, int h,
                            int F, int Fp, T* __restrict__ up_gate, T* __restrict__ down) {
    constexpr int V = Vec16<T>::N;
    const long long vec_per_row = h / V;
    const long long n1 = (long long)E * 2 * Fp * vec_per_row;
    const long long n2 = (long long)E * h * (F / V);
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n1; i += stride) {
        const long long row = i / vec_per_row;
        const int c = (int)(i - row * vec_per_row) * V;
        const int e = (int)(row / (2 * Fp));
        const int rr = (int)(row - (long long)e * 2 * Fp);
        const int blk = rr / 256, w = rr % 256;
        const int f = blk * 128 + (w & 127);
        Vec16<T> v;
        v.v = {};
        if (f < F) {
            const T* src = (w < 128 ? wg : wu) + ((long long)e * F + f) * h + c;
            v = ld16(src);
        }
        st16(up_gate + row * h + c, v);
    }
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n2; i += stride)
        st16(down + i * V, ld16(wd + i * V));
}

// Backward packing (the dgrad GEMMs' K-major weight operands):
//   region 1, [E][F][h]: W_down^T (row f of expert e = column f of W_down[e]); d_act = d_eout W_down reads it.
//   region 2, [E][h][2Fp]: W_gu^T with its 2Fp columns in the forward's packed order (128 gate columns, then
//     the up columns of the same f, block after block; f >= F zero); d_buf = d_gu W_gu reads it, d_gu being
//     written in the same packed column order by the SwiGLU backward epilogue.
// Both are 32 x 32 tiled transposes through shared memory; blockIdx.z is the expert.
template <typename T>
__global__ void __launch_bounds__(256)
pack_down_t_kernel(const T* __restrict__ wd, int h, int F, T* __restrict__ out) {
    __shared__ T tile[32][33];
    const int e = blockIdx.z, d0 = blockIdx.x * 32, f0 = blockIdx.y * 32;
    const T* src = wd + (size_t)e * h * F;                 // [h][F]
    T* dst = out + (size_t)e * F * h;                      // [F][h]
    for (int r = threadIdx.y; r < 32; r += 8) {
        const int d = d0 + r, f = f0 + threadIdx.x;
        if (d < h && f < F) tile[r][threadIdx.x] = src[(size_t)d * F + f];
    }
    __syncthreads();
    for (int r = threadIdx.y; r < 32; r += 8) {
        const int f = f0 + r, d = d0 + threadIdx.x;
        if (f < F && d < h) dst[(size_t)f * h + d] = tile[threadIdx.x][r];
    }
}

template <typename T>
__global__ void __launch_bounds__(256)
pack_gu_t_kernel(const T* __restrict__ wg, const T* __restrict__ wu, int h, int F, int Fp, T* __restrict__ out) {
    __shared__ T tile[32][33];
    const int e = blockIdx.z, d0 = blockIdx.x * 32, p0 = blockIdx.y * 32;       // p: packed column in [0, 2Fp)
    const int blk = p0 / 256, w0 = p0 % 256;                                     // a 32-column tile never straddles
    const T* src = (w0 < 128 ? wg : wu) + (size_t)e * F * h;                     // [F][h]
    const int fb = blk * 128 + (w0 & 127);
    T* dst = out + (size_t)e * h * 2 * Fp;                                        // [h][2Fp]
    for (int r = threadIdx.y; r < 32; r += 8) {                                  // r: f offset, x: d offset
        const int f = fb + r, d = d0 + threadIdx.x;
        tile[r][threadIdx.x] = (f < F && d < h) ? src[(size_t)f * h + d] : T(0.f);
    }
    __syncthreads();
    for (int r = threadIdx.y; r < 32; r += 8) {
        const int d = d0 + r;
        if (d < h) dst[(size_t)d * 2 * Fp + p0 + threadIdx.x] = tile[threadIdx.x][r];
    }
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_packed_weights_bytes(int E, int h, int F, int dtype) {
    if (E <= 0 || h <= 0 || F <= 0) return 0;
    const PackedLayout L = packed_layout(E, h, F, dtype == MOE_F32 ? 4 : 2);
    return L.total_bytes;
}

extern "C" int moe_pack_expert_weights(const void* w_gate, const void* w_up, const void* w_down, int E, int h, int F,
                                       int dtype, void* packed, void* stream) {
    MOE_REQUIRE(dtype == MOE_F32 || dtype == MOE_BF16, MOE_ERR_UNSUPPORTED, "moe_pack_expert_weights: dtype %d", dtype);
    MOE_REQUIRE(E >= 1 && h > 0 && F > 0 && h % 8 == 0 && F % 8 == 0, MOE_ERR_INVALID_ARG,
                "moe_pack_expert_weights: E=%d h=%d F=%d (need h%%8==0, F%%8==0)", E, h, F);
    MOE_REQUIRE(w_gate && w_up && w_down && packed, MOE_ERR_INVALID_ARG, "moe_pack_expert_weights: null pointer");
    MOE_REQUIRE(aligned16(w_gate) && aligned16(w_up) && aligned16(w_down) && aligned16(packed), MOE_ERR_INVALID_ARG,
                "moe_pack_expert_weights: pointers must be 16-byte aligned");
    const int el = dtype == MOE_F32 ? 4 : 2;
    const PackedLayout L = packed_layout(E, h, F, el);
    char* base = static_cast<char*>(packed);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int grid = 4 * num_sms();
    if (dtype == MOE_BF16)
        pack_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(w_gate),
            static_cast<const __nv_bfloat16*>(w_up), static_cast<const __nv_bfloat16*>(w_down), E, h, F, L.Fp,
            reinterpret_cast<__nv_bfloat16*>(base + L.up_gate_off), reinterpret_cast<__nv_bfloat16*>(base + L.down_off));
    else
        pack_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(w_gate), static_cast<const float*>(w_up),
            static_cast<const float*>(w_down), E, h, F, L.Fp, reinterpret_cast<float*>(base + L.up_gate_off),
            reinterpret_cast<float*>(base + L.down_off));
    return check_launch("pack_kernel");
}

extern "C" size_t moe_packed_weights_backward_bytes(int E, int h, int F, int dtype) {
    if (E <= 0 || h <= 0 || F <= 0) return 0;
    const PackedBwdLayout L = packed_bwd_layout(E, h, F, dtype == MOE_F32 ? 4 : 2);
    return L.total_bytes;
}

extern "C" int moe_pack_expert_weights_backward(const void* w_gate, const void* w_up, const void* w_down, int E, int h,
                                                int F, int dtype, void* packed_bwd, void* stream) {
    MOE_REQUIRE(dtype == MOE_F32 || dtype == MOE_BF16, MOE_ERR_UNSUPPORTED, "moe_pack_expert_weights_backward: dtype %d",
                dtype);
    MOE_REQUIRE(E >= 1 && E <= 65535 && h > 0 && F > 0 && h % 8 == 0 && F % 8 == 0, MOE_ERR_INVALID_ARG,
                "moe_pack_expert_weights_backward: E=%d h=%d F=%d (need h%%8==0, F%%8==0)", E, h, F);
    MOE_REQUIRE(w_gate && w_up && w_down && packed_bwd, MOE_ERR_INVALID_ARG,
                "moe_pack_expert_weights_backward: null pointer");
    MOE_REQUIRE(aligned16(packed_bwd), MOE_ERR_INVALID_ARG, "moe_pack_expert_weights_backward: packed_bwd alignment");
    const int el = dtype == MOE_F32 ? 4 : 2;
    const PackedBwdLayout L = packed_bwd_layout(E, h, F, el);
    char* base = static_cast<char*>(packed_bwd);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const dim3 block(32, 8), gd(cdiv(h, 32), cdiv(F, 32), E), gg(cdiv(h, 32), 2 * L.Fp / 32, E);
    if (dtype == MOE_BF16) {
        using B = __nv_bfloat16;
        pack_down_t_kernel<B><<<gd, block, 0, s>>>(static_cast<const B*>(w_down), h, F,
                                                   reinterpret_cast<B*>(base + L.down_t_off));
        if (int rc = check_launch("pack_down_t_kernel")) return rc;
        pack_gu_t_kernel<B><<<gg, block, 0, s>>>(static_cast<const B*>(w_gate), static_cast<const B*>(w_up), h, F, L.Fp,
                                                 reinterpret_cast<B*>(base + L.gu_t_off));
    } else {
        pack_down_t_kernel<float><<<gd, block, 0, s>>>(static_cast<const float*>(w_down), h, F,
                                                       reinterpret_cast<float*>(base + L.down_t_off));
        if (int rc = check_launch("pack_down_t_kernel")) return rc;
        pack_gu_t_kernel<float><<<gg, block, 0, s>>>(static_cast<const float*>(w_gate), static_cast<const float*>(w_up),
                                                     h, F, L.Fp, reinterpret_cast<float*>(base + L.gu_t_off));
    }
    return check_launch("pack_gu_t_kernel");
}
