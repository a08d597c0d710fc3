// Grouped SwiGLU expert FFN on the CUDA cores (fp32 operands, fp32 accumulation).
//
// The fp32 path of the library: the tcgen05 tensor cores have no full-fp32 input kind (tf32 rounds the
// operands to 10 mantissa bits), so an fp32 layer is computed with FFMA. Classic shared-memory tiling:
// 64 x 64 output tiles, 16-deep K steps, 4 x 4 outputs per thread. Row ranges come from the device tile
// schedule (two 64-row halves per 128-row schedule tile); blocks past the schedule's tile count exit.
#include <math.h>
#include "ffn.cuh"

namespace moe {

template <typename T>
__global__ void __launch_bounds__(256)
ffn_simt_up_gate_kernel(const T* __restrict__ buf, const int32_t* __restrict__ sched, const T* __restrict__ wug, int h,
                        int F, int Fp, T* __restrict__ act) {
    __shared__ float As[16][64 + 4];
    __shared__ float Gs[16][64 + 4];
    __shared__ float Us[16][64 + 4];
    const int ntiles = sched[0], E = sched[1];
    const int tile = blockIdx.y >> 1;
    if (tile >= ntiles) return;
    const int4 ent = reinterpret_cast<const int4*>(sched + sched_tiles_offset(E))[tile];
    const int e = ent.x, r0 = ent.y + (blockIdx.y & 1) * 64, r1 = ent.z;
    if (r0 >= r1) return;
    const int f0 = blockIdx.x * 64;
    const T* Wg = wug + ((size_t)e * 2 * Fp + (size_t)(f0 / 128) * 256 + (f0 % 128)) * h;
    const T* Wu = Wg + (size_t)128 * h;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float ag[4][4] = {}, au[4][4] = {};
    for (int k0 = 0; k0 < h; k0 += 16) {
        for (int i = threadIdx.x; i < 64 * 16; i += 256) {
            const int r = i >> 4, c = i & 15, kk = k0 + c;
            const int row = r0 + r;
            As[c][r] = (row < r1 && kk < h) ? to_f32(buf[(size_t)row * h + kk]) : 0.f;
            Gs[c][r] = kk < h ? to_f32(Wg[(size_t)r * h + kk]) : 0.f;
            Us[c][r] = kk < h ? to_f32(Wu[(size_t)r * h + kk]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a[4], g[4], u[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) { a[i] = As[kk][ty * 4 + i]; g[i] = Gs[kk][tx * 4 + i]; u[i] = Us[kk][tx * 4 + i]; }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) { ag[i][j] = fmaf(a[i], g[j], ag[i][j]); au[i][j] = fmaf(a[i], u[j], au[i][j]); }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = r0 + ty * 4 + i;
        if (row >= r1) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int f = f0 + tx * 4 + j;
            if (f < F) {
                const float g = ag[i][j];
                act[(size_t)row * F + f] = from_f32<T>(g / (1.f + expf(-g)) * au[i][j]);
            }
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(256)
ffn_simt_down_kernel(const T* __restrict__ act, const int32_t* __restrict__ sched, const T* __restrict__ wd, int h, int F,
                     T* __restrict__ eout) {
    __shared__ float As[16][64 + 4];
    __shared__ float Bs[16][64 + 4];
    const int ntiles = sched[0], E = sched[1];
    const int tile = blockIdx.y >> 1;
    if (tile >= ntiles) return;
    const int4 ent = reinterpret_cast<const int4*>(sched + sched_tiles_offset(E))[tile];
    const int e = ent.x, r0 = ent.y + (blockIdx.y & 1) * 64, r1 = ent.z;
    if (r0 >= r1) return;
    const int n0 = blockIdx.x * 64;
    const T* W = wd + (size_t)e * h * F;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < F; k0 += 16) {
        for (int i = threadIdx.x; i < 64 * 16; i += 256) {
            const int r = i >> 4, c = i & 15, kk = k0 + c;
            const int row = r0 + r, n = n0 + r;
            As[c][r] = (row < r1 && kk < F) ? to_f32(act[(size_t)row * F + kk]) : 0.f;
            Bs[c][r] = (n < h && kk < F) ? to_f32(W[(size_t)n * F + kk]) : 0.f;
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
        const int row = r0 + ty * 4 + i;
        if (row >= r1) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n < h) eout[(size_t)row * h + n] = from_f32<T>(acc[i][j]);
        }
    }
}

int ffn_simt_up_gate(const void* buf, const int32_t* sched, const void* packed, int E, int h, int F, int rows, int dtype,
                     void* act, cudaStream_t s) {
    const int el = dtype == MOE_F32 ? 4 : 2;
    const PackedLayout L = packed_layout(E, h, F, el);
    dim3 grid(cdiv(F, 64), 2 * (unsigned)sched_max_tiles(rows, E));
    const char* p = static_cast<const char*>(packed) + L.up_gate_off;
    if (dtype == MOE_F32)
        ffn_simt_up_gate_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(buf), sched,
            reinterpret_cast<const float*>(p), h, F, L.Fp, static_cast<float*>(act));
    else
        ffn_simt_up_gate_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(buf), sched,
            reinterpret_cast<const __nv_bfloat16*>(p), h, F, L.Fp, static_cast<__nv_bfloat16*>(act));
    return check_launch("ffn_simt_up_gate_kernel");
}

int ffn_simt_down(const void* act, const int32_t* sched, const void* packed, int E, int h, int F, int rows, int dtype,
                  void* eout, cudaStream_t s) {
    const int el = dtype == MOE_F32 ? 4 : 2;
    const PackedLayout L = packed_layout(E, h, F, el);
    dim3 grid(cdiv(h, 64), 2 * (unsigned)sched_max_tiles(rows, E));
    const char* p = static_cast<const char*>(packed) + L.down_off;
    if (dtype == MOE_F32)
        ffn_simt_down_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(act), sched,
            reinterpret_cast<const float*>(p), h, F, static_cast<float*>(eout));
    else
        ffn_simt_down_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(act), sched,
            reinterpret_cast<const __nv_bfloat16*>(p), h, F, static_cast<__nv_bfloat16*>(eout));
    return check_launch("ffn_simt_down_kernel");
}

}  // namespace moe
