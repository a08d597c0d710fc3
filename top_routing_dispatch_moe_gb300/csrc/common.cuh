// Shared host/device helpers of the MoE library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/moe.h"

namespace moe {

// ------------------------------------------------------------------------------------------------
// host side: error reporting
// ------------------------------------------------------------------------------------------------
int set_error(int code, const char* fmt, ...);          // records the message, returns code
int check_launch(const char* what);                       // MOE_ERR_CUDA if the last launch failed
int check_launch(cudaError_t launch_result, const char* what);   // the same for a launch that returned a status
int num_sms();                                            // SM count of the current device (cached)
unsigned* device_error_word();                            // device address of the error word (current device)
// Unique id of the calling thread's current CUDA context (0: none, or the driver cannot tell). Per-device caches
// of device addresses and kernel attributes keep the id they were filled under and are filled again when it
// changes: after cudaDeviceReset a device gets a new primary context, in which the library's device variables
// may sit at other addresses and kernel attributes are unset.
unsigned long long context_id();
long long wait_limit();                                   // iteration limit of bounded device waits

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int cdiv(long long a, long long b) { return (int)((a + b - 1) / b); }

// Programmatic dependent launch: a kernel launched by launch_pdl may start while the previous kernel of its
// stream still runs (once every block of that kernel has called pdl_trigger, or exited); it must call pdl_wait
// before it reads anything the previous kernel writes (pdl_wait returns when that kernel has completed and its
// writes are visible). Both are no-ops for kernels launched without the attribute.
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
#endif
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

#define MOE_REQUIRE(cond, code, ...) \
    do { if (!(cond)) return ::moe::set_error((code), __VA_ARGS__); } while (0)

// Tile schedule layout (int32 words), written by dispatch, read by the expert FFN:
//   [0] number of MOE_TILE_M-row tiles, [1] E,
//   [2 .. 2+E]  tile_prefix: first tile index of each expert (E+1 words),
//   then, from word sched_tiles_offset(E) (16-byte aligned), 4 words per tile: {expert, row_begin,
//   row_end, 0}, ordered by expert then row.
constexpr int kSchedHeader = 2;
__host__ __device__ inline int sched_tiles_offset(int E) { return (kSchedHeader + E + 1 + 3) & ~3; }
inline size_t sched_max_tiles(long long rows, int E) { return (size_t)cdiv(rows, MOE_TILE_M) + (size_t)E; }
inline size_t sched_words(long long rows, int E) { return (size_t)sched_tiles_offset(E) + 4 * sched_max_tiles(rows, E); }

// ------------------------------------------------------------------------------------------------
// device side
// ------------------------------------------------------------------------------------------------
// Device error word (two unsigned: flags, site of the last error), one per device that loads the
// library; kernels that can give up receive its address and latch bit flags into it.
enum : unsigned { kDevErrTimeout = 1u, kDevErrBadIndex = 2u };

__device__ __forceinline__ void latch_device_error(unsigned* err, unsigned code, unsigned site) {
    atomicOr(err, code);
    atomicExch(err + 1, site);
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// 16-byte vector of elements: 8 bf16 or 4 fp32.
template <typename T> struct Vec16;
template <> struct Vec16<float> {
    static constexpr int N = 4;
    float4 v;
    __device__ __forceinline__ float get(int i) const { return (&v.x)[i]; }
    __device__ __forceinline__ void set(int i, float f) { (&v.x)[i] = f; }
};
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    uint4 v;
    __device__ __forceinline__ float get(int i) const {
        const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
        float2 f = __bfloat1622float2(p[i >> 1]);
        return (i & 1) ? f.y : f.x;
    }
    __device__ __forceinline__ void set(int i, float f) {
        reinterpret_cast<__nv_bfloat16*>(&v)[i] = __float2bfloat16_rn(f);
    }
};

template <typename T>
__device__ __forceinline__ Vec16<T> ld16(const T* p) {
    Vec16<T> r;
    if constexpr (sizeof(T) == 4) r.v = __ldg(reinterpret_cast<const float4*>(p));
    else r.v = __ldg(reinterpret_cast<const uint4*>(p));
    return r;
}
template <typename T>
__device__ __forceinline__ Vec16<T> ld16_stream(const T* p) {   // read-once data: do not keep in L1
    Vec16<T> r;
    if constexpr (sizeof(T) == 4) r.v = __ldcs(reinterpret_cast<const float4*>(p));
    else r.v = __ldcs(reinterpret_cast<const uint4*>(p));
    return r;
}
template <typename T>
__device__ __forceinline__ void st16(T* p, const Vec16<T>& r) {
    if constexpr (sizeof(T) == 4) *reinterpret_cast<float4*>(p) = r.v;
    else *reinterpret_cast<uint4*>(p) = r.v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
// Warp argmax over (value, index): larger value wins; equal values -> smaller index.
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, v, o);
        int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
    }
}

// Inclusive block scan of one int per thread (blockDim.x == 1024).
__device__ __forceinline__ int block_inclusive_scan(int v, int* s_tmp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) s_tmp[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = s_tmp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        s_tmp[lane] = w;
    }
    __syncthreads();
    if (warp > 0) v += s_tmp[warp - 1];
    __syncthreads();
    return v;
}

}  // namespace moe
