// placeholder: tcgen05 grouped GEMM (bf16) -- temporarily routed to the CUDA-core kernels
#include "ffn.cuh"
namespace moe {
int ffn_tc_up_gate(const void* buf, const int32_t* sched, const void* packed, int E, int h, int F, int rows, void* act,
                   cudaStream_t s) {
    return ffn_simt_up_gate(buf, sched, packed, E, h, F, rows, MOE_BF16, act, s);
}
int ffn_tc_down(const void* act, const int32_t* sched, const void* packed, int E, int h, int F, int rows, void* eout,
                cudaStream_t s) {
    return ffn_simt_down(act, sched, packed, E, h, F, rows, MOE_BF16, eout, s);
}
}  // namespace moe
