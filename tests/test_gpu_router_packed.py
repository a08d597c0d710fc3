"""moe_router_packed (the router on a weight repacked once by moe_pack_router_weight) against moe_router on
the plain weight: every output bitwise equal, on every path the router takes (small-E fused kernels in bf16
and fp32, the tensor-core logits GEMM with and without the K split, the CUDA-core GEMM for E % 4 != 0), and the
packed bf16 weight equal to the transpose of w_r."""
import pytest

pytestmark = pytest.mark.gpu

SHAPES = [  # T, h, E, k, dtype
    (1000, 512, 8, 2, "bf16"),       # fused mma.sync kernel, one 8-expert block
    (777, 264, 24, 4, "bf16"),       # fused mma.sync kernel, E not a multiple of 8, h not a multiple of 32
    (300, 128, 4, 2, "f32"),         # fused fp32 kernel
    (4096, 1024, 256, 8, "bf16"),    # tensor-core logits, split over K
    (16384, 256, 128, 8, "bf16"),    # tensor-core logits, one part
    (500, 256, 66, 3, "bf16"),       # CUDA-core logits GEMM (E % 4 != 0) on the transposed weight
    (300, 64, 40, 2, "f32"),         # CUDA-core logits GEMM, fp32
]


@pytest.mark.parametrize("T,h,E,k,dt", SHAPES)
@pytest.mark.parametrize("gating", ["softmax", "sigmoid_bias_renorm"])
def test_packed_router_bitwise(T, h, E, k, dt, gating):
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    dtype = torch.bfloat16 if dt == "bf16" else torch.float32
    g = torch.Generator(device="cuda").manual_seed(T + E)
    x = torch.randn(T, h, device="cuda", generator=g).to(dtype)
    w = (0.02 * torch.randn(h, E, device="cuda", generator=g)).to(dtype)
    b = 0.1 * torch.randn(E, device="cuda", generator=g)
    packed = moe.moe_pack_router_weight(w)
    a = moe.moe_router(x, w, b, k, gating)
    p = moe.moe_router(x, w, b, k, gating, w_packed=packed)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
    if dt == "bf16":
        got = packed[:E * h * 2].view(torch.bfloat16).view(E, h)
        assert torch.equal(got.view(torch.int16), w.t().contiguous().view(torch.int16))
    for key in ["logits", "ids", "gates", "counts", "f", "P", "aux"]:
        assert torch.equal(a[key], p[key]), key
