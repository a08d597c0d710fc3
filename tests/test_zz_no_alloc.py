"""moe_dispatch_static: the dispatch entry point for callers that cannot allocate device memory (a plugin
whose host framework owns all device memory, a latency-critical thread that may not allocate, a program
that reserves all of its memory at start-up). It keeps its scratch in a fixed 1 MiB array inside the
library instead of taking a workspace. This file is collected last so that a run that stops at the first
failure has run every other test before it."""
import ctypes

import pytest

OUT_KEYS = ["buf", "offsets", "kept_counts", "dest_row", "drop_mask", "src_token", "src_slot", "rank_counts",
            "rank_offsets", "tile_sched"]


def test_rejects_sizes_beyond_the_static_scratch():
    """Checked on the host before anything is enqueued (no GPU needed): T=300000 tokens with k=1 and E=1024
    needs 293 chunks x 1024 experts x 4 B > 1 MiB of scratch."""
    from top_routing_dispatch_moe_gb300 import build
    build.build()
    from top_routing_dispatch_moe_gb300 import moe
    raw = moe.raw_lib()
    ok = ctypes.c_void_p(0x1000)
    rc = raw.moe_dispatch_static(ok, ok, 300000, 64, 1024, 1, 0, 1, moe.MOE_BF16, *([ok] * 10), None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    assert "static" in moe.moe_last_error_string()


@pytest.mark.gpu
@pytest.mark.parametrize("T,h,E,k,C,R", [(4096, 512, 8, 2, 1280, 8), (2000, 256, 128, 8, 0, 8),
                                          (700, 512, 256, 8, 0, 8), (333, 128, 4, 2, 100, 2),
                                          (262144, 64, 1024, 1, 0, 8)])
def test_static_dispatch_matches_workspace_dispatch(T, h, E, k, C, R):
    """Two calls in a row with different inputs; each must equal moe_dispatch with a caller workspace
    (indices and the copied payload bit-exactly). The last size needs exactly the whole 1 MiB array (256 chunks of
    1024 assignments x 1024 experts x 4 bytes) and takes the separate count / scan / scatter / copy launches, whose
    scan rewrites the array's last words in place."""
    from top_routing_dispatch_moe_gb300 import moe as _m
    if T == 262144:
        assert _m.raw_lib().moe_dispatch_workspace_size(T, E, k, C) == 1 << 20
    import torch
    from top_routing_dispatch_moe_gb300 import moe
    dev = "cuda"
    for call in range(2):
        g = torch.Generator(device=dev).manual_seed(1000 * call + T)
        x = torch.randn(T, h, device=dev, generator=g).to(torch.bfloat16)
        w = (0.02 * torch.randn(h, E, device=dev, generator=g)).to(torch.bfloat16)
        r = moe.moe_router(x, w, None, k)
        ref = moe.moe_dispatch(x, r["ids"], E, C, R)
        got = moe.moe_dispatch_static(x, r["ids"], E, C, R)
        torch.cuda.synchronize()
        assert moe.moe_check_device_error() == moe.MOE_OK, moe.moe_last_error_string()
        for key in OUT_KEYS:
            a, b = got[key], ref[key]
            if key == "tile_sched":   # defined words: header + prefix, then the tile list (the pad between
                off = (2 + E + 1 + 3) & ~3   # them and the words past the last tile are not part of the output)
                n = int(b[0].item())
                a = torch.cat([a[:2 + E + 1], a[off:off + 4 * n]])
                b = torch.cat([b[:2 + E + 1], b[off:off + 4 * n]])
            if a.dtype == torch.bfloat16:
                a, b = a.view(torch.int16), b.view(torch.int16)
            assert torch.equal(a, b), f"call {call}: {key} differs"
