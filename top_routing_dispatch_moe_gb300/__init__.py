"""GB300-native (sm_103a) MoE layer forward hot path: router -> dispatch -> grouped SwiGLU FFN -> combine.

The compute lives in the C-ABI library libmoe_gb300.so (include/moe.h); `moe` is its Python binding and
`layer.MoELayer` chains the four steps over preallocated device buffers. Build with `build.build()`.
"""
__all__ = ["moe", "layer", "build"]


def __getattr__(name):
    if name in ("moe", "layer", "build"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
