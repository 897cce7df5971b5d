"""GB300-native ZeRO sharded-optimizer step.

One ZeRO step over N simulated data-parallel ranks whose buffers all live in a
single GPU's HBM: reduce-scatter-mean of the N gradients, AdamW on each shard,
all-gather into every replica -- fused into one CUDA kernel for sm_103a behind
the C-ABI library ``libzero_gb300.so`` (declared in ``include/zero_gb300.h``).

``zero_sharded_optimizer_gb300.abi`` is the thin binding over that library; it
raises at import when the library has not been built.
"""

__all__ = ["abi", "inputs", "optimizer"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
