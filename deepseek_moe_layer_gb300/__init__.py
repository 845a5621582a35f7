"""DeepSeek-style MoE FFN forward on one GB300 (sm_103a).

The layer runs as hand-written CUDA kernels behind the C ABI in ``include/moe_gb300.h``
(library ``_build/libmoe_gb300.so``, built by ``deepseek_moe_layer_gb300.build``).
``deepseek_moe_layer_gb300.binding`` exposes the same calls on torch tensors;
``deepseek_moe_layer_gb300.inputs`` draws the seeded synthetic workloads.
"""

__all__ = ["binding", "build", "inputs"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
