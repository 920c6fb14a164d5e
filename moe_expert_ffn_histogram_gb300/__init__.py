"""GB300 (sm_103a) routed mixture-of-experts FFN: C-ABI CUDA library + thin Python binding.

``moe_expert_ffn_histogram_gb300.capi`` loads the in-tree ``libmoe_ffn_gb300.so`` and exposes
the entry points declared in ``include/moe_ffn.h``; ``inputs`` builds seeded synthetic workloads.
The library is loaded lazily by ``capi`` so that the input generators import without a GPU.
"""
__all__ = ["capi", "inputs"]
