"""BeaconKV eviction step on NVIDIA B300 (sm_103a).

``kv_cache_eviction_04_b300.bkv`` is the binding of the C ABI (libbkv.so,
include/bkv.h); ``kv_cache_eviction_04_b300.workload`` makes seeded synthetic
inputs.  The binding is imported on demand so that the workload generator can
be used on machines without the compiled library.
"""
__all__ = ["bkv", "workload", "build"]
