"""GB300-native engine for the data-parallel hot path of agentic KV-cache engineering.

    build     compile libakv.so for sm_103a (``python -m agentic_kv_cache_gb300.build``)
    akv       ctypes binding of the C ABI in include/akv.h (Engine, make_pools, ...)
    synth     seeded synthetic workloads shared by tests and benchmarks
    runner    drives a synthetic workload through the engine

The binding is imported lazily so that ``synth`` can be used without the library.
"""
