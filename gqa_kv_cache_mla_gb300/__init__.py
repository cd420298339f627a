"""GB300-native fused per-token KV-cache write library.

``gqa_kv_cache_mla_gb300.kvw``        binding of the C ABI (``include/kvw.h``)
``gqa_kv_cache_mla_gb300.workloads``  seeded synthetic inputs
``gqa_kv_cache_mla_gb300.device``     upload of those inputs to a CUDA device
``gqa_kv_cache_mla_gb300.build``      in-tree nvcc build of ``libkvw.so``
"""
