"""GB300-native paged (block) KV cache hot path.

``paged_kv_cache_slot_gb300.bkv`` binds libbkv.so (slot mapping, block
expansion, KV cache scatter, GQA paged decode); ``workloads`` draws the seeded
synthetic inputs; ``build`` compiles the CUDA sources for sm_103a.
"""
__version__ = "0.3.0"
