"""rate_adaptive_kv_block_b300 -- write-time quantization of the KV cache with a
rate-adaptive, entropy-constrained unbiased scalar quantizer applied per cache
block, on B300 (sm_103a) CUDA kernels behind a C ABI (include/kvq.h).

The CUDA library is loaded on first use; there is no CPU fallback.
"""
__all__ = ["kvq", "synth"]
