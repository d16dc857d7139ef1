"""decode_attention_kv_softmax_b300: single-token decode attention over a KV
cache on B300 (sm_103a).

The compute lives in ``libkvdec.so`` (hand-written CUDA, C ABI in
``include/kvdec.h``); ``kvdec`` is its Python binding.  Nothing here falls
back to a CPU or PyTorch implementation.
"""
from . import kvdec  # noqa: F401  (the .so is loaded on first use)

__all__ = ["kvdec"]
