"""B300-native SepLLM attention: index build, Sep-Attention forward and
backward, and the streaming four-block KV cache, all in hand-written sm_103a
CUDA behind the C ABI declared in ``include/sepattn.h``.

Importing this package loads nothing; ``separator_token_kv_sep_b300.api``
loads the shared library and raises if it is missing.
"""

__all__ = ["api", "synth"]
