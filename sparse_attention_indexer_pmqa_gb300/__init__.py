"""GB300-native FP8 paged MQA-logits indexer with per-row top-k.

The computation lives in libpmqa.so (hand-written sm_103a CUDA behind the C ABI
of include/pmqa.h); ``pmqa`` is its ctypes binding and ``build`` compiles it.
"""

from . import build  # noqa: F401
