"""GB300-native (sm_103a) EAGLE-2 dynamic draft-tree cycle.

The compute path is libeagle.so (hand-written CUDA behind the C ABI declared
in include/eagle.h). `speculative_decoding_dynamic_gb300.eagle` is the ctypes
binding (same names as the C entry points) and `.cycle` sequences one
draft-verify cycle on device buffers. Build with
`python -m speculative_decoding_dynamic_gb300.build`.
"""

__all__ = ["eagle", "cycle", "build"]
