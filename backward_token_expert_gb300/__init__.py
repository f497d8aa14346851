"""GB300-native (sm_103a) LRMoE backward recalibration of an MoE layer's FC2.

The compute lives in liblrm.so (C ABI in include/lrm.h); ``lrm`` is its
ctypes binding, ``pipeline`` enqueues the whole path on one stream (and
captures it as a CUDA graph or runs it on host buffers), ``replicas`` holds
the multi-rank totals and ``build`` compiles the library.  Importing this
package does not load the library; the first call does.
"""

__all__ = ["lrm", "pipeline", "replicas", "build"]
