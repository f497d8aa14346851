"""GB300-native (sm_103a) LRMoE backward recalibration of an MoE layer's FC2.

The compute lives in liblrm.so (C ABI in include/lrm.h); ``lrm`` is its
ctypes binding and ``pipeline`` enqueues the whole path on one stream.
Importing this package does not load the library; the first call does.
"""

__all__ = ["lrm", "pipeline", "build"]
