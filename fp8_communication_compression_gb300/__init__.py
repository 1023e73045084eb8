"""GB300-native (sm_103a) FP8 communication compression.

TACO's fused ASH + DS FP8 block compressor for tensor-parallel intermediate
tensors, its inverse, the local reduce of the two-shot AllReduce, and AGoQ's
FP8 gradient accumulation and reduce, as a C-ABI library (libtaco.so,
include/taco.h) with a thin Python binding.
"""

from .api import (HostPipeline, TwoShotLocal, agoq_fp8_accumulate, agoq_laaq_dequantize,
                  agoq_laaq_quantize, agoq_reduce_shards, taco_compress,
                  taco_compress_int8, taco_decompress, taco_decompress_int8, taco_device_error,
                  taco_e4m3_encode, taco_reduce_decompress, taco_reduce_shards)

__all__ = ["taco_compress", "taco_decompress", "taco_compress_int8", "taco_decompress_int8", "taco_reduce_shards", "taco_reduce_decompress",
           "agoq_fp8_accumulate", "agoq_laaq_quantize", "agoq_laaq_dequantize",
           "agoq_reduce_shards", "taco_e4m3_encode", "taco_device_error", "TwoShotLocal", "HostPipeline"]
