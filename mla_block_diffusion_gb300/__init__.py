"""GB300-native DSpark draft-and-verify step: libdspark (C ABI, sm_103a CUDA) and its Python binding."""
from .dspark import (DSpark, DSparkError, Geom, KV, Sample, GREEDY, PROBABILISTIC, BLOCK, FMT_BF16, FMT_FP8, FMT_NVFP4, FMT_MXFP4,
                     LIB_PATH, EXPORTS, lib, geom_struct)

__all__ = ["DSpark", "DSparkError", "Geom", "KV", "Sample", "GREEDY", "PROBABILISTIC", "BLOCK", "FMT_BF16", "FMT_FP8",
           "FMT_NVFP4", "FMT_MXFP4", "LIB_PATH", "EXPORTS", "lib", "geom_struct"]
