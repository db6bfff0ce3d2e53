"""GB300 (sm_103a) mixed-granularity E4M3 linear layer: 1×128 / 128×128
quantisers, the 1×128→128×1 requantise-transpose, RMSNorm+quant, and the
three block-scaled FP8 GEMMs, behind the C ABI of include/jetfp8.h."""
from . import jetfp8  # noqa: F401
from .jetfp8 import JetFP8Error, load_library  # noqa: F401
