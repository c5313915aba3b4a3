"""GB300-native weight-only quantized dequant-GEMV (INT8 per tensor and
outlier-aware INT4), a C-ABI CUDA library (libqz) with a thin Python API."""
from .api import *  # noqa: F401,F403
from .api import Int4oMatrix, Int8Matrix, Pager, QzError  # noqa: F401
