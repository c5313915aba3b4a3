"""GB300-native weight-only quantized dequant-GEMV (INT8 per tensor and
outlier-aware INT4), a C-ABI CUDA library (libqz) with a thin Python API."""
from .api import (  # noqa: F401
    Int4oMatrix, Int8Matrix, Pager, QzError, check_perm, default_n_out,
    gemm_int4_outlier, gemm_int8, gemv_int4_outlier, gemv_int4_outlier_grouped,
    gemv_int8, gemv_int8_grouped, int4o_layout, quantize_int4_outlier,
    quantize_int8, saliency_accumulate, select_outliers)
