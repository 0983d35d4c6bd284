"""GB300-native mixed-precision SparseGemv: y = W_hat . x with W_hat an N:4
pruned (2:4 / 1:4), INT4 group-quantised weight in 2bit-CSR form, x and y
in binary16, fp32 accumulation (Dong et al., "Efficient LLM ad generation
via model compression and parallel verification", arXiv 2605.11582,
sections 1 and 3.2-3.3).

The compute path is the CUDA library libsgemv.so (include/sgemv.h); this
package is a thin ctypes binding over it.
"""
from ._native import (SGEMV_ERR_ARG, SGEMV_ERR_CUDA, SGEMV_ERR_NONFINITE,
                      SGEMV_ERR_RANGE, SGEMV_ERR_STATE, SGEMV_ERR_TIMEOUT,
                      SGEMV_ERR_UNSUPPORTED, SGEMV_MAX_M, SGEMV_OK, SIGNATURES,
                      SgemvError, SparseGemv, load, LIB_PATH, run_group, run_group_host)

__all__ = ["SparseGemv", "SgemvError", "load", "LIB_PATH", "SIGNATURES", "run_group", "run_group_host",
           "SGEMV_OK", "SGEMV_ERR_ARG", "SGEMV_ERR_UNSUPPORTED",
           "SGEMV_ERR_CUDA", "SGEMV_ERR_STATE", "SGEMV_ERR_TIMEOUT",
           "SGEMV_ERR_NONFINITE", "SGEMV_ERR_RANGE", "SGEMV_MAX_M"]


def build(force: bool = False) -> str:
    from .build import build as _build
    return _build(force=force)
