"""GB300-native sparse x dense products: CSR SpMV (and the A v / A^T u pair),
CSR SpMM and tensor-core BSR SpMM behind the C ABI of libspx.so.

The compute path is the CUDA library; ``spx`` is its ctypes binding.
"""
from . import spx  # noqa: F401
from .spx import (Csr, Plan, SpxError, launch_count, spx_build_bsr, spx_build_csr, spx_check_csr,  # noqa: F401
                  spx_last_device_error, spx_plan_csr, spx_plan_opts_default, spx_row_stats, spx_spmm_bsr,
                  spx_spmm_csr, spx_spmm_csr_bf16, spx_spmm_csr_f16, spx_spmm_csr_planned, spx_spmm_csr_variant, spx_spmv_coo, spx_spmv_csr,
                  spx_spmv_csr_dual, spx_spmv_csr_noalloc, spx_plan_autotune, Sell, spx_spmv_sell, spx_transpose_csr)
