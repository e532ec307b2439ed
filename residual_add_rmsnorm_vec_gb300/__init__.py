"""GB300 (sm_103a) fused residual-add + RMSNorm.

The compute runs in the hand-written CUDA kernels of ``csrc/`` behind the C
ABI of ``include/rmsnorm.h``; this package only marshals arguments (PyTorch
provides device memory and streams).  Operation, per token row (blog
"CuTeDSL at Perplexity", section "QK norm", fused with the residual add and
the FP8 output of section "Blackwell support"):

    h = RN_in(x + residual);  residual_out = h
    y = (weight + weight_offset) * h * rsqrt(mean(h^2) + eps) + bias
    out = RN_out(y)   or   FP8-E4M3 codes of y * 448 / max|y| with scale max|y| / 448
"""
from __future__ import annotations

from ._lib import (  # noqa: F401
    EXPORTED, RMSN_EALIGN, RMSN_ECUDA, RMSN_EINVAL, RMSN_EUNSUPPORTED, RMSN_HAS_BIAS,
    RMSN_HAS_RESIDUAL, RMSN_HAS_WEIGHT, RMSN_IN_BF16, RMSN_IN_F16, RMSN_IN_F32, RMSN_OK,
    RMSN_OUT_BF16, RMSN_OUT_F16,
    RMSN_PDL, RMSN_PDL_EARLY_PARAMS, RMSN_QK_DIRECT, RMSN_QK_RING, RMSN_RESIDUAL_F32, RMSN_FMT_MXFP8, RMSN_FMT_MXFP4, RMSN_FMT_NVFP4, BLOCK_FORMATS,
    RMSN_OUT_F32, RMSN_OUT_FP8E4M3, VARIANT_BLOCK_ROW, VARIANT_BULK_PIPE, VARIANT_BULK_ROW, VARIANT_CLUSTER, VARIANT_GENERIC, VARIANT_RAGGED,
    VARIANT_NAMES, VARIANT_WARP_ROWS, RmsnConfig, RmsnError, library_path, load,
    rmsnorm_fwd, rmsnorm_fwd_ex, rmsnorm_fwd_blockscaled, rmsnorm_fwd_host, rmsnorm_list_configs, rmsnorm_qk_fwd,
    rmsnorm_query_config,
    rmsnorm_read_status, rmsnorm_set_wait_limit, status_string)
from .api import (block_format_configs, check_row_args, fused_add_rmsnorm, fused_add_rmsnorm_blockscaled,  # noqa: F401
                  fused_add_rmsnorm_host, make_flags, qk_norm_)
