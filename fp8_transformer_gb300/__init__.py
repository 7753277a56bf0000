"""GB300-native (sm_103a) fused normalization + feed-forward block.

The compute lives in libte_gb300.so (hand-written CUDA: register-streamed norm forward and a
TMA-ring norm backward, tcgen05/TMEM GEMMs fed by TMA with fused bias/activation/amax/E4M3
epilogues, bandwidth-bound activation, quantize and dact+dbias kernels) behind the C ABI of
include/te_gb300.h.  This package is its thin Python binding; the functions keep the C names.
"""

from .binding import (ACT_TUPLES, ACT_TYPES, EXPORTED, KERNEL_KINDS, NORM_TYPES, Quantizer,
                      QuantizerSet, TEError, dact_dbias_noalloc_capacity, get_device_status, lib,
                      lib_path, profile_begin, profile_end, selftest_wait_timeout, status_string,
                      stream_probe, te_act_lu,
                      te_dact_dbias_quantize, te_dact_dbias_quantize_noalloc, te_gemm,
                      te_layernorm_dense_bwd, te_layernorm_dense_fwd, te_layernorm_mlp_bwd,
                      te_layernorm_mlp_fwd, te_layernorm_mlp_fwd_host, te_norm_bwd, te_norm_fwd,
                      te_quantize, version, workspace_size)
from .binding import *  # noqa: F401,F403  (enum constants)

__all__ = ["Quantizer", "QuantizerSet", "TEError", "te_norm_fwd", "te_act_lu",
           "te_dact_dbias_quantize", "te_quantize", "te_gemm", "te_layernorm_dense_fwd",
           "te_layernorm_mlp_fwd", "te_layernorm_mlp_bwd", "te_layernorm_dense_bwd",
           "te_norm_bwd", "lib", "lib_path", "version",
           "get_device_status", "status_string", "workspace_size", "EXPORTED", "ACT_TYPES",
           "ACT_TUPLES", "NORM_TYPES", "KERNEL_KINDS", "profile_begin", "profile_end",
           "te_dact_dbias_quantize_noalloc", "dact_dbias_noalloc_capacity",
           "selftest_wait_timeout", "te_layernorm_mlp_fwd_host", "stream_probe"]
