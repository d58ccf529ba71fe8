"""GB300-native Global-QSGD compress / aggregate / decompress (Xin, Canini, Richtarik, Horvath,
"Global-QSGD: Practical Floatless Quantization for Distributed Learning with Theoretical
Guarantees", arXiv 2305.18627).

The compute lives in libgq.so (hand-written CUDA for sm_103a, C ABI in include/gq.h); this
package is a thin ctypes binding with the same names.  PyTorch supplies device memory and
streams only.  There is no CPU fallback: importing the package without a built libgq.so raises.
"""
from ._binding import (  # noqa: F401
    BF16, EXP, F16, F32, LINEAR, NORM_INF, NORM_L2, ORDER_RING, ORDER_TREE, ROUND_U16, SUM_I32,
    SUM_I8,
    GQError, gq_abi_version, gq_allreduce_mean, gq_allreduce_mean_noalloc,
    gq_allreduce_mean_segments, gq_allreduce_mean_to, gq_allreduce_mean_with_norm,
    gq_allreduce_mean_with_norm_ws, gq_code_bits,
    gq_code_bytes, gq_code_pitch, gq_debug_status, gq_dequantize, gq_dequantize_sums, gq_dequantize_to,
    gq_exp_allreduce, gq_exp_combine, gq_exp_dequantize, gq_exp_ring_stream, gq_exp_tree_stream,
    gq_fused_launches, gq_get_status, gq_global_norm, gq_noalloc_max_blocks, gq_norm_blocks,
    gq_norm_finish, gq_norm_partial, gq_philox4x32_10, gq_quantize,
    gq_quantize_codes, gq_quantize_sum, gq_quantize_ws, gq_reduce_codes, gq_selftest_wait_timeout,
    gq_status_string, gq_workspace, gq_workspace_bytes, lib, library_path)
