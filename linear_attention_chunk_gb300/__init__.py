"""libgla: the Simple Gated Linear Attention mixer on GB300 (sm_103a).

The hot path (chunked forward, chunked backward, decode step) runs in the
hand-written CUDA kernels of libgla.so behind the C ABI in include/gla.h;
this package holds those sources (csrc/), the in-tree build (build.py) and
a thin ctypes binding with the ABI's names (binding.py).
"""
from .binding import (  # noqa: F401
    ABI_FUNCTIONS,
    GLA_BF16,
    GLA_ERR_CUDA,
    GLA_ERR_INVALID_ARG,
    GLA_ERR_TIMEOUT,
    GLA_ERR_UNSUPPORTED,
    GLA_ERR_WORKSPACE,
    GLA_FP32,
    GLA_OK,
    GlaError,
    gla_check,
    gla_chunk_bwd,
    gla_chunk_bwd_gated,
    gla_chunk_bwd_gated_workspace_size,
    gla_chunk_bwd_workspace_size,
    gla_chunk_fwd,
    gla_chunk_fwd_gated,
    gla_chunk_fwd_gated_workspace_size,
    gla_chunk_fwd_mixer,
    gla_chunk_fwd_noalloc,
    gla_chunk_fwd_varlen,
    gla_chunk_fwd_varlen_gated,
    gla_chunk_fwd_workspace_size,
    gla_conv1d_fwd,
    gla_conv1d_step,
    gla_conv1d_varlen,
    gla_decode_step,
    gla_decode_step_gated,
    gla_decode_step_mixer,
    gla_last_launch_count,
    gla_mixer_epilogue,
    gla_selftest_wait_timeout,
    gla_status_string,
    gla_version,
    lib,
)
