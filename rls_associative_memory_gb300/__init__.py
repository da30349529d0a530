"""GB300-native (sm_103a) forward recurrence of Variational Linear Attention.

The compute path is ``libvla.so`` (CUDA kernels behind the C ABI of
``include/vla.h``); this package is its thin Python binding.
"""

from ._lib import (  # noqa: F401
    VLA_BF16,
    VLA_ERR_ALIGN,
    VLA_ERR_ARG,
    VLA_ERR_CUDA,
    VLA_ERR_SCRATCH_LIMIT,
    VLA_ERR_TIMEOUT,
    VLA_ERR_UNSUPPORTED_DIM,
    VLA_ERR_WORKSPACE,
    VLA_F32,
    VLA_KERNEL_AUTO,
    VLA_KERNEL_CHUNK,
    VLA_KERNEL_CHUNK_TC,
    VLA_KERNEL_DECODE,
    VLA_KERNEL_SEQ,
    VLA_NOALLOC_SCRATCH_BYTES,
    VLA_OK,
    VLAError,
    lib,
    lib_path,
    vla_backward,
    vla_backward_workspace_bytes,
    vla_chunk_lengths,
    vla_debug_inject,
    vla_device_status,
    vla_forward_host,
    vla_forward,
    vla_host_ranges,
    vla_last_launch_count,
    vla_select_kernel,
    vla_set_launch_events,
    vla_status_str,
    vla_workspace_bytes,
)
