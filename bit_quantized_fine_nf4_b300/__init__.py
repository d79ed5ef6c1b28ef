"""B300-native QLoRA NF4 linear: NF4 quantise / dequantise with double quantisation,
fused forward and backward through the dequantised weight with a LoRA side path.

The compute lives in ``libqlora_nf4.so`` (hand-written sm_103a CUDA behind the C
ABI in ``include/qlora_nf4.h``); this package is its thin ctypes binding plus
the data-parallel gradient exchange helper.
"""

from ._binding import (  # noqa: F401
    ACCUM_DA,
    ACCUM_DB,
    ACCUM_DX,
    EXPORTS,
    GroupedForward,
    LIB_PATH,
    NF4Weight,
    QloraError,
    QLORA_ERR_CUDA,
    QLORA_ERR_INVALID_ARGUMENT,
    QLORA_ERR_NONFINITE,
    QLORA_ERR_TIMEOUT,
    QLORA_ERR_UNSUPPORTED,
    QLORA_OK,
    bwd_workspace_bytes,
    check_status,
    dequantize,
    device_sm_count,
    fwd_workspace_bytes,
    get_status,
    launch_count,
    linear_bwd,
    linear_fwd,
    linear_fwd_grouped,
    load,
    lowrank_update,
    merge,
    profile_enable,
    profile_read,
    profile_reset,
    quantize,
    quantize_noalloc,
    quantize_workspace_bytes,
    selftest_wait_timeout,
    set_wait_limit_ns,
    silu_mul_bwd,
    silu_mul_fwd,
)
