"""GB300-native (sm_103a) exact attention, FlashAttention-2 style.

The compute path is libfa.so (hand-written tcgen05 / TMA / TMEM CUDA
kernels behind the C ABI of include/fa.h).  This package is its Python
binding: the ``fa_*`` functions have the C names and marshal torch tensors
and the current torch stream into the C calls; ``forward`` and ``backward``
also allocate the outputs.  PyTorch provides device memory and streams only.
"""

from ._binding import (  # noqa: F401
    FA_ERR_CUDA,
    FA_ERR_INVALID_ARG,
    FA_BWD_NOALLOC_SCRATCH_BYTES,
    FA_CAUSAL_BOTTOM_RIGHT,
    FA_CAUSAL_NONE,
    FA_CAUSAL_TOP_LEFT,
    FA_ERR_NO_MEMORY,
    FA_ERR_SCRATCH_TOO_SMALL,
    FA_ERR_TIMEOUT,
    FA_ERR_UNSUPPORTED,
    FA_OK,
    FaError,
    backward,
    declared_symbols,
    fa_abi_version,
    fa_bwd,
    fa_bwd_general,
    fa_bwd_gqa,
    fa_bwd_noalloc,
    fa_bwd_plan,
    fa_fwd,
    fa_fwd_ex,
    fa_fwd_general,
    fa_fwd_gqa,
    fa_fwd_plan,
    fa_poll_status,
    fa_selftest_wait_timeout,
    fa_set_wait_timeout_ns,
    fa_strerror,
    fa_launch_count,
    fa_timing_enable,
    fa_timing_read,
    fa_trim_workspace,
    forward,
    load,
)

FA_KERNEL_FWD = 0
FA_KERNEL_COMBINE = 1
FA_KERNEL_BWD_PRE = 2
FA_KERNEL_BWD = 3
FA_KERNEL_BWD_DQ = 4
