"""Exact single-query decode attention for B300 (sm_103a).

Split-KV (Flash-Decoding) attention and bifurcated attention for
single-context batch sampling, implemented as hand-written CUDA kernels in
``libfd_decode.so`` behind a C ABI (``include/fd_decode.h``).  This package
is the thin Python binding: it passes torch CUDA tensors as descriptors and
the current CUDA stream; it never computes anything itself.
"""

from .api import (  # noqa: F401
    FdError,
    bifurcated_attention,
    check_device_error,
    choose_num_splits,
    decode_attention,
    decode_attention_partials,
    decode_attention_multi,
    decode_attention_paged,
    decode_attention_quant,
    lse_combine,
    profile_enable,
    profile_read,
    split_bounds,
    version,
    workspace_bytes,
)
from ._lib import FD_KERNEL_BIF_CTX, FD_KERNEL_COMBINE, FD_KERNEL_SPLIT  # noqa: F401
