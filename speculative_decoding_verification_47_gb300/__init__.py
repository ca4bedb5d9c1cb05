"""GB300-native batched lossless speculative-decoding verification.

The product is the C-ABI library ``libspecverify.so`` (CUDA kernels for
sm_103a; header ``include/specverify.h``).  ``binding`` exposes its calls to
Python under the same names; ``build`` compiles it in-tree; ``workloads``
draws seeded synthetic inputs.
"""

from .binding import (  # noqa: F401
    SVError,
    sv_kv_commit,
    sv_last_error,
    sv_lmhead_rmsnorm,
    sv_lmhead_workspace_size,
    sv_read_device_flags,
    sv_spec_verify,
    sv_version,
    sv_workspace_size,
)
