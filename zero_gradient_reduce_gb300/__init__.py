"""GB300-native ZeRO synchronisation-and-update step.

The product is the C-ABI CUDA library libzdp (include/zdp.h); ``zdp`` is its
thin Python binding, ``streaming`` drives a ZeRO-2 step bucket by bucket on
two CUDA streams, and ``workloads`` generates seeded synthetic inputs.
"""

from . import streaming, workloads, zdp  # noqa: F401
from .zdp import (  # noqa: F401
    ZdpError, zdp_all_gather, zdp_adamw_shard, zdp_last_error, zdp_reduce_scatter,
    zdp_shard_size, zdp_step, zdp_step_workspace_bytes, zdp_version, make_step_args,
)

__all__ = [
    "zdp", "streaming", "workloads", "ZdpError", "zdp_all_gather", "zdp_adamw_shard", "zdp_last_error",
    "zdp_reduce_scatter", "zdp_shard_size", "zdp_step", "zdp_step_workspace_bytes",
    "zdp_version", "make_step_args",
]
