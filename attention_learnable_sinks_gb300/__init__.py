"""Attention with learnable per-head sinks on one NVIDIA GB300 (sm_103a).

The computation lives in libsinkattn.so (C ABI: include/sinkattn.h); this
package is its thin PyTorch binding. Importing the package does not load the
library; the first call does, and raises if it is missing.
"""

from .api import backward, decode, forward, sink_attention, workspace_bytes  # noqa: F401

__all__ = ["sink_attention", "forward", "backward", "workspace_bytes"]
