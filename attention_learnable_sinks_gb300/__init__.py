"""Attention with learnable per-head sinks on one NVIDIA GB300 (sm_103a).

The computation lives in libsinkattn.so (C ABI: include/sinkattn.h); this
package is its thin PyTorch binding. Importing the package does not load the
library; the first call does, and raises if it is missing.
"""

from .api import (SinkAttention, backward, decode, forward, sink_attention,  # noqa: F401
                  workspace_bytes)

__all__ = ["SinkAttention", "sink_attention", "forward", "backward", "decode", "workspace_bytes"]
