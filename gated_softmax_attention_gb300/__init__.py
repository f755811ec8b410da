"""GB300 (sm_103a) gated softmax attention: the G1 sigmoid gate on the SDPA output.

The compute path is the C-ABI library ``libgsdpa.so`` built from ``csrc/``;
this package only marshals arguments to it (see ``binding``). Importing the
package does not load the library; the first call does, and it raises if the
library is missing. There is no CPU fallback.
"""
from .workloads import WORKLOADS, Workload, make_inputs  # noqa: F401

__all__ = ["WORKLOADS", "Workload", "make_inputs"]
