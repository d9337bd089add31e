"""Single-GPU MoE layer for GB300 (sm_103a): top-k routing, device-side plan,
gather, tcgen05 grouped expert FFNs, fixed-order combine and the backward,
behind the C ABI of include/mok.h (libmok.so, bound in ``mok``)."""
from . import workloads  # noqa: F401
