"""GB300-native attention stage: RMSNorm, RoPE at data positions, in-place KV append
and grouped-query attention, as hand-written sm_103a CUDA kernels behind a C ABI
(include/minf.h, libminf.so).  `binding` holds the thin Python marshalling layer
with the C ABI's names; `kv` the device KV-region manager; `workloads` the seeded
synthetic inputs."""
from . import binding, kv, workloads  # noqa: F401
from .binding import *  # noqa: F401,F403
