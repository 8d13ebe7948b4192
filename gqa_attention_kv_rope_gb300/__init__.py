"""GB300-native attention stage: RMSNorm, RoPE at data positions, in-place KV append
and grouped-query attention, as hand-written sm_103a CUDA kernels behind a C ABI."""
