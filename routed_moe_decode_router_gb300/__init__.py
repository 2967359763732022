"""GB300-native routed MoE forward for 1..8 token rows (decode, verify,
prefill sub-chunks): router, top-k, union of the selected experts, NVFP4
expert sweep and shared-expert blend, behind a C-ABI CUDA library."""
