"""GB300-native grouped (MoE) block-scaled quantize + grouped GEMM.

The compute path is the C-ABI library ``libmxg.so`` (hand-written sm_103a
kernels, declared in ``include/mxg.h``); ``moe_grouped_block_gb300.mxg`` is the
thin Python binding over it.  ``moe_grouped_block_gb300.workloads`` holds the
seeded synthetic inputs.  Nothing is imported here, so the input generator can
be used on a machine without a GPU: import the submodules explicitly.
"""
