"""GB300 (sm_103a) ternary-weight linear layer: C-ABI CUDA library + binding.

The compute lives in libtern.so (include/tern.h); ``binding`` marshals
arguments to it.  Build with ``ternary_weight_linear_block_gb300.build.build()``.
"""
