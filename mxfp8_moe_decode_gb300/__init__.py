"""GB300 (sm_103a) MXFP8 MoE decode step: the FFN half of one decode step.

``MoeDecode`` (mxfp8_moe_decode_gb300.api) wraps the C ABI of
libmoe_decode.so (include/moe_decode.h); ``workloads`` draws seeded synthetic
inputs; ``build`` compiles the library in-tree with nvcc.
"""

from .api import MoeDecode, expected_shapes, kernel_names  # noqa: F401
