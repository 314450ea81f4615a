"""GB300 (sm_103a) MXFP8 MoE decode step: the FFN half of one decode step.

``MoeDecode`` and ``attn_seam_x8`` (mxfp8_moe_decode_gb300.api) wrap the C ABI of
libmoe_decode.so (include/moe_decode.h); ``workloads`` draws seeded synthetic
inputs; ``build`` compiles the library in-tree with nvcc.
"""

from .api import MoeDecode, attn_seam_x8, expected_shapes, kernel_names  # noqa: F401
