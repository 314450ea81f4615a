"""CPU oracle for the MXFP8 MoE decode step (FFN half of one decode step).

TEST INFRASTRUCTURE ONLY. Only the test suite, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product path (the C-ABI library and its Python binding) never calls it and
shares no code, table or constant generator with it.

The oracle is plain numpy in float64 over the exact values of the bf16 / E4M3 /
E8M0 inputs. Every function cites the passage of the source pages it follows:

* "vllm.models.deepseek_v41.amd.mono.layer" (the layer page): ``store_normed``,
  ``store_x8`` and ``run_ffn``;
* "vllm.models.deepseek_v41.amd.mono.runner" (the runner page):
  ``MonoLayerWeights`` and its ``check``, ``DSV41MonoLayer.ffn``;
* "vllm.models.deepseek_v41.amd.mono.attention.device" (the device page):
  ``mx_code``, ``ceil_exp``, ``div_rn``, ``mx_mul``, ``fp8_pack4``,
  ``fp8x8_bf16``, ``mfma_scaled``.

Modules:

* :mod:`oracle.numerics` -- bf16 / fp32 rounding and the OCP E4M3 and E2M1 codecs.
* :mod:`oracle.mx`       -- the E8M0 scale code, 32-group quantisation, and
  the dequantisation of 32 x 32-block E4M3 and per-row 1 x 32 E2M1 weights.
* :mod:`oracle.moe`      -- RMSNorm, router, experts, combine, whole step.

Pinning status (what fixes each function other than itself) is listed in each
module's header. The end-to-end step composes pinned pieces; its numbers have
no worked example on the pages ("parity unpinned" for the composition as a
whole, see :mod:`oracle.moe`).
"""
