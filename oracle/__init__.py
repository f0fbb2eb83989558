"""CPU oracle for the routed NVFP4 MoE expert block with the MuseSpark1x
post-expert finalize.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may use it. It shares no code,
tables or constants with the CUDA path under
``nvfp4_mixture_experts_route_gb300/``; the two meet only in the seeded input
generators (``nvfp4_mixture_experts_route_gb300.inputs``), which hold none of
the method's arithmetic.

Plain, slow and meant to be read against the pages:

* ``codecs``   e2m1 / e4m3 / bf16 codecs written from the format definitions.
* ``quant``    NVFP4 quantization of 16-element blocks with an fp32 global
               scale (``ops.scaled_fp4_quant`` role on the flashinfer_ops and
               model pages).
* ``routing``  the routing metadata by its definition (flashinfer_ops page,
               ``FlashInferOps.slot`` and ``gemm2_rows``).
* ``gemm``     block-scaled FP4 products, exact in int64, plus an fp64
               dequantize-and-matmul mode for large shapes.
* ``layer``    the whole expert block route by route, and the post-expert
               finalize (muse_moe_runner page, ``_finalize_native`` /
               ``_finalize_chunk`` / ``_effective_weight``).
* ``layout``   the prepared weight layout, packed and unpacked by its
               documented definition, and the expert-TP slice views
               (expert_tp page, module docstring and ``slice_views``).
* ``calibrate`` writes the stored global scales of the synthetic layers.

Parity status of each function is stated in its docstring; every function
here is pinned by a ``-m "not gpu"`` test in ``tests/test_oracle_*.py``.
"""
