"""CPU oracle for the weight-only-quantized fused MoE forward.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
in ``__graft_entry__`` and the ``cpu_baseline`` / ``--impl reference`` legs of
``bench.py`` may import this package.  The CUDA library never calls it and
shares no code with it; the two meet only at the seeded synthetic inputs.

Everything here is plain numpy, written to be read against the vLLM API pages
it restates:

* "vllm.model_executor.layers.quantization.experts_int8"  -- the W8A16 path
  (``ExpertsInt8MoEMethod.create_weights`` / ``apply`` /
  ``quantizing_weight_loader`` and ``quantize_in_place_and_get_scales``);
* "vllm.model_executor.layers.quantization.moe_wna16" -- the W4A16
  group-quantised storage (``MoeWNA16Method.create_weights`` and the AWQ/GPTQ
  conversions inside ``get_weight_loader``) and its 8-bit form (uint8 codes,
  per-row scales and zeros);
* "vllm.model_executor.layers.fused_moe.oracle.int8" -- the per-tensor
  ("tensor" strategy) int8 scale.

Precision: the forward runs in float64.  The two quantisers take their
integer decisions in float32 (the precision the GPU kernels use), because a
quantised code is an integer decided by floating point and both sides must
decide it the same way.

Pins: every function below is checked, in ``tests/test_oracle_*.py``, against
something other than itself (brute force, closed forms, invariants, library
routines).  No function here is "parity unpinned".
"""

from .moe_oracle import (  # noqa: F401
    quantize_int8_per_channel,
    dequantize_int8_per_channel,
    quantize_uint4_group,
    pack_uint4_along_k,
    unpack_uint4_along_k,
    pack_uint4_along_n,
    unpack_uint4_along_n,
    dequantize_uint4_group,
    dequantize_uint8_per_channel,
    topk_route,
    topk_route_ex,
    align_capacity,
    align_block,
    silu,
    round_to_bf16,
    moe_forward,
    Int8Experts,
    Uint4Experts,
    Uint8Experts,
    Int8TensorExperts,
)
