"""Weight-only-quantised fused MoE forward for GB300 (sm_103a).

The compute lives in ``libmoeq.so`` (CUDA kernels behind the C ABI declared
in ``include/moeq.h``); ``binding`` exposes the same entry points to Python
for torch tensors.  ``synth`` draws the seeded synthetic inputs.
"""

from .binding import (  # noqa: F401
    MoeqError,
    lib,
    mq_device_status,
    mq_kernel_launch_count,
    mq_profile_enable,
    mq_test_layer_wait_extra,
    mq_profile_read,
    mq_status_string,
    moe_align_block,
    moe_align_capacity,
    moe_quant_forward,
    moe_quant_forward_logits,
    moe_quant_forward_workspace,
    moe_quantize_int8_per_channel,
    moe_quantize_uint4_group,
    moe_topk_route,
    MQ_DEV_BAD_EXPERT_ID,
    MQ_DEV_WAIT_TIMEOUT,
    MQ_FWD_W8_UINT8,
    MQ_FWD_SCALE_F16,
    MQ_FWD_SCALE_BF16,
    MQ_FWD_SCALE_PER_TENSOR,
    MQ_FWD_ACT_F16,
    MQ_FWD_ROUTER_WEIGHT_ON_INPUT,
    MQ_FWD_PATH_TENSOR_CORE,
    MQ_FWD_PATH_DECODE,
    MQ_FWD_PATH_LAYER,
    MQ_SCORING_SOFTMAX,
    MQ_SCORING_SIGMOID,
    MqRouteOpts,
    forward_flags,
)
