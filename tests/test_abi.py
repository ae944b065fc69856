"""CPU checks of the C ABI: the library builds, loads, exports every symbol
that include/moeq.h declares, and rejects bad arguments on the host before
launching anything (no GPU needed for these paths)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from weight_quantized_moe_gb300 import binding, build
    build.build()
    return binding.lib()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "moeq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(?:int|int64_t|size_t|long long|const char\*)\s+(\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    from weight_quantized_moe_gb300 import binding
    assert binding.mq_status_string(0) == "ok"
    assert "invalid" in binding.mq_status_string(1)


def test_align_capacity(lib):
    from weight_quantized_moe_gb300 import binding
    import oracle
    for args in [(16, 2, 8, 16), (1, 2, 8, 64), (8192, 2, 8, 128), (4096, 8, 128, 64), (0, 2, 8, 16)]:
        assert binding.moe_align_capacity(*args) == oracle.align_capacity(*args)
    assert binding.moe_align_capacity(-1, 2, 8, 16) == -1


def test_host_side_rejections(lib):
    from weight_quantized_moe_gb300 import binding
    vp = ctypes.c_void_p
    fake = vp(0x1000)  # never dereferenced: every case fails validation first
    # unsupported format (bits=8 with a group size)
    assert lib.moe_quant_forward(fake, 4, 128, 128, 8, 2, 8, 128, 0, fake, fake, fake, fake,
                                 None, None, fake, fake, fake, 1 << 20, fake, None) == 2
    # H not a multiple of 128
    assert lib.moe_quant_forward(fake, 4, 100, 128, 8, 2, 8, -1, 0, fake, fake, fake, fake,
                                 None, None, fake, fake, fake, 1 << 20, fake, None) == 2
    # k > E
    assert lib.moe_quant_forward(fake, 4, 128, 128, 2, 3, 8, -1, 0, fake, fake, fake, fake,
                                 None, None, fake, fake, fake, 1 << 20, fake, None) == 1
    # workspace too small
    assert lib.moe_quant_forward(fake, 4, 128, 128, 8, 2, 8, -1, 0, fake, fake, fake, fake,
                                 None, None, fake, fake, fake, 16, vp(0x9000), None) == 4
    # out overlapping x
    assert lib.moe_quant_forward(fake, 4, 128, 128, 8, 2, 8, -1, 0, fake, fake, fake, fake,
                                 None, None, fake, fake, fake, 1 << 30, vp(0x1100), None) == 1
    assert b"overlap" in lib.mq_last_error_message()
    # moe_quant_forward_ex: options that do not fit the format, unknown bits,
    # both scale dtypes, zeros with int8 codes; out == x (in place) passes
    # validation up to the workspace check
    ex = lib.moe_quant_forward_ex
    args = lambda bits, gs, zp, z, flags, out=vp(0x9000), ws=1 << 30: (
        fake, 4, 128, 128, 8, 2, bits, gs, zp, fake, fake, fake, fake, z, z, fake, fake, fake,
        ws, out, flags, None)
    assert ex(*args(4, 128, 0, None, binding.MQ_FWD_W8_UINT8)) == 2
    assert ex(*args(4, 128, 0, None, binding.MQ_FWD_SCALE_PER_TENSOR)) == 2
    assert ex(*args(8, -1, 0, None, 0x400)) == 2
    assert ex(*args(8, -1, 0, None, binding.MQ_FWD_SCALE_F16 | binding.MQ_FWD_SCALE_BF16)) == 2
    assert ex(*args(8, -1, 1, fake, 0)) == 2
    assert ex(*args(8, -1, 1, None, binding.MQ_FWD_W8_UINT8)) == 1
    assert ex(*args(8, -1, 0, None, 0, out=vp(0x1100))) == 1
    assert ex(*args(8, -1, 0, None, binding.MQ_FWD_ACT_F16, out=fake, ws=16)) == 4
    # kernel selection: at most one path flag; the one-launch layer takes 8-bit codes
    assert ex(*args(8, -1, 0, None, binding.MQ_FWD_PATH_LAYER | binding.MQ_FWD_PATH_TENSOR_CORE)) == 1
    assert ex(*args(8, -1, 0, None, binding.MQ_FWD_PATH_LAYER | binding.MQ_FWD_PATH_DECODE)) == 1
    assert ex(*args(4, 128, 0, None, binding.MQ_FWD_PATH_LAYER)) == 2
    assert ex(*args(8, -1, 0, None, binding.MQ_FWD_PATH_LAYER, ws=16)) == 4
    # moe_quant_forward_logits: null logits; workspace query includes routing
    assert lib.moe_quant_forward_logits(fake, None, 4, 128, 128, 8, 2, 1, 8, -1, 0, fake, fake,
                                        fake, fake, None, None, fake, 1 << 30, vp(0x9000), 0,
                                        None) == 1
    assert (lib.moe_quant_forward_logits_workspace(64, 128, 128, 8, 2, 8, -1)
            > lib.moe_quant_forward_workspace(64, 128, 128, 8, 2, 8, -1))
    # null pointers, odd rows, bad group size, k > 32
    assert lib.moe_quantize_int8_per_channel(None, 4, 8, fake, fake, None) == 1
    assert lib.moe_quantize_int8_per_channel(fake, 4, 12, fake, fake, None) == 1
    assert lib.moe_quantize_uint4_group(fake, 3, 256, 128, fake, fake, fake, None) == 1
    assert lib.moe_quantize_uint4_group(fake, 4, 256, 96, fake, fake, fake, None) == 1
    assert lib.moe_topk_route(fake, 4, 64, 33, 1, fake, fake, None) == 1
    assert lib.moe_topk_route(fake, 4, 2048, 8, 1, fake, fake, None) == 2
    assert lib.moe_align_block(fake, 4, 2, 8, 16, fake, fake, fake, fake, 8, None) == 1
    assert lib.moe_quant_forward_workspace(4, 128, 128, 8, 2, 8, -1) > 0
    assert lib.moe_quant_forward_workspace(4, 128, 128, 8, 2, 3, -1) == 0
    # the bounded-wait testing hook takes extra >= 0 (0 restores)
    assert lib.mq_test_layer_wait_extra(-1) == 1
    assert lib.mq_test_layer_wait_extra(0) == 0


def test_route_options_rejections(lib):
    """moe_topk_route_ex / moe_quant_forward_logits_ex check the router
    options on the host before anything is launched."""
    from weight_quantized_moe_gb300 import binding
    vp = ctypes.c_void_p
    fake = vp(0x1000)

    def opts(**kw):
        base = dict(scoring_func=binding.MQ_SCORING_SIGMOID, renormalize=1, num_expert_group=8,
                    topk_group=4, e_score_correction_bias=None, routed_scaling_factor=2.5)
        base.update(kw)
        return ctypes.byref(binding.MqRouteOpts(**base))

    def route(o, E=256, k=8):
        return lib.moe_topk_route_ex(fake, 4, E, k, o, fake, fake, None)

    assert lib.moe_topk_route_ex(fake, 4, 256, 8, None, fake, fake, None) == 1  # null opts
    assert route(opts(scoring_func=2)) == 1
    assert route(opts(num_expert_group=33, topk_group=1)) == 1
    assert route(opts(num_expert_group=-1)) == 1
    assert route(opts(num_expert_group=6)) == 1           # 6 does not divide 256
    assert route(opts(topk_group=0)) == 1
    assert route(opts(topk_group=9)) == 1
    assert route(opts(topk_group=1), k=33) == 1          # k > 32
    assert route(opts(topk_group=1, num_expert_group=32), k=9) == 1  # 9 > 1 group of 8
    assert route(opts(routed_scaling_factor=float("inf"))) == 1
    assert route(opts(routed_scaling_factor=float("nan"))) == 1
    assert route(opts(e_score_correction_bias=0x1004)) == 1  # misaligned bias
    assert route(opts(), E=2048) == 2
    # T = 0 with valid options: nothing to do
    assert lib.moe_topk_route_ex(fake, 0, 256, 8, opts(), fake, fake, None) == 0
    assert lib.moe_quant_forward_logits_ex(fake, fake, 4, 128, 128, 256, 8, opts(topk_group=0), 8,
                                           -1, 0, fake, fake, fake, fake, None, None, fake,
                                           1 << 30, fake, 0, None) == 1
    assert lib.moe_quant_forward_logits_ex(fake, fake, 4, 128, 128, 256, 8, None, 8, -1, 0,
                                           fake, fake, fake, fake, None, None, fake, 1 << 30,
                                           fake, 0, None) == 1


def test_route_opts_marshalling():
    """The binding's mq_route_opts matches the C layout, and only the
    defaults count as the plain router."""
    from weight_quantized_moe_gb300 import binding
    assert ctypes.sizeof(binding.MqRouteOpts) == 32
    assert binding.MqRouteOpts.e_score_correction_bias.offset == 16
    assert binding.MqRouteOpts.routed_scaling_factor.offset == 24
    o, plain = binding.route_opts(64, True)
    assert plain and o.scoring_func == binding.MQ_SCORING_SOFTMAX and o.renormalize == 1
    assert o.routed_scaling_factor == 1.0 and not o.e_score_correction_bias
    for kw in (dict(scoring_func="sigmoid"), dict(num_expert_group=8, topk_group=2),
               dict(routed_scaling_factor=2.5)):
        o, plain = binding.route_opts(64, False, **kw)
        assert not plain
    o, plain = binding.route_opts(64, False, num_expert_group=1, topk_group=0)
    assert plain
    with pytest.raises(ValueError):
        binding.route_opts(64, True, scoring_func="tanh")


def test_binding_rejects_bad_weight_tensors():
    """Every forward wrapper checks the weights, scales and zero points
    before any pointer reaches the library: host tensors and wrong dtypes
    are refused (the GPU tests cover strided views)."""
    import torch
    from weight_quantized_moe_gb300 import binding
    w13 = torch.zeros(2, 8, 16, dtype=torch.int8)
    w2 = torch.zeros(2, 16, 4, dtype=torch.int8)
    s13 = torch.zeros(2, 8)
    s2 = torch.zeros(2, 16)
    with pytest.raises(ValueError, match="CUDA"):
        binding.check_weights(w13, w2, s13, s2, 8, False)
    with pytest.raises(TypeError):
        binding.check_weights(w13.float(), w2, s13, s2, 8, False)
    with pytest.raises(TypeError):  # uint4 storage is uint8
        binding.check_weights(w13, w2, s13.half(), s2.half(), 4, True)
    with pytest.raises(ValueError, match="bits"):
        binding.check_weights(w13, w2, s13, s2, 6, False)
