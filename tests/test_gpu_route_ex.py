"""GPU parity of the router options (moe_topk_route_ex and
moe_quant_forward_logits_ex): sigmoid scoring, expert groups, the
score-correction bias and the routed scaling factor, against the oracle's
``topk_route_ex``."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from moe_helpers import route_tolerance
from weight_quantized_moe_gb300 import synth

pytestmark = pytest.mark.gpu

mq = pytest.importorskip("weight_quantized_moe_gb300")

# name: (E, k, options); options as moe_topk_route's keyword arguments
CASES = {
    # 256 experts in 8 groups, 4 kept, sigmoid with a bias, scaled by 2.5
    "groups_sigmoid_bias": (256, 8, dict(scoring_func="sigmoid", num_expert_group=8, topk_group=4,
                                         bias=0.05, routed_scaling_factor=2.5)),
    # 160 experts in 8 groups, 3 kept, softmax, scaled by 16, not renormalised
    "groups_softmax": (160, 6, dict(num_expert_group=8, topk_group=3, routed_scaling_factor=16.0)),
    "sigmoid": (128, 8, dict(scoring_func="sigmoid")),
    "sigmoid_k1": (16, 1, dict(scoring_func="sigmoid")),
    "softmax_bias": (64, 6, dict(bias=0.02)),
    "groups_one_lane": (32, 4, dict(num_expert_group=4, topk_group=2)),
    "max_sizes": (1024, 32, dict(scoring_func="sigmoid", num_expert_group=32, topk_group=8,
                                 bias=0.01)),
    "scale_only": (8, 2, dict(routed_scaling_factor=0.5)),
}


def _options(E, opts, seed):
    o = dict(opts)
    sd = o.pop("bias", None)
    bias = None
    if sd is not None:
        bias = torch.from_numpy(np.random.default_rng(seed).normal(0, sd, E).astype(np.float32))
    return o, bias


def _keys(lg, o, bias):
    """The oracle's selection keys (float32), to judge near-ties."""
    if bias is None:
        return lg
    return oracle.moe_oracle._scores_f32(lg, o.get("scoring_func", "softmax")) + bias[None, :]


def _compare_ids(gpu, ref, key, exact):
    """Bitwise, or (with a bias, where the key is a float32 sum that CPU and
    GPU exp() may round apart) equal on >= 99% of tokens and, elsewhere,
    equal up to a near-tie: the two choices' keys agree within 1e-5."""
    same = (gpu == ref).all(1)
    if exact:
        assert same.all()
        return
    assert same.mean() >= 0.99
    for t in np.nonzero(~same)[0]:
        np.testing.assert_allclose(np.sort(key[t, gpu[t]]), np.sort(key[t, ref[t]]), atol=1e-5)


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("renorm", [True, False])
@pytest.mark.parametrize("T", [1, 300])
def test_route_ex_parity(name, renorm, T):
    E, k, opts = CASES[name]
    o, bias = _options(E, opts, seed=E + k)
    lg = synth.router_logits(T, E, seed=T + E, bias="zipf" if E >= 64 else None)
    w, ids = mq.moe_topk_route(lg.cuda(), k, renorm, **o,
                               e_score_correction_bias=None if bias is None else bias.cuda())
    torch.cuda.synchronize()
    ow, oid = oracle.topk_route_ex(lg.numpy(), k, renorm, **o,
                                   e_score_correction_bias=None if bias is None else bias.numpy())
    gid = ids.cpu().numpy()
    key = _keys(lg.numpy(), o, None if bias is None else bias.numpy())
    _compare_ids(gid, oid, key, exact=bias is None)
    same = (gid == oid).all(1)
    np.testing.assert_allclose(w.cpu().numpy()[same], ow[same], rtol=route_tolerance(E), atol=0)
    assert np.isfinite(w.cpu().numpy()).all()


def test_route_ex_defaults_equal_plain_router():
    """The options path with the defaults is bitwise the plain router."""
    from weight_quantized_moe_gb300 import binding
    lg = synth.router_logits(500, 128, seed=3, bias="zipf").cuda()
    for renorm in (True, False):
        w0, i0 = mq.moe_topk_route(lg, 8, renorm)
        opts, _ = binding.route_opts(128, renorm)
        w1 = torch.empty_like(w0)
        i1 = torch.empty_like(i0)
        binding._check(binding.lib().moe_topk_route_ex(
            binding._ptr(lg), 500, 128, 8, ctypes.byref(opts), binding._ptr(w1),
            binding._ptr(i1), binding._stream()))
        torch.cuda.synchronize()
        assert torch.equal(i0, i1) and torch.equal(w0, w1)


def test_route_ex_group_ties_and_nan():
    """Equal group maxima keep the lower group; NaN logits never win."""
    lg = torch.tensor([[1.0, 0.0, 0.0, 1.0, 0.0, 0.0, 0.0, 0.0],
                       [float("nan"), 0.5, 0.5, 0.5, 0.0, 0.0, 0.0, 0.0],
                       [0.0] * 8])
    for kw in (dict(num_expert_group=2, topk_group=1), dict(num_expert_group=4, topk_group=2,
                                                           scoring_func="sigmoid")):
        w, ids = mq.moe_topk_route(lg.cuda(), 2, True, **kw)
        torch.cuda.synchronize()
        ow, oid = oracle.topk_route_ex(lg.numpy(), 2, True, **kw)
        assert np.array_equal(ids.cpu().numpy(), oid)
        # a NaN logit makes the oracle's softmax row NaN; compare the others
        np.testing.assert_allclose(w.cpu().numpy()[[0, 2]], ow[[0, 2]], rtol=1e-6)


@pytest.mark.parametrize("T", [1, 64, 700])
def test_forward_logits_ex_equals_route_then_forward(T):
    """moe_quant_forward_logits with router options gives bitwise the result
    of moe_topk_route with those options followed by moe_quant_forward."""
    from moe_helpers import Layer, inputs
    layer = Layer(synth.WORKLOADS["fine"], seed=2)
    layer.free_bf16()
    x, lg = inputs(layer.wl, T, seed=T)
    bias = torch.from_numpy(np.random.default_rng(7).normal(0, 0.05, layer.E)
                            .astype(np.float32)).cuda()
    kw = dict(scoring_func="sigmoid", num_expert_group=8, topk_group=4,
              e_score_correction_bias=bias, routed_scaling_factor=2.5)
    tw, tid = mq.moe_topk_route(lg, layer.k, True, **kw)
    ref = layer.forward(x, tw, tid)
    got = mq.moe_quant_forward_logits(x, lg, layer.q13, layer.q2, layer.s13, layer.s2, layer.k,
                                      True, bits=layer.bits, group_size=layer.gs, **kw)
    torch.cuda.synchronize()
    assert mq.mq_device_status() == 0
    assert torch.equal(got, ref)
