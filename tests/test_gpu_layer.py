"""GPU parity of the one-launch layer (both expert GEMMs of an 8-bit layer
in one persistent tcgen05 kernel: gate/up units first, then down units, a
down unit's activations loaded once every gate/up unit of its token tile
has stored them) against the oracle, forced with path="layer".

The 8-bit format options (uint8 codes, scale dtypes, per-tensor scales,
float16 activations, router weight on the input) run on this path too, in
test_gpu_variants.  Covered here: 1..300 tokens (64- and 128-row token
tiles, an expert spread over several tiles, ragged last tiles), the
fine-grained layer (zero-token experts, Zipf routing), the Mixtral-shaped
layer (split-K down GEMM across CTAs), in-place output, bitwise equality
with the two-launch path where both use the same tiles (the same
arithmetic in the same order), determinism and token-permutation
exactness, and the refusal of uint4 weights.
"""

import numpy as np
import pytest
import torch

import oracle
from moe_helpers import Layer, check_forward, inputs
from test_gpu_logits_oracle import sample_tokens
from weight_quantized_moe_gb300 import synth

pytestmark = pytest.mark.gpu

mq = pytest.importorskip("weight_quantized_moe_gb300")

W = synth.WORKLOADS


def _check(layer, x, tw, tid, what, tokens=None, **kw):
    ids = tid.cpu().numpy()
    sel = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)
    ex = layer.oracle_experts(np.unique(ids[sel]))
    ref = oracle.moe_forward(x.float().cpu().numpy(), ex, tw.cpu().numpy(), ids, tokens=sel)
    out = layer.forward(x, tw, tid, path="layer", **kw)
    torch.cuda.synchronize()
    assert mq.mq_device_status() == 0
    check_forward(out.float().cpu().numpy()[sel], ref, what=f"{what} path=layer")
    return out


@pytest.fixture(scope="module")
def tiny():
    return Layer(W["tiny"], seed=0)


@pytest.mark.parametrize("T", [1, 5, 33, 64, 65, 130, 300])
def test_layer_tiny(tiny, T):
    x, lg = inputs(tiny.wl, T, seed=300 + T)
    tw, tid = mq.moe_topk_route(lg, tiny.k, True)
    _check(tiny, x, tw, tid, f"tiny T={T}")


def test_layer_hot_expert_spans_tiles(tiny):
    """Every token routes to expert 5: with 300 tokens its segment takes three
    128-row tiles, whose down units each wait for their own tile."""
    T = 300
    x, _ = inputs(tiny.wl, T, seed=11)
    lg = synth.router_logits(T, tiny.E, seed=11, device="cuda")
    lg[:, 5] += 20.0
    tw, tid = mq.moe_topk_route(lg, tiny.k, True)
    assert (tid.cpu().numpy()[:, 0] == 5).all()
    _check(tiny, x, tw, tid, "hot expert")


@pytest.mark.parametrize("T", [40, 64, 200])
def test_layer_fine_grained_matches_two_launches(T):
    """E=128, k=8, Zipf routing (zero-token experts): the oracle on a sample
    holding every expert's first and last token, and bitwise equality with
    the two-launch tcgen05 path (the same tiles: 64 rows up to 64 tokens,
    128 beyond)."""
    layer = Layer(W["fine"], seed=2)
    x, lg = inputs(layer.wl, T, seed=400 + T)
    tw, tid = mq.moe_topk_route(lg, layer.k, True)
    assert len(np.unique(tid.cpu().numpy())) < layer.E
    sel = sample_tokens(tid.cpu().numpy(), seed=T)
    out = _check(layer, x, tw, tid, f"fine T={T}", tokens=sel)
    two = layer.forward(x, tw, tid, path="tc")
    torch.cuda.synchronize()
    assert torch.equal(out, two)


def test_layer_mixtral_split_k():
    """Mixtral-shaped layer (E=8, H=4096, I=14336) at T=3: 64-row tiles and
    the down GEMM split over K, every token."""
    layer = Layer(W["mixtral_decode"], seed=4)
    x, lg = inputs(layer.wl, 3, seed=6)
    tw, tid = mq.moe_topk_route(lg, layer.k, True)
    _check(layer, x, tw, tid, "mixtral T=3")


def test_layer_128_row_tiles_with_k_splits():
    """Two experts, H = 512, I = 4096, T = 100: 128-row tiles and the down
    units split eight ways over K, every split waiting for its token tile;
    bitwise equal to the two-launch path with the same tiles."""
    wl = synth.Workload("layer_split", E=2, k=1, H=512, I=4096, Ts=(100,))
    layer = Layer(wl, seed=12)
    x, lg = inputs(wl, 100, seed=12)
    tw, tid = mq.moe_topk_route(lg, wl.k, True)
    out = _check(layer, x, tw, tid, "two experts, K splits")
    two = layer.forward(x, tw, tid, path="tc")
    torch.cuda.synchronize()
    assert torch.equal(out, two)


def test_layer_in_place(tiny):
    """out == x (fused_experts' inplace): x is gathered before any output is
    written, also when one launch runs both GEMMs."""
    T = 90
    x, lg = inputs(tiny.wl, T, seed=21)
    tw, tid = mq.moe_topk_route(lg, tiny.k, True)
    ref = tiny.forward(x, tw, tid, path="layer").clone()
    xi = x.clone()
    got = tiny.forward(xi, tw, tid, path="layer", inplace=True)
    torch.cuda.synchronize()
    assert got.data_ptr() == xi.data_ptr()
    assert torch.equal(got, ref)


@pytest.mark.parametrize("name,T", [("tiny", 150), ("fine", 64)])
def test_layer_deterministic_and_permutation_exact(name, T):
    layer = Layer(W[name], seed=0)
    layer.free_bf16()
    x, lg = inputs(layer.wl, T, seed=9)
    tw, tid = mq.moe_topk_route(lg, layer.k, True)
    outs = [layer.forward(x, tw, tid, path="layer").clone() for _ in range(3)]
    perm = torch.from_numpy(np.random.default_rng(T).permutation(T)).cuda()
    tw_p, tid_p = mq.moe_topk_route(lg[perm].contiguous(), layer.k, True)
    out_p = layer.forward(x[perm].contiguous(), tw_p, tid_p, path="layer")
    torch.cuda.synchronize()
    assert mq.mq_device_status() == 0
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    assert torch.equal(out_p, outs[0][perm])


def test_layer_refuses_uint4():
    wl = synth.Workload("w4_layer", E=4, k=2, H=128, I=128, Ts=(4,), bits=4, group_size=128,
                        has_zp=True)
    layer = Layer(wl, seed=1)
    x, lg = inputs(wl, 4, seed=1)
    tw, tid = mq.moe_topk_route(lg, wl.k, True)
    with pytest.raises(mq.MoeqError) as ei:
        layer.forward(x, tw, tid, path="layer")
    assert ei.value.status == mq.binding.MQ_ERR_UNSUPPORTED
