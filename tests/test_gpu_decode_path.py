"""GPU parity of the warp-MMA consumers of the expert GEMMs (for experts
holding a few token-slots: the converter warps multiply the exactly
dequantised, TMA-staged weight tiles with mma.sync themselves) against the
oracle, forced for both GEMMs with path="decode", beside the tcgen05
consumers (path="tc") on the same inputs.

Covered: 1..64 tokens (one and two 8-token MMA groups, 16- and 32-row
chunks), an expert with more slots than a chunk (several chunks stream its
weights), uint4 with group sizes 128 and 256 with and without zero points,
the fine-grained layer (zero-token experts, uneven K steps per warp), and
the refusal of uint4 group sizes the warp-MMA consumers do not take.
"""

import numpy as np
import pytest
import torch

import oracle
from moe_helpers import Layer, check_forward, inputs
from weight_quantized_moe_gb300 import synth

pytestmark = pytest.mark.gpu

mq = pytest.importorskip("weight_quantized_moe_gb300")

W = synth.WORKLOADS


def _check_paths(layer, x, tw, tid, what, tokens=None, paths=("decode", "tc")):
    """Forward on each path, each against the oracle."""
    ids = tid.cpu().numpy()
    sel = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)
    ex = layer.oracle_experts(np.unique(ids[sel]))
    ref = oracle.moe_forward(x.float().cpu().numpy(), ex, tw.cpu().numpy(), ids, tokens=sel)
    outs = {}
    for path in paths:
        out = layer.forward(x, tw, tid, path=path)
        torch.cuda.synchronize()
        assert mq.mq_device_status() == 0
        check_forward(out.float().cpu().numpy()[sel], ref, what=f"{what} path={path}")
        outs[path] = out
    return outs


@pytest.fixture(scope="module")
def tiny():
    return Layer(W["tiny"], seed=0)


@pytest.mark.parametrize("T", [1, 2, 5, 8, 9, 16, 17, 37, 64])
def test_decode_tiny(tiny, T):
    x, lg = inputs(tiny.wl, T, seed=100 + T)
    tw, tid = mq.moe_topk_route(lg, tiny.k, True)
    _check_paths(tiny, x, tw, tid, f"tiny T={T}")


@pytest.mark.parametrize("T", [1, 64, 130])
def test_decode_fine_grained(T):
    """E=128, k=8, I=768 (12 K steps of the down GEMM over 4 warps), Zipf
    routing with zero-token experts; T=130 forces the warp-MMA consumers past
    their default batch, with experts of several chunks."""
    layer = Layer(W["fine"], seed=0)
    x, lg = inputs(layer.wl, T, seed=200 + T)
    tw, tid = mq.moe_topk_route(lg, layer.k, True)
    assert len(np.unique(tid.cpu().numpy())) < layer.E  # zero-token experts exist
    _check_paths(layer, x, tw, tid, f"fine T={T}")


def test_decode_hot_expert_spans_chunks(tiny):
    """Every token routes to expert 3 (64 slots: two 32-row chunks stream
    its weights twice), the second slot spread over the others."""
    T = 64
    x, _ = inputs(tiny.wl, T, seed=7)
    lg = synth.router_logits(T, tiny.E, seed=7, device="cuda")
    lg[:, 3] += 20.0
    tw, tid = mq.moe_topk_route(lg, tiny.k, True)
    assert (tid.cpu().numpy()[:, 0] == 3).all()
    _check_paths(tiny, x, tw, tid, "hot expert")


@pytest.mark.parametrize("gs,zp,H,I,T", [(128, True, 256, 384, 11), (256, False, 512, 256, 3),
                                         (128, False, 384, 640, 29), (256, True, 256, 512, 1)])
def test_decode_w4a16(gs, zp, H, I, T):
    wl = synth.Workload(f"w4_dec_gs{gs}", E=6, k=2, H=H, I=I, Ts=(T,), bits=4, group_size=gs,
                        has_zp=zp)
    layer = Layer(wl, seed=gs + H)
    x, lg = inputs(wl, T, seed=gs + T)
    tw, tid = mq.moe_topk_route(lg, wl.k, True)
    _check_paths(layer, x, tw, tid, f"w4a16 gs={gs} zp={zp} T={T}")


def test_decode_w4a16_full_layer():
    """The W4A16 layer (E=64, k=6, H=2048, I=1408 = 11 uint4 K steps over 4
    warps, gs=128) at T=8 on both paths."""
    layer = Layer(W["w4a16"], seed=1)
    x, lg = inputs(layer.wl, 8, seed=8)
    tw, tid = mq.moe_topk_route(lg, layer.k, True)
    _check_paths(layer, x, tw, tid, "w4a16 T=8")


def test_decode_mixtral_sampled():
    """Mixtral-shaped layer (K split of the down GEMM across CTAs) at T=2 on
    both paths, every token."""
    layer = Layer(W["mixtral_decode"], seed=3)
    x, lg = inputs(layer.wl, 2, seed=5)
    tw, tid = mq.moe_topk_route(lg, layer.k, True)
    _check_paths(layer, x, tw, tid, "mixtral T=2")


@pytest.mark.parametrize("name,T", [("tiny", 37), ("fine", 64), ("w4a16", 20)])
def test_decode_deterministic_and_permutation_exact(name, T):
    """Fixed summation order everywhere with warp-MMA consumers: repeated
    calls are bitwise equal, and permuting the batch permutes the output
    bitwise."""
    layer = Layer(W[name], seed=0)
    layer.free_bf16()
    x, lg = inputs(layer.wl, T, seed=9)
    tw, tid = mq.moe_topk_route(lg, layer.k, True)
    outs = [layer.forward(x, tw, tid, path="decode").clone() for _ in range(3)]
    perm = torch.from_numpy(np.random.default_rng(T).permutation(T)).cuda()
    tw_p, tid_p = mq.moe_topk_route(lg[perm].contiguous(), layer.k, True)
    out_p = layer.forward(x[perm].contiguous(), tw_p, tid_p, path="decode")
    torch.cuda.synchronize()
    assert mq.mq_device_status() == 0
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    assert torch.equal(out_p, outs[0][perm])


def test_decode_refuses_small_uint4_groups():
    wl = synth.Workload("w4_gs64", E=4, k=2, H=128, I=128, Ts=(4,), bits=4, group_size=64,
                        has_zp=True)
    layer = Layer(wl, seed=1)
    x, lg = inputs(wl, 4, seed=1)
    tw, tid = mq.moe_topk_route(lg, wl.k, True)
    with pytest.raises(mq.MoeqError) as ei:
        layer.forward(x, tw, tid, path="decode")
    assert ei.value.status == mq.binding.MQ_ERR_UNSUPPORTED
    layer.forward(x, tw, tid)  # the default takes tcgen05 for it
    torch.cuda.synchronize()
    assert mq.mq_device_status() == 0
