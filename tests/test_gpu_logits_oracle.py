"""GPU parity of moe_quant_forward_logits -- the one-call forward the
benchmark times (routing, align, both expert GEMMs, combine) -- against the
oracle, at the benchmark's decode sizes and in its launch configurations.

Each case routes with the oracle from the same logits, and compares a token
sample that holds, for every touched expert, the token of its first and of
its last slot (so the first and the last token tile of every expert are
checked), topped up with random tokens to at least 16; every output column
of every sampled token is compared.  The sizes span the kernels' plans:
16-token tiles with two MMA issuers and split-K 4-8 in the down GEMM
(Mixtral-shaped T = 1, 8, 32), 64-token tiles (T = 64), the fused router in
the align kernel (small T·k·ceil(E/32)) and the separate router kernel
(fine-grained T = 512), and the uint4 path at T = 1 to 192 (16- and 32-row
tiles) -- each with the
default kernels (tcgen05 consumers; one launch for both GEMMs of the
fine-grained layer at T = 512), with the warp-level-MMA consumers forced
for both GEMMs, and (8-bit) with both GEMMs forced into one launch.
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


def sample_tokens(ids, n_min=16, seed=0):
    """Tokens of every expert's first and last slot (slot s = t * k + j, in
    slot order within the expert's segment), plus random ones up to n_min."""
    T, k = ids.shape
    flat = ids.reshape(-1)
    chosen = set()
    for e in np.unique(flat):
        slots = np.nonzero(flat == e)[0]
        chosen.add(int(slots[0]) // k)
        chosen.add(int(slots[-1]) // k)
    rng = np.random.default_rng(seed)
    rest = [t for t in range(T) if t not in chosen]
    rng.shuffle(rest)
    while len(chosen) < min(n_min, T):
        chosen.add(rest.pop())
    return np.array(sorted(chosen))


def _logits_case(layer, T, seed, path="auto"):
    x, lg = inputs(layer.wl, T, seed)
    out = mq.moe_quant_forward_logits(x, lg, layer.q13, layer.q2, layer.s13, layer.s2, layer.k,
                                      layer.wl.renormalize, bits=layer.bits, group_size=layer.gs,
                                      has_zp=layer.has_zp, z13=layer.z13, z2=layer.z2, path=path)
    torch.cuda.synchronize()
    assert mq.mq_device_status() == 0
    ow, oid = oracle.topk_route(lg.cpu().numpy(), layer.k, layer.wl.renormalize)
    # the library's router decides the same ids (bit-exact)
    _, tid = mq.moe_topk_route(lg, layer.k, layer.wl.renormalize)
    assert np.array_equal(tid.cpu().numpy(), oid)
    sel = sample_tokens(oid, seed=T)
    ex = layer.oracle_experts(np.unique(oid[sel]))
    ref = oracle.moe_forward(x.float().cpu().numpy(), ex, ow, oid, tokens=sel)
    got = out.float().cpu().numpy()[sel]
    return check_forward(got, ref, what=f"{layer.wl.name} T={T} path={path} ({sel.size} tokens)")


@pytest.fixture(scope="module")
def mixtral():
    layer = Layer(W["mixtral_decode"], seed=0)
    yield layer
    del layer
    torch.cuda.empty_cache()


@pytest.mark.parametrize("path", ["auto", "decode", "layer"])
@pytest.mark.parametrize("T", [1, 8, 32, 64])
def test_logits_forward_mixtral_decode(mixtral, T, path):
    _logits_case(mixtral, T, seed=20 + T, path=path)


@pytest.mark.parametrize("path", ["auto", "tc", "decode", "layer"])
@pytest.mark.parametrize("T", [1, 24, 64, 512])
def test_logits_forward_fine_grained(T, path):
    layer = Layer(W["fine"], seed=0)
    _logits_case(layer, T, seed=30 + T, path=path)


@pytest.mark.parametrize("path", ["auto", "decode"])
@pytest.mark.parametrize("T", [1, 32, 48, 64])
def test_logits_forward_w4a16(T, path):
    layer = Layer(W["w4a16"], seed=0)
    _logits_case(layer, T, seed=40 + T, path=path)


@pytest.mark.parametrize("T", [128, 192])
def test_logits_forward_w4a16_mid_batches(T):
    """32-row uint4 tiles beyond 64 tokens (mean slots per expert 12 and 18)."""
    layer = Layer(W["w4a16"], seed=0)
    _logits_case(layer, T, seed=40 + T)


def test_sample_tokens_covers_first_and_last_slot():
    """The sampler itself: every expert's first and last slot's token is in."""
    ids = np.array([[0, 1], [1, 2], [0, 2], [3, 1], [2, 0]])
    # expert 0: slots 0, 4, 9 -> tokens 0, 4; expert 1: slots 1, 2, 7 -> 0, 3;
    # expert 2: slots 3, 5, 8 -> 1, 4; expert 3: slot 6 -> 3
    assert sample_tokens(ids, n_min=0).tolist() == [0, 1, 3, 4]
    assert len(sample_tokens(ids, n_min=5)) == 5
