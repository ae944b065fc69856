"""GPU parity of the quantisers, the router and the block alignment against
the oracle: bit-exact codes, scales, ids and align arrays."""

import numpy as np
import pytest
import torch

import oracle
from moe_helpers import route_tolerance

pytestmark = pytest.mark.gpu

mq = pytest.importorskip("weight_quantized_moe_gb300")


def _bf16(shape, seed, std=0.02, device="cuda"):
    g = torch.Generator(device=device).manual_seed(seed)
    return (torch.randn(*shape, generator=g, device=device) * std).to(torch.bfloat16)


# ------------------------------------------------------------- quantisers --
@pytest.mark.parametrize("rows,cols", [(1, 8), (5, 136), (513, 4096), (8 * 512, 128), (33, 14336)])
def test_quant_int8_bit_exact(rows, cols):
    w = _bf16((rows, cols), seed=rows + cols)
    w[rows // 2] = 0                                          # an all-zero row
    q, s = mq.moe_quantize_int8_per_channel(w)
    oq, os_ = oracle.quantize_int8_per_channel(w.float().cpu().numpy())
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), os_.view(np.uint32))


def test_quant_int8_special_values():
    """Exact ties, tiny (subnormal-scale) rows and large rows."""
    rows = [
        [0.9921875, 0.5, -0.25, 0.01171875, 0.01953125, -0.02734375, 0.0, -0.0078125],
        [1e-38, -3e-39, 5e-39, 0, 0, 0, 0, 0],
        [3.0e38, -1.5e38, 1.0, 0, 0, 0, 0, 0],
        [-0.0, 0.0, 0, 0, 0, 0, 0, 0],
    ]
    w = torch.tensor(rows, dtype=torch.float32).to(torch.bfloat16).cuda()
    q, s = mq.moe_quantize_int8_per_channel(w)
    oq, os_ = oracle.quantize_int8_per_channel(w.float().cpu().numpy())
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), os_.view(np.uint32))


def test_quant_int8_full_mixtral_w13_sampled_rows():
    """Full Mixtral-sized w13 ([8 * 28672, 4096]) quantised in one call;
    1024 sampled rows compared with the oracle."""
    from weight_quantized_moe_gb300 import synth
    w = synth.expert_weights(8, 2 * 14336, 4096, seed=0, which="w13", device="cuda")
    q, s = mq.moe_quantize_int8_per_channel(w)
    rows = np.random.default_rng(0).choice(8 * 2 * 14336, 1024, replace=False)
    wf = w.reshape(-1, 4096)[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    oq, os_ = oracle.quantize_int8_per_channel(wf)
    assert np.array_equal(q.reshape(-1, 4096)[torch.from_numpy(rows).cuda()].cpu().numpy(), oq)
    assert np.array_equal(s.reshape(-1)[torch.from_numpy(rows).cuda()].cpu().numpy(), os_)


@pytest.mark.parametrize("gs", [32, 64, 128, 256])
@pytest.mark.parametrize("rows,cols", [(2, 256), (6, 512), (130, 2048)])
def test_quant_uint4_bit_exact(gs, rows, cols):
    w = _bf16((rows, cols), seed=gs + rows)
    w[1, :gs] = 0                                             # an all-zero group
    qw, sc, qz = mq.moe_quantize_uint4_group(w, gs)
    q, s, z = oracle.quantize_uint4_group(w.float().cpu().numpy(), gs)
    assert np.array_equal(qw.cpu().numpy(), oracle.pack_uint4_along_k(q))
    assert np.array_equal(sc.cpu().numpy().view(np.uint16), s.view(np.uint16))
    assert np.array_equal(qz.cpu().numpy(), oracle.pack_uint4_along_n(z))


# ------------------------------------------------------------------ router --
@pytest.mark.parametrize("T,E,k,renorm", [(16, 8, 2, True), (37, 8, 2, False), (64, 128, 8, True),
                                          (1000, 64, 6, True), (3, 1024, 32, True), (5, 32, 32, True),
                                          (4096, 128, 8, True)])
def test_route_parity(T, E, k, renorm):
    from weight_quantized_moe_gb300 import synth
    lg = synth.router_logits(T, E, seed=T + E, bias="zipf" if E >= 64 else None)
    w, ids = mq.moe_topk_route(lg.cuda(), k, renorm)
    ow, oid = oracle.topk_route(lg.numpy(), k, renorm)
    assert np.array_equal(ids.cpu().numpy(), oid)
    np.testing.assert_allclose(w.cpu().numpy(), ow, rtol=route_tolerance(E), atol=0)


def test_route_ties_and_constant_logits():
    lg = torch.zeros(4, 16)
    lg[1, 3] = lg[1, 9] = 2.0
    lg[2] = torch.tensor([-0.0, 0.0] * 8)
    w, ids = mq.moe_topk_route(lg.cuda(), 4, True)
    ow, oid = oracle.topk_route(lg.numpy(), 4, True)
    assert np.array_equal(ids.cpu().numpy(), oid)
    np.testing.assert_allclose(w.cpu().numpy(), ow, rtol=route_tolerance(16))


def test_route_empty():
    w, ids = mq.moe_topk_route(torch.zeros(0, 8, device="cuda"), 2, True)
    assert w.shape == (0, 2)


# ------------------------------------------------------------------- align --
@pytest.mark.parametrize("T,k,E,bm", [(16, 2, 8, 16), (1, 2, 8, 16), (37, 3, 5, 4), (64, 8, 128, 16),
                                      (8192, 2, 8, 128), (4096, 8, 128, 64), (2048, 6, 64, 128),
                                      (100, 1, 1024, 1), (0, 2, 8, 16)])
def test_align_bit_exact(T, k, E, bm):
    rng = np.random.default_rng(T * 7 + E)
    # skewed expert popularity so that some experts get nothing
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    ids = np.stack([rng.choice(E, size=k, replace=False, p=p / p.sum()) for _ in range(T)]) \
        if T else np.zeros((0, k), np.int64)
    ids = ids.astype(np.int32)
    sorted_ids, blocks, offsets, npad = mq.moe_align_block(torch.from_numpy(ids).cuda(), E, bm)
    r = oracle.align_block(ids, E, bm)
    n = int(npad.item())
    assert n == r.num_padded
    assert np.array_equal(sorted_ids.cpu().numpy()[:n], r.sorted_slot_ids)
    assert np.array_equal(blocks.cpu().numpy()[:n // bm], r.block_expert)
    assert np.array_equal(offsets.cpu().numpy(), r.expert_offsets)
    assert mq.mq_device_status() == 0


def test_align_flags_invalid_ids():
    ids = np.array([[2, 2], [0, 2], [7, -1]], dtype=np.int32)
    sorted_ids, blocks, offsets, npad = mq.moe_align_block(torch.from_numpy(ids).cuda(), 4, 2)
    r = oracle.align_block(ids, 4, 2)
    assert mq.mq_device_status() == mq.MQ_DEV_BAD_EXPERT_ID
    assert mq.mq_device_status() == 0                         # read clears
    n = int(npad.item())
    assert np.array_equal(sorted_ids.cpu().numpy()[:n], r.sorted_slot_ids)
    assert np.array_equal(offsets.cpu().numpy(), r.expert_offsets)
