"""GPU parity of moe_quant_forward (route + align + expert GEMMs + combine)
against the oracle, within the forward tolerance of moe_helpers."""

import numpy as np
import pytest
import torch

import oracle
from moe_helpers import FWD_TOL, Layer, check_forward, forward_error, inputs, plain_error
from weight_quantized_moe_gb300 import synth

pytestmark = pytest.mark.gpu

mq = pytest.importorskip("weight_quantized_moe_gb300")

W = synth.WORKLOADS


def _run(layer, T, seed=0, tokens=None, out_cols=None, renorm=True):
    x, lg = inputs(layer.wl, T, seed)
    tw, tid = mq.moe_topk_route(lg, layer.k, renorm)
    out = layer.forward(x, tw, tid)
    torch.cuda.synchronize()
    assert mq.mq_device_status() == 0
    ids = tid.cpu().numpy()
    ow, oid = oracle.topk_route(lg.cpu().numpy(), layer.k, renorm)
    assert np.array_equal(ids, oid)
    sel = np.arange(T) if tokens is None else np.asarray(tokens)
    ex = layer.oracle_experts(np.unique(ids[sel]))
    ref = oracle.moe_forward(x.float().cpu().numpy(), ex, ow, oid, tokens=sel, out_cols=out_cols)
    got = out.float().cpu().numpy()[sel]
    if out_cols is not None:
        got = got[:, out_cols]
    return check_forward(got, ref, what=f"{layer.wl.name} T={T}")[0]


@pytest.fixture(scope="module")
def tiny():
    return Layer(W["tiny"], seed=0)


@pytest.mark.parametrize("T", [16, 1, 37, 300])
def test_forward_tiny(tiny, T):
    assert _run(tiny, T, seed=T) <= FWD_TOL


def test_forward_tiny_no_renormalise(tiny):
    assert _run(tiny, 16, seed=5, renorm=False) <= FWD_TOL


def test_forward_k_equals_e_identical_experts():
    """Dense-MLP identity on the GPU: k = E, equal logits."""
    wl = synth.Workload("dense", E=4, k=4, H=128, I=128, Ts=(8,))
    layer = Layer(wl, seed=3)
    w13, w2 = layer._bf16
    w13[1:] = w13[0]
    w2[1:] = w2[0]
    layer.q13, layer.s13 = mq.moe_quantize_int8_per_channel(w13)
    layer.q2, layer.s2 = mq.moe_quantize_int8_per_channel(w2)
    x = synth.hidden_states(8, 128, seed=1, device="cuda")
    lg = torch.zeros(8, 4, device="cuda")
    tw, tid = mq.moe_topk_route(lg, 4, True)
    out = layer.forward(x, tw, tid).float().cpu().numpy()
    ex = layer.oracle_experts([0])
    W13, W2 = ex.deq13(0), ex.deq2(0)
    h = x.float().cpu().numpy().astype(np.float64) @ W13.T
    ref = (oracle.silu(h[:, :128]) * h[:, 128:]) @ W2.T
    check_forward(out, ref, what="dense identity")


def test_forward_zero_input(tiny):
    x = torch.zeros(4, 128, dtype=torch.bfloat16, device="cuda")
    tw, tid = mq.moe_topk_route(synth.router_logits(4, 8, 1, device="cuda"), 2, True)
    assert torch.count_nonzero(tiny.forward(x, tw, tid)).item() == 0


def test_forward_invalid_ids_flagged(tiny):
    x, lg = inputs(tiny.wl, 6, seed=9)
    tw, tid = mq.moe_topk_route(lg, 2, True)
    tid[1, 1] = 8
    tid[4, 0] = -3
    out = tiny.forward(x, tw, tid)
    assert mq.mq_device_status() == mq.MQ_DEV_BAD_EXPERT_ID
    ids = tid.cpu().numpy()
    ex = tiny.oracle_experts()
    ref = oracle.moe_forward(x.float().cpu().numpy(), ex, tw.cpu().numpy(), ids)
    check_forward(out.float().cpu().numpy(), ref, what="invalid ids")


def test_forward_empty_batch(tiny):
    x = torch.zeros(0, 128, dtype=torch.bfloat16, device="cuda")
    tw = torch.zeros(0, 2, device="cuda")
    tid = torch.zeros(0, 2, dtype=torch.int32, device="cuda")
    assert tiny.forward(x, tw, tid).shape == (0, 128)


@pytest.mark.parametrize("path", ["auto", "tc", "decode", "layer"])
def test_logits_forward_empty_batch(tiny, path):
    """T = 0 through the one-call forward on every path: an empty output,
    no launch that reads a token, and a clean device status."""
    x = torch.zeros(0, tiny.H, dtype=torch.bfloat16, device="cuda")
    lg = torch.zeros(0, tiny.E, dtype=torch.float32, device="cuda")
    out = mq.moe_quant_forward_logits(x, lg, tiny.q13, tiny.q2, tiny.s13, tiny.s2, tiny.k, True,
                                      path=path)
    torch.cuda.synchronize()
    assert out.shape == (0, tiny.H)
    assert mq.mq_device_status() == 0


def test_forward_empty_batch_uint4():
    wl = synth.Workload("w4a16_empty", E=6, k=2, H=256, I=384, Ts=(0,), bits=4, group_size=128,
                        has_zp=True)
    layer = Layer(wl, seed=5)
    x = torch.zeros(0, wl.H, dtype=torch.bfloat16, device="cuda")
    tw = torch.zeros(0, wl.k, device="cuda")
    tid = torch.zeros(0, wl.k, dtype=torch.int32, device="cuda")
    out = layer.forward(x, tw, tid)
    torch.cuda.synchronize()
    assert out.shape == (0, wl.H)
    assert mq.mq_device_status() == 0


@pytest.mark.parametrize("bits,T", [(8, 50), (8, 300), (4, 50)])
def test_forward_single_expert(bits, T):
    """E = 1, k = 1: the MoE layer is one dense MLP whose router weight is 1;
    every token lands in the one expert's segment (several token tiles)."""
    wl = synth.Workload(f"dense_b{bits}_T{T}", E=1, k=1, H=256, I=384, Ts=(T,), bits=bits,
                        group_size=128 if bits == 4 else -1, has_zp=bits == 4)
    layer = Layer(wl, seed=T + bits)
    assert _run(layer, T, seed=T) <= FWD_TOL


@pytest.mark.parametrize("T", [16, 64, 128, 256])
def test_forward_hot_expert_fills_whole_tiles(tiny, T):
    """Every token's first choice is expert 5, so its segment holds exactly T
    slots: a whole number of token tiles (16, 32 or 128 rows), no ragged
    tail, with the second choices spread over the other experts."""
    x, _ = inputs(tiny.wl, T, seed=T + 7)
    lg = synth.router_logits(T, tiny.E, seed=T + 7, device="cuda")
    lg[:, 5] += 20.0
    tw, tid = mq.moe_topk_route(lg, tiny.k, True)
    ids = tid.cpu().numpy()
    assert (ids[:, 0] == 5).all() and (ids[:, 1] != 5).all()
    out = tiny.forward(x, tw, tid)
    torch.cuda.synchronize()
    assert mq.mq_device_status() == 0
    ex = tiny.oracle_experts(np.unique(ids))
    ref = oracle.moe_forward(x.float().cpu().numpy(), ex, tw.cpu().numpy(), ids)
    check_forward(out.float().cpu().numpy(), ref, what=f"hot expert T={T}")


@pytest.mark.parametrize("bits", [8, 4])
def test_forward_128_row_tiles_with_k_splits(bits):
    """Two experts, H = 512, I = 4096, T = 100: 128-row token tiles, and
    the down GEMM split eight ways over K to fill the SMs (the split rule of
    batches beyond 64 tokens)."""
    wl = synth.Workload(f"split_b{bits}", E=2, k=1, H=512, I=4096, Ts=(100,), bits=bits,
                        group_size=128 if bits == 4 else -1, has_zp=bits == 4)
    layer = Layer(wl, seed=bits)
    assert _run(layer, 100, seed=3) <= FWD_TOL


def test_forward_fine_grained_full():
    """E=128, k=8, H=2048, I=768 with Zipf-skewed routing (zero-token experts)."""
    layer = Layer(W["fine"], seed=0)
    assert _run(layer, 64, seed=1) <= FWD_TOL


def test_forward_w4a16():
    wl = synth.Workload("w4a16_small", E=8, k=3, H=256, I=384, Ts=(24,), bits=4, group_size=128,
                        has_zp=True)
    layer = Layer(wl, seed=2)
    assert _run(layer, 24, seed=2) <= FWD_TOL


@pytest.mark.parametrize("gs,zp,H,I", [(64, False, 256, 384), (32, True, 128, 256),
                                       (256, True, 512, 256), (128, True, 384, 640)])
def test_forward_w4a16_group_sizes(gs, zp, H, I):
    """Group sizes 32..256, implicit zero point (8), and K not a multiple of
    256 (a half-filled last weight stage)."""
    wl = synth.Workload(f"w4a16_gs{gs}", E=6, k=2, H=H, I=I, Ts=(20,), bits=4, group_size=gs,
                        has_zp=zp)
    layer = Layer(wl, seed=gs)
    assert _run(layer, 20, seed=gs) <= FWD_TOL


@pytest.mark.parametrize("E,k,H,I,gs,zp,T", [(6, 2, 256, 384, 128, True, 48),
                                              (20, 3, 640, 384, 128, False, 64),
                                              (20, 4, 384, 256, 64, True, 120),
                                              (20, 10, 640, 384, 128, False, 64)])
def test_forward_w4a16_tile_shapes(E, k, H, I, gs, zp, T):
    """uint4 tile widths: 32 rows (up to 16 experts, 33-64 tokens), 16 and
    32 rows for layers of more experts while the mean slots per expert stay
    below 10 and 28 (T = 64 and T = 120 here), 64 rows beyond that (k = 10
    of 20 experts at T = 64: one accumulator buffer, three stages); units of
    one, two and three MMA steps, the last stage of a unit half-filled
    (K = 384, 640).

    These layers are small (the down GEMM sums 256 to 384 products per
    output), and the act intermediate's bf16 rounding alone then reaches the
    bound at the outliers (E=20, I=256, T=120: 1.1e-2 of the RMS against the
    exact oracle, the same with every tile width).  As for the format
    variants, the bound is checked against the oracle with that rounding
    modelled; the error against the exact oracle is printed beside it."""
    wl = synth.Workload(f"w4a16_E{E}_T{T}", E=E, k=k, H=H, I=I, Ts=(T,), bits=4, group_size=gs,
                        has_zp=zp)
    layer = Layer(wl, seed=E + T)
    x, lg = inputs(wl, T, T)
    tw, tid = mq.moe_topk_route(lg, k, True)
    out = layer.forward(x, tw, tid)
    torch.cuda.synchronize()
    assert mq.mq_device_status() == 0
    ids = tid.cpu().numpy()
    ow, oid = oracle.topk_route(lg.cpu().numpy(), k, True)
    assert np.array_equal(ids, oid)
    ex = layer.oracle_experts(np.unique(ids))
    xf = x.float().cpu().numpy()
    got = out.float().cpu().numpy()
    exact = oracle.moe_forward(xf, ex, ow, oid)
    ref = oracle.moe_forward(xf, ex, ow, oid, intermediate="bf16")
    check_forward(got, ref, what=f"{wl.name} vs the bf16-intermediate oracle (forward error "
                  f"{forward_error(got, exact):.3e}, plain {plain_error(got, exact):.3e} vs the "
                  f"exact oracle);")


@pytest.mark.parametrize("T", [24, 40, 100])
def test_forward_int8_tile_shapes_many_experts(T):
    """8-bit layer of 20 experts (more than 16) with K = 384 and 640 (a
    half-filled last stage): 32-row tiles from 17 tokens, 64-row tiles from
    33, 128-row tiles (one launch for both GEMMs) beyond 64."""
    wl = synth.Workload(f"int8_E20_T{T}", E=20, k=4, H=384, I=640, Ts=(T,))
    layer = Layer(wl, seed=T)
    assert _run(layer, T, seed=T + 1) <= FWD_TOL


def test_forward_w4a16_full_sampled():
    """The full W4A16 layer (E=64, k=6, H=2048, I=1408, gs=128) at T=32."""
    layer = Layer(W["w4a16"], seed=0)
    assert _run(layer, 32, seed=3, tokens=[0, 7, 31]) <= FWD_TOL


@pytest.mark.parametrize("name,T", [("mixtral_decode", 64), ("fine", 64), ("w4a16", 32),
                                    ("w4a16", 64), ("mixtral_prefill", 1024)])
def test_forward_is_deterministic(name, T):
    """No atomics anywhere: repeated calls give bitwise identical outputs
    (a check that no kernel reads data before it has landed)."""
    layer = Layer(W[name], seed=0)
    layer.free_bf16()
    x, lg = inputs(layer.wl, T, seed=4)
    tw, tid = mq.moe_topk_route(lg, layer.k, True)
    outs = [layer.forward(x, tw, tid).clone() for _ in range(4)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


@pytest.mark.parametrize("name,T", [("mixtral_decode", 64), ("fine", 256), ("w4a16", 64),
                                    ("w4a16", 256), ("mixtral_prefill", 1024)])
def test_forward_token_permutation_is_exact(name, T):
    """Each token's output depends only on its own row: every GEMM column is
    an independent dot product in a fixed K order, and the combine sums a
    token's slots in a fixed order.  Permuting the batch therefore permutes
    the output bitwise, although the tokens land in other blocks and block
    positions.  (Any read of a stage before its data landed breaks this.)"""
    layer = Layer(W[name], seed=0)
    layer.free_bf16()
    x, lg = inputs(layer.wl, T, seed=6)
    perm = torch.from_numpy(np.random.default_rng(T).permutation(T)).cuda()
    tw, tid = mq.moe_topk_route(lg, layer.k, True)
    out = layer.forward(x, tw, tid)
    tw_p, tid_p = mq.moe_topk_route(lg[perm].contiguous(), layer.k, True)
    out_p = layer.forward(x[perm].contiguous(), tw_p, tid_p)
    torch.cuda.synchronize()
    assert mq.mq_device_status() == 0
    assert torch.equal(out_p, out[perm])


def test_forward_mixtral_decode_sampled():
    """Mixtral-shaped layer at T=64, the benchmarked decode size: two sampled
    tokens, 512 sampled output columns."""
    layer = Layer(W["mixtral_decode"], seed=0)
    cols = np.sort(np.random.default_rng(0).choice(4096, 512, replace=False))
    assert _run(layer, 64, seed=0, tokens=[5, 40], out_cols=cols) <= FWD_TOL


@pytest.mark.parametrize("name,T,tokens", [("mixtral_prefill", 1024, [0, 511, 1023]),
                                           ("mixtral_prefill", 4096, [0, 2047, 4095]),
                                           ("mixtral_prefill", 8192, [0, 5000, 8191]),
                                           ("fine", 4096, [1, 3000]),
                                           ("w4a16", 2048, [5, 2047])])
def test_forward_prefill_sizes_sampled(name, T, tokens):
    """The prefill-sized layers in their default launch configuration
    (128-token tiles; the down GEMM split over K in two at T=1024 on the
    Mixtral-shaped layer, unsplit beyond; 16,384 token-slots sorted at
    T=8192): sampled tokens and 512 sampled output columns against the
    oracle."""
    layer = Layer(W[name], seed=0)
    cols = np.sort(np.random.default_rng(T).choice(layer.H, 512, replace=False))
    assert _run(layer, T, seed=5, tokens=tokens, out_cols=cols) <= FWD_TOL


def test_forward_captures_into_a_cuda_graph():
    """The whole forward (routing included) launches only kernels, with no
    host synchronisation or allocation, so it can be captured into a CUDA
    graph; replays reproduce the eager result bitwise."""
    layer = Layer(W["mixtral_decode"], seed=0)
    layer.free_bf16()
    x, lg = inputs(layer.wl, 8, seed=12)
    ws = torch.empty(mq.lib().moe_quant_forward_logits_workspace(8, layer.H, layer.I, layer.E,
                                                                 layer.k, 8, -1),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty(8, layer.H, dtype=torch.bfloat16, device="cuda")
    fwd = lambda: mq.moe_quant_forward_logits(x, lg, layer.q13, layer.q2, layer.s13, layer.s2,
                                              layer.k, True, workspace=ws, out=out)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fwd()
    torch.cuda.current_stream().wait_stream(s)
    ref = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fwd()
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert mq.mq_device_status() == 0
    assert torch.equal(out, ref)


@pytest.mark.parametrize("E,k,T", [(1024, 32, 5), (1024, 1, 16), (33, 32, 3)])
def test_forward_maximum_experts_and_top_k(E, k, T):
    """The ABI limits: E = 1024 experts, top_k = 32 (and k = E - 1 < 32
    with an odd expert count)."""
    wl = synth.Workload("edge", E=E, k=k, H=128, I=128, Ts=(T,))
    layer = Layer(wl, seed=4)
    assert _run(layer, T, seed=E + k) <= FWD_TOL


def test_bench_end_to_end_loop_delivers_each_output():
    """The benchmark's pipelined serving loop (uploads and downloads on their
    own streams, two buffers of each) leaves every step's output on the host
    equal to the forward's result."""
    import bench
    prob = bench.Problem(W["tiny"], 16, seed=3)
    ref = prob.step().clone()
    run = bench.EndToEnd(prob)
    for _ in range(5):
        run.step()
    run.finish()
    torch.cuda.synchronize()
    assert mq.mq_device_status() == 0
    for h in run.out_h:
        assert torch.equal(h, ref.cpu())
