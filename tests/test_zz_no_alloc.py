"""moe_quant_forward_noalloc against moe_quant_forward, on the GPU.

The no-allocation entry point serves callers that cannot allocate device
memory or pass a workspace (for example a plugin whose host application owns
all device memory).  It runs the same forward with its scratch in a fixed
array inside the library, so its output must match the workspace version.
Two calls in a row with different batches check that nothing stale from the
first call leaks into the second.  This file is collected last on purpose.
"""

import ctypes

import pytest
import torch

from moe_helpers import Layer, inputs
from weight_quantized_moe_gb300 import synth

pytestmark = pytest.mark.gpu

mq = pytest.importorskip("weight_quantized_moe_gb300")


def _noalloc_via_cabi(layer, x, tw, tid):
    """Call the C entry point directly through ctypes."""
    from weight_quantized_moe_gb300 import binding
    L = binding.lib()
    out = torch.empty(x.shape[0], layer.H, dtype=torch.bfloat16, device=x.device)
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    status = L.moe_quant_forward_noalloc(
        p(x), x.shape[0], layer.H, layer.I, layer.E, layer.k, layer.bits, layer.gs,
        int(layer.has_zp), p(layer.q13), p(layer.q2), p(layer.s13), p(layer.s2), p(layer.z13),
        p(layer.z2), p(tw), p(tid), p(out), st)
    return status, out


@pytest.mark.parametrize("name,Ts", [("mixtral_decode", (64, 8)), ("fine", (64, 37)),
                                     ("w4a16", (32, 7))])
def test_noalloc_matches_workspace_forward_twice(name, Ts):
    """Both calls run the same kernels on the same inputs as the workspace
    forward, so the outputs must be bitwise equal; the second, smaller call
    finds the first call's data in the shared scratch (the uint4 case also
    rewrites its act rows in place there)."""
    layer = Layer(synth.WORKLOADS[name], seed=0)
    layer.free_bf16()
    for call, T in enumerate(Ts):
        x, lg = inputs(layer.wl, T, seed=10 + call)
        tw, tid = mq.moe_topk_route(lg, layer.k, True)
        ref = layer.forward(x, tw, tid)
        status, got = _noalloc_via_cabi(layer, x, tw, tid)
        assert status == 0, mq.binding.lib().mq_last_error_message().decode()
        torch.cuda.synchronize()
        assert mq.mq_device_status() == 0
        assert torch.equal(got, ref), (name, call, T)


def test_noalloc_python_wrapper_matches_workspace_forward():
    """The binding's wrapper of the same entry point (argument checks, then
    the C call) gives the workspace forward's result."""
    layer = Layer(synth.WORKLOADS["w4a16"], seed=1)
    layer.free_bf16()
    x, lg = inputs(layer.wl, 5, seed=3)
    tw, tid = mq.moe_topk_route(lg, layer.k, True)
    ref = layer.forward(x, tw, tid)
    got = mq.binding.moe_quant_forward_noalloc(x, layer.q13, layer.q2, layer.s13, layer.s2, tw,
                                               tid, bits=4, group_size=layer.gs, has_zp=True,
                                               z13=layer.z13, z2=layer.z2)
    torch.cuda.synchronize()
    assert mq.mq_device_status() == 0
    assert torch.equal(got, ref)


def test_noalloc_rejects_oversized_batch():
    """Scratch larger than the fixed array is refused before any launch."""
    from weight_quantized_moe_gb300 import binding
    L = binding.lib()
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: rejected on the host
    status = L.moe_quant_forward_noalloc(fake, 8192, 4096, 14336, 8, 2, 8, -1, 0, fake, fake,
                                         fake, fake, None, None, fake, fake,
                                         ctypes.c_void_p(0x10000000), None)
    assert status == binding.MQ_ERR_UNSUPPORTED
    assert b"scratch" in L.mq_last_error_message()


def test_noalloc_python_wrapper_rejects_strided_weights():
    """A transposed (non-contiguous) weight view is refused by the wrapper's
    checks before its pointer reaches the library."""
    layer = Layer(synth.WORKLOADS["tiny"], seed=0)
    x, lg = inputs(layer.wl, 4, seed=1)
    tw, tid = mq.moe_topk_route(lg, layer.k, True)
    bad = layer.q13.transpose(1, 2)
    with pytest.raises(ValueError, match="contiguous"):
        mq.binding.moe_quant_forward_noalloc(x, bad, layer.q2, layer.s13, layer.s2, tw, tid)
