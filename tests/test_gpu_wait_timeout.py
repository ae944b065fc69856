"""The bounded waits, exercised on the GPU without a fault: the testing hook
mq_test_layer_wait_extra makes the one-launch layer's down units wait for
gate/up completions that never come.  Each such wait gives up after its
limit of about a second; the kernel then stops its CTAs cleanly (their
copies and MMAs drained, tensor memory freed), the status word reports
MQ_DEV_WAIT_TIMEOUT, and the next forward on the same context runs
normally and matches the oracle."""

import time

import numpy as np
import pytest
import torch

import oracle
from moe_helpers import Layer, check_forward, inputs
from weight_quantized_moe_gb300 import synth

pytestmark = pytest.mark.gpu

mq = pytest.importorskip("weight_quantized_moe_gb300")


def test_layer_wait_runs_out_and_context_recovers():
    layer = Layer(synth.WORKLOADS["tiny"], seed=0)
    T = 40
    x, lg = inputs(layer.wl, T, seed=5)
    tw, tid = mq.moe_topk_route(lg, layer.k, True)
    ref_out = layer.forward(x, tw, tid, path="layer").clone()
    torch.cuda.synchronize()
    assert mq.mq_device_status() == 0

    mq.mq_test_layer_wait_extra(1)
    try:
        t0 = time.monotonic()
        layer.forward(x, tw, tid, path="layer")
        torch.cuda.synchronize()
        waited = time.monotonic() - t0
    finally:
        mq.mq_test_layer_wait_extra(0)
    assert mq.mq_device_status() & mq.binding.MQ_DEV_WAIT_TIMEOUT
    assert waited < 30.0  # every wait is bounded

    # the context is usable: the same forward again, bitwise as before, and
    # against the oracle
    out = layer.forward(x, tw, tid, path="layer")
    torch.cuda.synchronize()
    assert mq.mq_device_status() == 0
    assert torch.equal(out, ref_out)
    ids = tid.cpu().numpy()
    ex = layer.oracle_experts(np.unique(ids))
    ref = oracle.moe_forward(x.float().cpu().numpy(), ex, tw.cpu().numpy(), ids)
    check_forward(out.float().cpu().numpy(), ref, what="after the timed-out launch")
