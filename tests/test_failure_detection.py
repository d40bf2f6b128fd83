"""Failure detection of the device-side waits, without a GPU fault.

Every wait in the expert launch is bounded: on expiry the kernel records
MOE_W4A16_ERR_TIMEOUT in the workspace's error word and returns.  The GPU test
runs the same wait helpers on an mbarrier phase that nothing completes and on a
counter that nothing raises, with a 20 ms bound, checks the reported status, and
then runs a layer on the same context against the oracle: the context stays
usable.  The host test checks the entry point's argument validation.
"""
import ctypes
import os

import numpy as np
import pytest

import oracle
from w4a16_moe_expert_router_gb300 import binding as B
from w4a16_moe_expert_router_gb300 import synth


def test_selftest_arguments_validated_before_any_launch():
    L = B.lib()
    assert L.moe_w4a16_selftest_wait_timeout(None, 4096, 1000000, None) == B.ERR_NULL
    assert L.moe_w4a16_selftest_wait_timeout(4100, 4096, 1000000, None) == B.ERR_ALIGN
    assert L.moe_w4a16_selftest_wait_timeout(4096, 100, 1000000, None) == B.ERR_WORKSPACE
    assert L.moe_w4a16_selftest_wait_timeout(4096, 4096, 0, None) == B.ERR_VALUE
    assert L.moe_w4a16_selftest_wait_timeout(4096, 4096, 3000000000, None) == B.ERR_VALUE


@pytest.mark.gpu
def test_bounded_waits_time_out_and_the_context_stays_usable():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a16_moe_expert_router_gb300 import build as libbuild
    libbuild.build()
    from w4a16_moe_expert_router_gb300 import runtime as rt
    wl = synth.WORKLOADS["tiny"]
    buf = rt.alloc_buffers(wl)
    assert B.moe_w4a16_read_error(buf.workspace) == B.OK
    B.moe_w4a16_selftest_wait_timeout(buf.workspace, 20_000_000)
    torch.cuda.synchronize()
    assert B.moe_w4a16_read_error(buf.workspace) == B.ERR_TIMEOUT
    # cleared by re-initialising the workspace; the next layer on this context is correct
    B.moe_w4a16_workspace_init(buf.workspace)
    x, lg, w = synth.make_x(wl), synth.make_logits(wl), synth.make_weights(wl)
    dw = rt.upload_weights(wl, w)
    rt.run_layer(buf, rt.to_device_x(x), rt.to_device_f32(lg), dw)
    torch.cuda.synchronize()
    assert B.moe_w4a16_read_error(buf.workspace) == B.OK
    idx, tw = oracle.route(lg, wl.top_k)
    ref = oracle.forward(x, idx, tw, w, group_gate_up=wl.group_gate_up, group_down=wl.group_down,
                         activation=wl.activation, nthreads=os.cpu_count() or 1)
    out = buf.out.cpu().numpy().astype(np.float64)
    assert np.abs(out - ref).max() <= 2e-2
    assert np.linalg.norm(out - ref) / np.linalg.norm(ref) <= 1e-3
