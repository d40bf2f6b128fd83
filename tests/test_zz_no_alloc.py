"""The allocation-free forward (moe_w4a16_forward_noalloc) against the
workspace-based moe_w4a16_forward.

The allocation-free call serves callers that cannot allocate device memory
themselves (a plugin whose host application owns the device heap, or a serving
loop that must not call cudaMalloc because it can synchronise the device); it
keeps its scratch in a static array of the library and otherwise runs the same
checks and kernels, so its output must equal moe_w4a16_forward's bit for bit,
for every weight format and reduction order.  This file is collected last so
that a run stopping at the first failure has run every other test.
"""
import dataclasses

import numpy as np
import pytest

import oracle
from w4a16_moe_expert_router_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
REL_FROB = 1e-3


@pytest.fixture(scope="module")
def rt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a16_moe_expert_router_gb300 import build as libbuild
    libbuild.build()
    from w4a16_moe_expert_router_gb300 import runtime
    return runtime


def _case(rt, wl, seed, norm):
    x, lg, w = synth.make_x(wl, seed), synth.make_logits(wl, seed), synth.make_weights(wl, seed)
    dw = rt.upload_weights(wl, w)
    buf = rt.alloc_buffers(wl)
    xd, ld = rt.to_device_x(x), rt.to_device_f32(lg)
    gamma = synth.make_gamma(wl, seed) if norm else None
    gd = rt.to_device_f32(gamma) if norm else None
    ref = rt.run_layer(buf, xd, ld, dw, gd, 1e-6).clone()
    torch.cuda.synchronize()
    return x, lg, w, gamma, dw, buf, xd, gd, ref


def _noalloc_twice(buf, xd, dw, gd, like):
    from w4a16_moe_expert_router_gb300 import binding as B
    outs = []
    for _ in range(2):
        out = torch.full_like(like, float("nan"))
        B.moe_w4a16_forward_noalloc(buf.shape, xd, buf.routing, dw.gate_up, dw.down, gd, 1e-6, out)
        torch.cuda.synchronize()
        outs.append(out)
    return outs


@pytest.mark.parametrize("fmt", [0, 1, 2])
@pytest.mark.parametrize("red", [0, 1])
@pytest.mark.parametrize("norm", [False, True])
def test_noalloc_bit_identical_to_workspace_forward(rt, fmt, red, norm):
    wl = dataclasses.replace(synth.WORKLOADS["tiny"], format=fmt, reduction=red)
    _, _, _, _, dw, buf, xd, gd, ref = _case(rt, wl, 4, norm)
    for out in _noalloc_twice(buf, xd, dw, gd, ref):
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("name", ["canvas64", "canvas256"])
def test_noalloc_bit_identical_full_size(rt, name):
    wl = synth.WORKLOADS[name]
    _, _, _, _, dw, buf, xd, gd, ref = _case(rt, wl, 5, False)
    for out in _noalloc_twice(buf, xd, dw, gd, ref):
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    from w4a16_moe_expert_router_gb300 import binding as B
    assert B.moe_w4a16_noalloc_read_error() == B.OK  # the device-side status of the last call


def test_noalloc_against_the_oracle(rt):
    wl = dataclasses.replace(synth.WORKLOADS["tiny"], format=1)
    x, lg, w, gamma, dw, buf, xd, gd, ref = _case(rt, wl, 6, True)
    idx, tw = oracle.route(lg, wl.top_k)
    want = oracle.forward(x, idx, tw, w, group_gate_up=wl.group_gate_up, group_down=wl.group_down, gamma=gamma,
                          eps=1e-6, fmt=1)
    for out in _noalloc_twice(buf, xd, dw, gd, ref):
        got = out.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got))
        assert np.abs(got - want).max() <= MAX_ABS
        assert np.linalg.norm(got - want) / np.linalg.norm(want) <= REL_FROB


def test_noalloc_rejects_shapes_beyond_its_static_scratch(rt):
    from w4a16_moe_expert_router_gb300 import binding as B
    wl = synth.WORKLOADS["zipf1024"]
    sh = rt.shape_of(wl)
    assert B.moe_w4a16_workspace_bytes(sh) > B.NOALLOC_SCRATCH_BYTES
    with pytest.raises(B.MoeW4A16Error) as e:
        B.moe_w4a16_forward_noalloc(sh, 16, B.RoutingBuffers(16, 16, 16, 16), 16, 16, None, 1e-6, 16)
    assert e.value.status == B.ERR_WORKSPACE
