"""The allocation-free forward (moe_w4a16_forward_noalloc) against the
workspace-based moe_w4a16_forward.

The allocation-free call serves callers that cannot allocate device memory
themselves (a plugin whose host application owns the device heap, or a serving
loop that must not call cudaMalloc because it can synchronise the device); it
keeps its scratch in a static array of the library.  This file is collected
last so that a run stopping at the first failure has run every other test.
"""
import numpy as np
import pytest

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


@pytest.mark.parametrize("name,norm", [("tiny", False), ("tiny", True), ("canvas256", False)])
def test_noalloc_matches_workspace_forward_on_two_calls(rt, name, norm):
    from w4a16_moe_expert_router_gb300 import binding as B
    wl = synth.WORKLOADS[name]
    x, lg, w = synth.make_x(wl, 4), synth.make_logits(wl, 4), synth.make_weights(wl, 4)
    dw = rt.upload_weights(wl, w)
    buf = rt.alloc_buffers(wl)
    xd, ld = rt.to_device_x(x), rt.to_device_f32(lg)
    gamma = rt.to_device_f32(synth.make_gamma(wl, 4)) if norm else None
    ref = rt.run_layer(buf, xd, ld, dw, gamma, 1e-6).clone()
    torch.cuda.synchronize()
    refd = ref.cpu().numpy().astype(np.float64)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        B.moe_w4a16_forward_noalloc(buf.shape, xd, buf.routing, dw.gate_up, dw.down, gamma, 1e-6, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got))
        assert np.abs(got - refd).max() <= MAX_ABS
        assert np.linalg.norm(got - refd) / np.linalg.norm(refd) <= REL_FROB


def test_noalloc_rejects_shapes_beyond_its_static_scratch(rt):
    from w4a16_moe_expert_router_gb300 import binding as B
    wl = synth.WORKLOADS["zipf1024"]
    sh = rt.shape_of(wl)
    assert B.moe_w4a16_workspace_bytes(sh) > B.NOALLOC_SCRATCH_BYTES
    with pytest.raises(B.MoeW4A16Error) as e:
        B.moe_w4a16_forward_noalloc(sh, 16, B.RoutingBuffers(16, 16, 16, 16), 16, 16, None, 1e-6, 16)
    assert e.value.status == B.ERR_WORKSPACE
