"""A batched multi-canvas serving step under CUDA-graph capture.

"razoring/diffusion.gguf" reuses captured CUDA graphs across denoising steps; a
server batches several canvases into one step.  The library launches only on the
stream it is given, allocates nothing and never synchronises, so route + forward
(and the sampler) can be captured once and replayed with new inputs copied into
the captured buffers.  Checked here: four 256-token canvases batched into one
1024-token call, captured and replayed on two different inputs, equal to the eager
calls bit for bit and, canvas by canvas, to each canvas run alone.
"""
import dataclasses

import numpy as np
import pytest

from w4a16_moe_expert_router_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a16_moe_expert_router_gb300 import build as libbuild
    libbuild.build()
    from w4a16_moe_expert_router_gb300 import runtime
    return runtime


@pytest.mark.parametrize("reduction", [0, 1])
def test_graph_replay_of_a_batched_multi_canvas_step(rt, reduction):
    canvas = dataclasses.replace(synth.WORKLOADS["canvas256"], reduction=reduction)
    batch = dataclasses.replace(canvas, name="canvas256x4", tokens=4 * canvas.tokens)
    w = synth.make_weights(batch)
    dw = rt.upload_weights(batch, w)
    buf = rt.alloc_buffers(batch)
    inputs = [(synth.make_x(batch, s), synth.make_logits(batch, s)) for s in (11, 12)]
    xd = rt.to_device_x(inputs[0][0])
    ld = rt.to_device_f32(inputs[0][1])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())

    eager = []
    with torch.cuda.stream(s):
        for x, lg in inputs:
            xd.copy_(rt.to_device_x(x))
            ld.copy_(rt.to_device_f32(lg))
            rt.run_layer(buf, xd, ld, dw, stream=s)
            eager.append(buf.out.clone())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            rt.run_layer(buf, xd, ld, dw, stream=s)
        replays = []
        for rep in range(3):
            x, lg = inputs[rep % 2]
            xd.copy_(rt.to_device_x(x))
            ld.copy_(rt.to_device_f32(lg))
            g.replay()
            replays.append(buf.out.clone())
    torch.cuda.synchronize()
    from w4a16_moe_expert_router_gb300 import binding as B
    assert B.moe_w4a16_read_error(buf.workspace) == B.OK
    for rep, out in enumerate(replays):
        assert torch.equal(out, eager[rep % 2])

    # each canvas alone gives its rows of the batched step
    x, lg = inputs[0]
    one = rt.alloc_buffers(canvas)
    for c in range(4):
        rows = slice(c * canvas.tokens, (c + 1) * canvas.tokens)
        rt.run_layer(one, rt.to_device_x(x[rows].copy()), rt.to_device_f32(lg[rows].copy()), dw)
        torch.cuda.synchronize()
        assert torch.equal(one.out, eager[0][rows])


def test_graph_replay_of_the_sampler(rt):
    """The sampler captured once and replayed with a new step counter in the captured
    configuration's place: replays equal eager calls (the config is read at capture
    time, so each step of a denoising loop is its own graph or its own eager call;
    here two graphs, two steps)."""
    from w4a16_moe_expert_router_gb300 import binding as B
    P, V = 256, 32768
    rng = np.random.default_rng(3)
    lg = torch.from_numpy((rng.standard_normal((P, V), dtype=np.float32) * 3).astype(np.float32)).cuda()
    rev = torch.zeros(P, dtype=torch.uint8, device="cuda")
    cfgs = [B.make_sampler(P, V, 1.0, 0, 20.0, step, 99) for step in (0, 1)]
    ws = torch.empty(B.moe_w4a16_sampler_workspace_bytes(cfgs[0]), dtype=torch.uint8, device="cuda")
    outs = [[torch.empty(P, dtype=d, device="cuda") for d in (torch.int32, torch.float32, torch.float32, torch.uint8)]
            for _ in range(2)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        eager = []
        for cfg in cfgs:
            B.moe_w4a16_sample(cfg, lg, rev, *outs[0], ws, stream=s)
            eager.append([t.clone() for t in outs[0]])
        graphs = []
        for i, cfg in enumerate(cfgs):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                B.moe_w4a16_sample(cfg, lg, rev, *outs[i], ws, stream=s)
            graphs.append(g)
        for _ in range(2):
            for g in graphs:
                g.replay()
    torch.cuda.synchronize()
    for i in range(2):
        for a, b in zip(outs[i], eager[i]):
            assert torch.equal(a, b)
    assert not torch.equal(eager[0][0], eager[1][0])  # another step draws other tokens


def test_graph_replay_of_the_moe_block_in_place(rt):
    """The MoE block (pre-norm, router projection, routing, experts, residual combine) of
    a two-layer stack captured once, in place (each layer's output overwrites its
    input), and replayed: equal to the eager calls bit for bit."""
    wl = synth.WORKLOADS["canvas256"]
    ws = [synth.make_weights(wl, 0, layer=l) for l in range(2)]
    dws = [rt.upload_weights(wl, w) for w in ws]
    gam = [rt.to_device_f32(synth.make_gamma_pre(wl, 0, layer=l)) for l in range(2)]
    rou = [rt.to_device_u16(synth.make_router(wl, 0, layer=l)) for l in range(2)]
    buf = rt.alloc_buffers(wl)
    x0 = [rt.to_device_x(synth.make_x(wl, s)) for s in (21, 22)]
    xd = x0[0].clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())

    def stack():
        for l in range(2):
            rt.run_block(buf, xd, gam[l], rou[l], dws[l], 1e-6, out=xd, stream=s)

    with torch.cuda.stream(s):
        eager = []
        for x in x0:
            xd.copy_(x)
            stack()
            eager.append(xd.clone())
        g = torch.cuda.CUDAGraph()
        xd.copy_(x0[0])
        with torch.cuda.graph(g, stream=s):
            stack()
        for rep in range(3):
            xd.copy_(x0[rep % 2])
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(xd.view(torch.int16), eager[rep % 2].view(torch.int16))
    from w4a16_moe_expert_router_gb300 import binding as B
    assert B.moe_w4a16_read_error(buf.workspace) == B.OK
