"""The MoE block around the layer through the C ABI against the oracle.

block(x) = x + layer(u), u = fp16(gamma * x / sqrt(mean(x^2) + eps)), router logits
= u . Wr (model card "srswti/axe-diffusion-ksl-xe", "the kernels we built": the
RMSNorm of a block in one launch; "what the model is": top-8 of 128 experts).

Bars:
  front    u and the router logits bit-identical to the oracle's (both follow the
           same fixed fp32 order of operations, which the header defines);
  routing  topk_idx, expert_offsets and pair_list of the block equal the oracle's
           routing of the oracle's logits, element for element;
  output   max |gpu - oracle| <= 2e-2 and ||gpu - oracle||_F / ||oracle||_F <= 1e-3,
           the oracle being x + the fp64 layer of the oracle's u (unrounded).
"""
import os

import numpy as np
import pytest

import oracle
from w4a16_moe_expert_router_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
REL_FROB = 1e-3
NCPU = os.cpu_count() or 1


@pytest.fixture(scope="module")
def rt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a16_moe_expert_router_gb300 import build as libbuild
    libbuild.build()
    from w4a16_moe_expert_router_gb300 import runtime
    return runtime


def _inputs(wl, seed, tokens=None):
    x = synth.make_x(wl, seed, tokens)
    return x, synth.make_gamma_pre(wl, seed), synth.make_router(wl, seed)


@pytest.mark.parametrize("wl,tokens", [
    (synth.WORKLOADS["tiny"], None),
    (synth.WORKLOADS["canvas256"], None),
    (synth.Workload("ragged", 13, 512, 128, 24, 3, 64, 64), None),
    (synth.Workload("e256", 9, 256, 64, 256, 8, 64, 32), None),
], ids=lambda v: getattr(v, "name", str(v)))
def test_block_front_bit_identical_to_oracle(rt, wl, tokens):
    from w4a16_moe_expert_router_gb300 import binding as B
    x, gamma, wr = _inputs(wl, 7, tokens)
    T, d, E = x.shape[0], wl.hidden, wl.experts
    sh = rt.shape_of(wl, T)
    u = torch.empty((T, d), dtype=torch.float16, device="cuda")
    lg = torch.empty((T, E), dtype=torch.float32, device="cuda")
    B.moe_w4a16_block_front(sh, rt.to_device_x(x), rt.to_device_f32(gamma), 1e-6, rt.to_device_u16(wr), u, lg)
    torch.cuda.synchronize()
    u_o, lg_o = oracle.block_front(x, gamma, 1e-6, wr)
    assert np.array_equal(u.cpu().numpy().view(np.uint16), u_o)
    assert np.array_equal(lg.cpu().numpy().view(np.uint32), lg_o.view(np.uint32))


def _block_case(rt, wl, seed, tokens=None, in_place=False):
    from w4a16_moe_expert_router_gb300 import binding as B
    x, gamma, wr = _inputs(wl, seed, tokens)
    w = synth.make_weights(wl, seed)
    T = x.shape[0]
    dw = rt.upload_weights(wl, w)
    buf = rt.alloc_buffers(wl, tokens=T)
    xd = rt.to_device_x(x)
    out = xd if in_place else buf.out
    rt.run_block(buf, xd, rt.to_device_f32(gamma), rt.to_device_u16(wr), dw, 1e-6, out=out)
    torch.cuda.synchronize()
    assert B.moe_w4a16_read_error(buf.workspace) == B.OK
    u_o, lg_o = oracle.block_front(x, gamma, 1e-6, wr)
    idx_o, tw_o = oracle.route(lg_o, wl.top_k)
    off_o, pl_o = oracle.permute(idx_o, wl.experts)
    r = buf.routing
    assert np.array_equal(r.topk_idx.cpu().numpy(), idx_o)
    assert np.array_equal(r.expert_offsets.cpu().numpy(), off_o)
    assert np.array_equal(r.pair_list.cpu().numpy()[:len(pl_o)], pl_o)
    ref = x.view(np.float16).astype(np.float64) + oracle.forward(
        u_o, idx_o, tw_o, w, group_gate_up=wl.group_gate_up, group_down=wl.group_down, activation=wl.activation,
        nthreads=NCPU, fmt=wl.format)
    got = out.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert err.max() <= MAX_ABS, (err.max(), rel)
    assert rel <= REL_FROB, (err.max(), rel)
    return got


def test_block_tiny(rt):
    _block_case(rt, synth.WORKLOADS["tiny"], 3)


@pytest.mark.parametrize("tokens", [1, 5, 33])
def test_block_ragged_token_counts(rt, tokens):
    _block_case(rt, synth.Workload("ragged", 64, 512, 128, 16, 4, 64, 64), tokens, tokens=tokens)


def test_block_canvas256_full_size(rt):
    """The whole block at the 256-token canvas: routing exact through the projected logits."""
    _block_case(rt, synth.WORKLOADS["canvas256"], 1)


def test_block_in_place_equals_separate_output(rt):
    wl = synth.WORKLOADS["tiny"]
    a = _block_case(rt, wl, 9)
    b = _block_case(rt, wl, 9, in_place=True)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("fmt,red", [(1, 0), (2, 0), (0, 1), (1, 1), (2, 1)])
def test_block_weight_formats_and_reduction_orders(rt, fmt, red):
    """The block with affine-bias (1) and symmetric (2) weights and the group-factorised
    order (reduction 1): same bars, the oracle dequantising the same format."""
    import dataclasses
    wl = dataclasses.replace(synth.WORKLOADS["tiny"], format=fmt, reduction=red)
    _block_case(rt, wl, 11 + fmt + 3 * red)


def test_block_256_experts_top8(rt):
    """E = 256, k = 8 through the whole block (front, routing of its logits, layer, residual)."""
    _block_case(rt, synth.Workload("e256", 9, 256, 64, 256, 8, 64, 32), 5)
