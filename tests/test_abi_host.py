"""Host-only tests of the C-ABI library: it loads, exports what the header
declares, validates shapes and pointers before touching a GPU, and its host
weight helpers (pack/unpack, prepare/unprepare) are exact permutations."""
import ctypes
import os
import re

import numpy as np
import pytest

from w4a16_moe_expert_router_gb300 import binding as B
from w4a16_moe_expert_router_gb300 import build as libbuild
from w4a16_moe_expert_router_gb300 import synth, runtime

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session", autouse=True)
def built_library():
    libbuild.build()
    return B.lib()


def _header_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"^MOE_W4A16_API\s+[\w\s\*]+?\b(moe_w4a16_\w+)\s*\(", text, flags=re.M)
    return names


def test_library_exports_every_declared_symbol():
    names = _header_functions()
    assert len(names) >= 11
    raw = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n
    assert set(names) == set(B.EXPORTED)


def test_status_strings():
    for code in range(9):
        assert B.moe_w4a16_status_string(code)
    assert B.moe_w4a16_status_string(99) == "unknown status"


VALID = dict(tokens=16, hidden=256, inter=128, experts=8, top_k=2, group_gate_up=64, group_down=64)


def _shape(**kw):
    d = dict(VALID)
    d.update(kw)
    return B.make_shape(**d)


@pytest.mark.parametrize("bad", [
    dict(hidden=192), dict(hidden=64), dict(inter=96), dict(experts=0), dict(experts=257), dict(top_k=0),
    dict(top_k=9), dict(experts=4, top_k=5), dict(group_gate_up=48), dict(group_gate_up=16),
    dict(group_down=128, inter=192), dict(activation=2), dict(reduction=2), dict(reduction=-1), dict(format=3), dict(format=-1), dict(tokens=-1), dict(tokens=1 << 20, top_k=8),
])
def test_invalid_shapes_rejected(bad):
    sh = _shape(**bad)
    assert B.moe_w4a16_workspace_bytes(sh) == 0
    assert B.moe_w4a16_prepared_bytes(sh, B.GATE_UP) == 0
    L = B.lib()
    r = B.Routing(16, 16, 16, 16)
    assert L.moe_w4a16_route(ctypes.byref(sh), 16, ctypes.byref(r), 16, 1 << 30, None) == B.ERR_SHAPE
    w = B.Weights(16, 16)
    assert L.moe_w4a16_forward(ctypes.byref(sh), 16, ctypes.byref(r), ctypes.byref(w), None, 1e-6, 16, 16,
                               1 << 30, None) == B.ERR_SHAPE


def test_workspace_size_covers_intermediates():
    sh = _shape()
    T, k, d, f = 16, 2, 256, 128
    assert B.moe_w4a16_workspace_bytes(sh) >= 256 + T * k * f * 2 + T * k * d * 4


def test_pointer_and_workspace_validation_before_any_launch():
    L = B.lib()
    sh = _shape()
    ws = B.moe_w4a16_workspace_bytes(sh)
    good = B.Routing(4096, 4096, 4096, 4096)
    w = B.Weights(4096, 4096)
    fwd = lambda x, r, wt, out, wsp, wsb, gamma=None, eps=1e-6: L.moe_w4a16_forward(
        ctypes.byref(sh), x, ctypes.byref(r), ctypes.byref(wt), gamma, eps, out, wsp, wsb, None)
    assert fwd(None, good, w, 4096, 4096, ws) == B.ERR_NULL
    assert fwd(4096, B.Routing(4096, None, 4096, 4096), w, 4096, 4096, ws) == B.ERR_NULL
    assert fwd(4096, good, B.Weights(4096, None), 4096, 4096, ws) == B.ERR_NULL
    assert fwd(4104, good, w, 4096, 4096, ws) == B.ERR_ALIGN
    assert fwd(4096, good, w, 4096, 4096, ws, gamma=4100) == B.ERR_ALIGN
    assert fwd(4096, good, w, 4096, 4096, ws - 1) == B.ERR_WORKSPACE
    assert fwd(4096, good, w, 4096, 4096, ws, eps=-1.0) == B.ERR_VALUE
    rt = lambda lg, r, wsb: L.moe_w4a16_route(ctypes.byref(sh), lg, ctypes.byref(r), 4096, wsb, None)
    assert rt(None, good, ws) == B.ERR_NULL
    assert rt(4097, good, ws) == B.ERR_ALIGN
    assert rt(4096, B.Routing(4096, 4096, 4104, 4096), ws) == B.ERR_ALIGN
    assert rt(4096, good, 100) == B.ERR_WORKSPACE
    assert L.moe_w4a16_route(ctypes.byref(sh), 4096, None, 4096, ws, None) == B.ERR_NULL


def test_block_validation_before_any_launch():
    """The MoE block's calls check shapes, pointers, alignment, workspace and eps on
    the host; d must be a multiple of 256 (the lanes' 8-column chunks)."""
    L = B.lib()
    sh = _shape()                      # d = 256
    ws = B.moe_w4a16_workspace_bytes(sh)
    r = B.Routing(4096, 4096, 4096, 4096)
    w = B.Weights(4096, 4096)
    blk = lambda x, g, wr, out, wsb, eps=1e-6, sh=sh, rr=r, ww=w: L.moe_w4a16_block(
        ctypes.byref(sh), x, g, eps, wr, ctypes.byref(rr), ctypes.byref(ww), out, 4096, wsb, None)
    assert blk(None, 4096, 4096, 4096, ws) == B.ERR_NULL
    assert blk(4096, None, 4096, 4096, ws) == B.ERR_NULL
    assert blk(4096, 4096, 4096, 4096, ws, rr=B.Routing(4096, 4096, None, 4096)) == B.ERR_NULL
    assert blk(4104, 4096, 4096, 4096, ws) == B.ERR_ALIGN
    assert blk(4096, 4096, 4100, 4096, ws) == B.ERR_ALIGN
    assert blk(4096, 4096, 4096, 4096, ws - 1) == B.ERR_WORKSPACE
    assert blk(4096, 4096, 4096, 4096, ws, eps=-1.0) == B.ERR_VALUE
    sh384 = _shape(hidden=384, group_gate_up=128)
    assert blk(4096, 4096, 4096, 4096, 1 << 30, sh=sh384) == B.ERR_SHAPE
    front = lambda x, g, wr, u, lg, sh=sh: L.moe_w4a16_block_front(ctypes.byref(sh), x, g, 1e-6, wr, u, lg, None)
    assert front(4096, 4096, 4096, 4096, None) == B.ERR_NULL
    assert front(4096, 4096, 4096, 4104, 4096) == B.ERR_ALIGN
    assert front(4096, 4096, 4096, 4096, 4096, sh=sh384) == B.ERR_SHAPE
    assert B.moe_w4a16_workspace_bytes(sh) >= 16 * 256 * 2 + 16 * 8 * 4  # room for u and the logits


def test_noalloc_read_error_checks_its_pointer():
    assert B.lib().moe_w4a16_noalloc_read_error(None, None) == B.ERR_NULL


def test_zero_tokens_is_a_no_op():
    L = B.lib()
    sh = _shape(tokens=0)
    r = B.Routing(None, None, None, None)
    w = B.Weights(None, None)
    assert L.moe_w4a16_route(ctypes.byref(sh), None, ctypes.byref(r), None, 0, None) == B.OK
    assert L.moe_w4a16_forward(ctypes.byref(sh), None, ctypes.byref(r), ctypes.byref(w), None, 1e-6, None, None, 0,
                               None) == B.OK


def test_pack_unpack_round_trip_all_bytes():
    packed = np.arange(256, dtype=np.uint8).reshape(4, 64)
    codes = B.moe_w4a16_unpack(packed)
    assert codes.shape == (4, 128)
    assert np.array_equal(B.moe_w4a16_pack(codes), packed)
    assert codes[2, 70] == 3 and codes[2, 71] == 10      # byte 163 = 0xA3 sits at row 2, column 35
    row = B.moe_w4a16_unpack(np.array([[0xA3]], np.uint8))
    assert list(row[0]) == [3, 10]


def test_pack_rejects_codes_above_15():
    with pytest.raises(B.MoeW4A16Error) as e:
        B.moe_w4a16_pack(np.array([[3, 16]], np.uint8))
    assert e.value.status == B.ERR_VALUE


@pytest.mark.parametrize("g1,g2,d,f,E", [(64, 64, 256, 128, 3), (32, 32, 256, 192, 2), (128, 64, 384, 64, 2),
                                         (128, 128, 256, 256, 1)])
def test_prepare_unprepare_round_trip(g1, g2, d, f, E):
    wl = synth.Workload("t", 4, d, f, E, 1, g1, g2)
    w = synth.make_weights(wl, seed=g1 + g2 + d)
    sh = runtime.shape_of(wl)
    for which, q, s, z in ((B.GATE_UP, "gate_up_q", "gate_up_scale", "gate_up_zero"),
                           (B.DOWN, "down_q", "down_scale", "down_zero")):
        prep = B.moe_w4a16_prepare(sh, which, w[q], w[s], w[z])
        assert prep.nbytes == w[q].nbytes + w[s].nbytes + w[z].nbytes == B.moe_w4a16_prepared_bytes(sh, which)
        q2, s2, z2 = B.moe_w4a16_unprepare(sh, which, prep, w[q].shape, w[s].shape)
        assert np.array_equal(q2, w[q]) and np.array_equal(s2, w[s]) and np.array_equal(z2, w[z])


def _check_strip(seg, ng, steps, rows, codes, scale, zero, grp0, c0):
    """One warp strip of one stage: (scale, zero) of rows (i, i + 8) per group, ordered
    [i][group]; then words [kk // 4][lane][kk % 4] where nibble n of word (lane, kk)
    holds strip row lane // 4 + 8 (n & 1), column c0 + 16 kk + 2 (lane % 4) + 8 ((n >> 1) & 1) + (n >> 2)."""
    sz = seg[:64 * ng].view(np.uint16).reshape(8, ng, 2, 2)
    for i in range(8):
        for j in range(ng):
            for h in range(2):
                assert sz[i, j, h, 0] == scale[rows[i + 8 * h], grp0 + j]
                assert sz[i, j, h, 1] == zero[rows[i + 8 * h], grp0 + j]
    words = seg[64 * ng:64 * ng + steps * 128].view(np.uint32)
    for kk in range(steps):
        for lane in (0, 5, 17, 31):
            gq, tq = lane // 4, lane % 4
            wd = int(words[(kk // 4) * 128 + lane * 4 + kk % 4])
            for n in range(8):
                r = gq + 8 * (n & 1)
                col = c0 + 16 * kk + 2 * tq + 8 * ((n >> 1) & 1) + (n >> 2)
                assert (wd >> (4 * n)) & 15 == codes[rows[r], col]


def test_prepared_word_layout_matches_documented_order():
    """Stages of 128 columns (the last of 64 when K is an odd multiple of 64); per
    stage, eight warp strips of 16 GEMM rows; gate_up strip w of block b holds gate
    rows 64b + 8w + (0..7) and the matching up rows f + 64b + 8w + (0..7), down strip
    w of block b holds rows 128b + 16w + (0..15)."""
    wl = synth.Workload("t", 4, 256, 192, 1, 1, 64, 64)   # d = 256 (2 stages), f = 192 (128 + 64)
    w = synth.make_weights(wl, seed=9)
    sh = runtime.shape_of(wl)
    f = wl.inter
    gu = B.moe_w4a16_prepare(sh, B.GATE_UP, w["gate_up_q"], w["gate_up_scale"], w["gate_up_zero"])
    codes = B.moe_w4a16_unpack(w["gate_up_q"])[0]          # [2f][d]
    sc, ze = w["gate_up_scale"][0], w["gate_up_zero"][0]
    strip = 8 * 128 + 2 * 64                                # one warp's part of a full stage, groups of 64
    block = 2 * 8 * strip                                   # K = 256: two full stages
    for b, st, wv in ((0, 0, 0), (0, 1, 3), (2, 1, 7)):
        rows = [64 * b + 8 * wv + r if r < 8 else f + 64 * b + 8 * wv + r - 8 for r in range(16)]
        off = b * block + st * 8 * strip + wv * strip
        _check_strip(gu[off:off + strip], 2, 8, rows, codes, sc, ze, 2 * st, 128 * st)
    dn = B.moe_w4a16_prepare(sh, B.DOWN, w["down_q"], w["down_scale"], w["down_zero"])
    dcodes = B.moe_w4a16_unpack(w["down_q"])[0]             # [d][f]
    sc, ze = w["down_scale"][0], w["down_zero"][0]
    tail = 4 * 128 + 64                                     # one warp's part of the last 64 columns
    dblock = 8 * strip + 8 * tail
    for b, wv in ((0, 2), (1, 6)):
        rows = [128 * b + 16 * wv + r for r in range(16)]
        off = b * dblock + wv * strip
        _check_strip(dn[off:off + strip], 2, 8, rows, dcodes, sc, ze, 0, 0)
        off = b * dblock + 8 * strip + wv * tail
        _check_strip(dn[off:off + tail], 1, 4, rows, dcodes, sc, ze, 2, 128)
    assert dn.nbytes == 2 * dblock


def test_prepare_rejects_out_of_range_scale_and_zero():
    wl = synth.WORKLOADS["tiny"]
    w = synth.make_weights(wl)
    sh = runtime.shape_of(wl)
    s = w["gate_up_scale"].copy()
    s[0, 0, 0] = np.float16(40.0).view(np.uint16)
    with pytest.raises(B.MoeW4A16Error) as e:
        B.moe_w4a16_prepare(sh, B.GATE_UP, w["gate_up_q"], s, w["gate_up_zero"])
    assert e.value.status == B.ERR_VALUE
    z = w["gate_up_zero"].copy()
    z[1, 2, 3] = np.float16(-0.5).view(np.uint16)
    with pytest.raises(B.MoeW4A16Error):
        B.moe_w4a16_prepare(sh, B.GATE_UP, w["gate_up_q"], w["gate_up_scale"], z)


SAMPLER_VALID = dict(positions=8, vocab=4096, inv_temperature=1.0, rule=0, bound=1.0, step=0, seed=0)


@pytest.mark.parametrize("bad", [
    dict(positions=0), dict(positions=1025), dict(vocab=0), dict(vocab=4098), dict(vocab=(1 << 30) + 4),
    dict(inv_temperature=0.0), dict(inv_temperature=-1.0), dict(inv_temperature=float("inf")),
    dict(inv_temperature=float("nan")), dict(rule=2), dict(bound=float("nan")), dict(bound=float("inf")),
    dict(noise=2), dict(noise=-1),
])
def test_sampler_invalid_configs_rejected(bad):
    d = dict(SAMPLER_VALID)
    d.update(bad)
    cfg = B.make_sampler(**d)
    assert B.moe_w4a16_sampler_workspace_bytes(cfg) == 0
    L = B.lib()
    assert L.moe_w4a16_sample(ctypes.byref(cfg), 16, 16, 16, 16, 16, 16, 16, 1 << 30, None) == B.ERR_SHAPE


def test_sampler_host_validation():
    cfg = B.make_sampler(**SAMPLER_VALID)
    need = B.moe_w4a16_sampler_workspace_bytes(cfg)
    def splits(P, V):  # about ceil(912 / P) splits, each a multiple of 4,096 elements
        want = -(-912 // P)
        chunk = -(-(-(-V // want)) // 4096) * 4096
        return -(-V // chunk)
    assert need == 8 * splits(8, 4096) * 32 == 8 * 1 * 32  # one 32-byte partial per position and split
    for P, V, S in ((8, 262144, 64), (256, 262144, 4), (64, 262144, 13), (1024, 262144, 1), (1, 4, 1),
                    (1, 1000000, 245), (600, 12300, 2)):
        assert splits(P, V) == S
        assert B.moe_w4a16_sampler_workspace_bytes(B.make_sampler(**dict(SAMPLER_VALID, positions=P, vocab=V))) == \
            P * S * 32
    L = B.lib()
    assert L.moe_w4a16_sample(None, 16, 16, 16, 16, 16, 16, 16, need, None) == B.ERR_NULL
    assert L.moe_w4a16_sample(ctypes.byref(cfg), None, 16, 16, 16, 16, 16, 16, need, None) == B.ERR_NULL
    assert L.moe_w4a16_sample(ctypes.byref(cfg), 16, 16, 16, 16, 16, 16, None, need, None) == B.ERR_NULL
    assert L.moe_w4a16_sample(ctypes.byref(cfg), 8, 16, 16, 16, 16, 16, 16, need, None) == B.ERR_ALIGN
    assert L.moe_w4a16_sample(ctypes.byref(cfg), 16, 16, 18, 16, 16, 16, 16, need, None) == B.ERR_ALIGN
    assert L.moe_w4a16_sample(ctypes.byref(cfg), 16, 16, 16, 16, 16, 16, 16, need - 1, None) == B.ERR_WORKSPACE


def test_prepare_per_format():
    """Format 1 keeps the bias in the zero-point slot and accepts negative values;
    format 2 needs no zero array and stores 8 there; out-of-range values are refused."""
    import dataclasses
    base = synth.WORKLOADS["tiny"]
    aff = dataclasses.replace(base, format=1)
    w = synth.make_weights(aff)
    assert (w["gate_up_zero"].view(np.float16) < 0).all()
    sh = runtime.shape_of(aff)
    prep = B.moe_w4a16_prepare(sh, B.GATE_UP, w["gate_up_q"], w["gate_up_scale"], w["gate_up_zero"])
    with pytest.raises(B.MoeW4A16Error):  # a bias is not a valid zero-point
        B.moe_w4a16_prepare(runtime.shape_of(base), B.GATE_UP, w["gate_up_q"], w["gate_up_scale"], w["gate_up_zero"])
    b = w["gate_up_zero"].copy()
    b[0, 0, 0] = np.float16(2000.0).view(np.uint16)
    with pytest.raises(B.MoeW4A16Error) as e:
        B.moe_w4a16_prepare(sh, B.GATE_UP, w["gate_up_q"], w["gate_up_scale"], b)
    assert e.value.status == B.ERR_VALUE
    sym = dataclasses.replace(base, format=2)
    ws = synth.make_weights(sym)
    sh2 = runtime.shape_of(sym)
    p_none = B.moe_w4a16_prepare(sh2, B.DOWN, ws["down_q"], ws["down_scale"], None)
    p_any = B.moe_w4a16_prepare(sh2, B.DOWN, ws["down_q"], ws["down_scale"], np.zeros_like(ws["down_zero"]))
    p_eight = B.moe_w4a16_prepare(runtime.shape_of(base), B.DOWN, ws["down_q"], ws["down_scale"],
                                  np.full_like(ws["down_zero"], 0x4800))
    assert np.array_equal(p_none, p_any) and np.array_equal(p_none, p_eight)
    assert prep.nbytes == B.moe_w4a16_prepared_bytes(sh, B.GATE_UP)


@pytest.mark.parametrize("fmt", [1, 2])
def test_prepare_unprepare_round_trip_per_format(fmt):
    """The stream keeps the affine bias unchanged, and the symmetric format's zero slot
    reads back as 8 whatever zero array was (or was not) given."""
    import dataclasses
    wl = dataclasses.replace(synth.WORKLOADS["tiny"], format=fmt)
    w = synth.make_weights(wl, 5)
    sh = runtime.shape_of(wl)
    for which, (q, s, z) in ((B.GATE_UP, ("gate_up_q", "gate_up_scale", "gate_up_zero")),
                             (B.DOWN, ("down_q", "down_scale", "down_zero"))):
        prep = B.moe_w4a16_prepare(sh, which, w[q], w[s], None if fmt == 2 else w[z])
        q2, s2, z2 = B.moe_w4a16_unprepare(sh, which, prep, w[q].shape, w[s].shape)
        assert np.array_equal(q2, w[q]) and np.array_equal(s2, w[s])
        assert np.array_equal(z2, w[z] if fmt == 1 else np.full_like(w[z], 0x4800))


def test_ctypes_structs_match_the_header(tmp_path):
    """The binding's ctypes structures have the sizes and field offsets the C compiler
    gives the header's structs (a program built with gcc against include/moe_w4a16.h)."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    structs = {"moe_w4a16_shape": B.Shape, "moe_w4a16_sampler": B.Sampler, "moe_w4a16_weights": B.Weights,
               "moe_w4a16_routing": B.Routing}
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "moe_w4a16.h"', "int main(void) {"]
    for cname, cls in structs.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for field, _ in cls._fields_:
            lines.append(f'  printf("{cname} {field} %zu\\n", offsetof({cname}, {field}));')
    lines.append("  return 0;\n}")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    include = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    subprocess.run(["gcc", "-std=c11", "-I", include, str(src), "-o", str(exe)], check=True)
    got = {}
    for ln in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.splitlines():
        name, field, val = ln.split()
        got[(name, field)] = int(val)
    for cname, cls in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(cls), cname
        for field, _ in cls._fields_:
            assert got[(cname, field)] == getattr(cls, field).offset, (cname, field)


def test_smoke_sampler_check_with_a_host_stand_in():
    """The sampler part of __graft_entry__.smoke() run on the CPU, with a stand-in for
    the GPU call that writes the oracle's own outputs: the check's marshalling and
    comparisons are exercised here; on a GPU the real call takes the stand-in's place."""
    import types
    import torch
    import oracle
    import __graft_entry__ as ge

    def fake_sample(cfg, logits, revealed, token, entropy, pmax, accept, workspace, stream=None):
        lg = logits.cpu().numpy()
        t, e, pm = oracle.sample(lg, cfg.inv_temperature, cfg.seed, cfg.step, noise=cfg.noise)
        token.copy_(torch.from_numpy(t))
        entropy.copy_(torch.from_numpy(e.astype(np.float32)))
        pmax.copy_(torch.from_numpy(pm.astype(np.float32)))
        acc = oracle.accept_entropy(e.astype(np.float32), revealed.cpu().numpy(), cfg.bound)
        accept.copy_(torch.from_numpy(acc))

    stand_in = types.SimpleNamespace(make_sampler=B.make_sampler,
                                     moe_w4a16_sampler_workspace_bytes=B.moe_w4a16_sampler_workspace_bytes,
                                     moe_w4a16_sample=fake_sample)
    assert ge._smoke_sampler(stand_in, device="cpu") <= 1e-6
