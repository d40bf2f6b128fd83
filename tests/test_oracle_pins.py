"""Pins of the fp64 CPU oracle against facts fixed outside the oracle itself.

Each test checks the oracle against something it does not compute: values
worked by hand from the weight-format definition (golden files), numpy/scipy
routines that implement an independent definition (IEEE half decoding, stable
argsort, softmax, the normal CDF), closed forms, brute force on tiny inputs and
invariants.  They are chosen so that a plausible mistake (a swapped nibble, a
transposed operand, gate and up exchanged, a wrong group index, a dropped
term, a sign error) fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle
from w4a16_moe_expert_router_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return [ln.split() for ln in fh if ln.strip() and not ln.startswith("#")]


# ------------------------------------------------------------------ fp16 ----

def test_half_decode_matches_numpy_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.signbit(got[finite]), np.signbit(ref[finite]))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_half_encode_round_to_nearest_even_matches_numpy():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000),
        # exact ties between neighbouring halves must round to even
        (np.arange(1024, 2048, dtype=np.float64) + 0.5) / 1024.0,
        np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 1e-9]),
    ])
    for v in vals:
        with np.errstate(over="ignore"):
            want = int(np.array(v, np.float64).astype(np.float16).view(np.uint16))
        assert oracle.double_to_half(float(v)) == want, v


# --------------------------------------------------------- weight format ----

def test_dequant_triples_worked_by_hand():
    rows = _rows("dequant_triples.txt")
    assert len(rows) >= 5
    for q, zb, sb, want in rows:
        assert oracle.dequant(int(q), int(zb, 16), int(sb, 16)) == float(want)


def test_nibble_order_golden_and_all_bytes():
    for b, lo, hi in _rows("nibble_order.txt"):
        row = np.array([int(b, 16)], np.uint8)
        assert oracle.code(row, 0) == int(lo)
        assert oracle.code(row, 1) == int(hi)
    # every byte value splits into two nibbles that rebuild it (low = even k)
    row = np.arange(256, dtype=np.uint8)
    for b in range(256):
        assert oracle.code(row, 2 * b) + 16 * oracle.code(row, 2 * b + 1) == b


# --------------------------------------------------------------- routing ----

def _brute_topk(lg, k):
    """Best ordered k-tuple under (value desc, index asc), by enumeration."""
    E = len(lg)
    best = max(itertools.permutations(range(E), k), key=lambda p: tuple((float(lg[e]), -e) for e in p))
    return list(best)


@pytest.mark.parametrize("E,k", [(2, 1), (3, 2), (5, 3), (8, 2), (10, 4), (6, 6)])
def test_topk_brute_force(E, k):
    rng = np.random.default_rng(E * 10 + k)
    cases = [rng.standard_normal(E).astype(np.float32) for _ in range(20)]
    cases.append(np.zeros(E, np.float32))                               # all equal -> 0..k-1
    cases.append(np.where(np.arange(E) % 2 == 0, 0.0, -0.0).astype(np.float32))  # +0 / -0 tie
    dup = rng.integers(0, 3, E).astype(np.float32)                      # duplicates across the k-th place
    cases.append(dup)
    straddle = np.zeros(E, np.float32)                                 # ties exactly at the k-th place
    straddle[E - 1] = 1.0
    cases.append(straddle)
    lg = np.stack(cases)
    idx, w = oracle.route(lg, k)
    for t in range(lg.shape[0]):
        assert list(idx[t]) == _brute_topk(lg[t], k), (lg[t], idx[t])
    assert list(idx[-4]) == list(range(k))   # all-equal logits pick the lowest ids


def test_softmax_over_selected_properties_and_library_softmax():
    rng = np.random.default_rng(7)
    lg = rng.standard_normal((50, 16)).astype(np.float32) * 3
    for k in (1, 2, 8, 16):
        idx, w = oracle.route(lg, k)
        assert np.all(w > 0)
        assert np.all(np.diff(w, axis=1) <= 0)                 # non-increasing in rank
        assert np.allclose(w.sum(1), 1.0, rtol=0, atol=1e-15)
        sel = np.take_along_axis(lg.astype(np.float64), idx, 1)
        assert np.allclose(w, scipy.special.softmax(sel, axis=1), rtol=1e-14, atol=0)
        if k == 1:
            assert np.all(w == 1.0)
        if k == 16:                                            # k = E: the full softmax
            full = scipy.special.softmax(lg.astype(np.float64), axis=1)
            assert np.allclose(np.take_along_axis(full, idx, 1), w, rtol=1e-14, atol=0)


def test_route_rejects_nonfinite():
    lg = np.zeros((2, 4), np.float32)
    lg[1, 2] = np.nan
    with pytest.raises(ValueError):
        oracle.route(lg, 2)
    lg[1, 2] = np.inf
    with pytest.raises(ValueError):
        oracle.route(lg, 2)


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (16, 8, 2), (64, 128, 8), (37, 5, 3)])
def test_permute_matches_stable_argsort(T, E, k):
    rng = np.random.default_rng(T + E + k)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    off, pl = oracle.permute(idx, E)
    order = np.argsort(idx.ravel(), kind="stable")
    assert np.array_equal(pl, order)
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(idx.ravel(), minlength=E))]))


# ------------------------------------------------------------ activation ----

def test_gelu_erf_form_is_a_times_normal_cdf():
    for a in np.linspace(-8, 8, 161):
        assert oracle.gelu(a, 1) == pytest.approx(a * scipy.stats.norm.cdf(a), rel=1e-13, abs=1e-15)


def test_gelu_tanh_form_closed_forms():
    assert oracle.gelu(0.0, 0) == 0.0
    for a in (0.3, 1.0, 2.5, 7.0):
        for act in (0, 1):                       # gelu(a) - gelu(-a) = a for both forms
            assert oracle.gelu(a, act) - oracle.gelu(-a, act) == pytest.approx(a, rel=1e-14)
    assert oracle.gelu(10.0, 0) == pytest.approx(10.0, rel=1e-15)
    assert abs(oracle.gelu(-10.0, 0)) < 1e-15 * 10
    # choose a so that sqrt(2/pi) (a + 0.044715 a^3) = atanh(y); then gelu(a) = a (1 + y) / 2
    for y in (-0.6, 0.25, 0.5, 0.9):
        u = math.atanh(y) / math.sqrt(2.0 / math.pi)
        roots = np.roots([0.044715, 0.0, 1.0, -u])
        a = float(roots[np.argmin(np.abs(roots.imag))].real)
        assert oracle.gelu(a, 0) == pytest.approx(0.5 * a * (1 + y), rel=1e-12)
    # the tanh form stays within 1e-3 of the exact (erf) GELU everywhere
    grid = np.linspace(-10, 10, 2001)
    dev = max(abs(oracle.gelu(a, 0) - a * scipy.stats.norm.cdf(a)) for a in grid)
    assert 1e-5 < dev < 1e-3


# ---------------------------------------------------------------- layer ----

def _half(v):
    return np.asarray(v, np.float64).astype(np.float16).view(np.uint16)


def _selector_layer(T, d, f, E, k, g1, g2, seed):
    """Weights whose every row has one nonzero: codes 9 at one column, 8 elsewhere,
    zero-point 8, so W[n][c] = s[n][group of c] * [c == col(n)].  Scales are powers
    of two that differ per row and per group, and the unused groups get scales that
    would change the result if they were ever applied."""
    rng = np.random.default_rng(seed)
    gu_col = rng.integers(0, d, (E, 2 * f))
    dn_col = rng.integers(0, f, (E, d))
    gu_codes = np.full((E, 2 * f, d), 8, np.uint8)
    dn_codes = np.full((E, d, f), 8, np.uint8)
    for e in range(E):
        gu_codes[e, np.arange(2 * f), gu_col[e]] = 9
        dn_codes[e, np.arange(d), dn_col[e]] = 9
    gu_s = 2.0 ** -rng.integers(0, 6, (E, 2 * f, d // g1))
    dn_s = 2.0 ** -rng.integers(0, 6, (E, d, f // g2))
    pack = lambda c: (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)
    weights = {
        "gate_up_q": pack(gu_codes), "gate_up_scale": _half(gu_s), "gate_up_zero": _half(np.full(gu_s.shape, 8.0)),
        "down_q": pack(dn_codes), "down_scale": _half(dn_s), "down_zero": _half(np.full(dn_s.shape, 8.0)),
    }
    x = rng.integers(-4, 5, (T, d)).astype(np.float64) / 4.0
    logits = rng.standard_normal((T, E)).astype(np.float32)

    def expected(idx, w, act):
        gelu = (lambda a: a * scipy.stats.norm.cdf(a)) if act == 1 else \
               (lambda a: 0.5 * a * (1 + np.tanh(np.sqrt(2 / np.pi) * (a + 0.044715 * a ** 3))))
        out = np.zeros((T, d))
        for t in range(T):
            for r in range(k):
                e = idx[t, r]
                n = np.arange(2 * f)
                a = gu_s[e, n, gu_col[e] // g1] * x[t, gu_col[e]]          # selector rows
                h = gelu(a[:f]) * a[f:]                                     # gate rows first, then up
                i = np.arange(d)
                y = dn_s[e, i, dn_col[e] // g2] * h[dn_col[e]]
                out[t] += w[t, r] * y
        return out

    return weights, _half(x), logits, expected


@pytest.mark.parametrize("act", [0, 1])
def test_selector_layer_closed_form(act):
    T, d, f, E, k, g1, g2 = 5, 64, 32, 4, 2, 32, 16
    weights, xb, logits, expected = _selector_layer(T, d, f, E, k, g1, g2, seed=11 + act)
    idx, w = oracle.route(logits, k)
    got = oracle.forward(xb, idx, w, weights, group_gate_up=g1, group_down=g2, activation=act)
    assert np.allclose(got, expected(idx, w, act), rtol=1e-13, atol=1e-15)


def test_tiny_constant_layer_hand_value():
    """T=1, E=2, k=1, d=f=g=64: expert 1 is chosen (logits 0, 1); its gate rows are
    (9-8)*2^-6, its up rows (10-8)*2^-6, its down rows (9-8)*2^-6, x = 1.  Then
    gate = 1, up = 2, h = 2 gelu(1), y = 64 * 2^-6 * h = 2 gelu(1); with the tanh form
    gelu(1) = 0.5 (1 + tanh(sqrt(2/pi) * 1.044715)).  Expert 0 holds other values."""
    d = f = g = 64
    gu = np.full((2, 2 * f, d), 9, np.uint8)
    gu[1, f:, :] = 10
    gu[0] = 3
    dn = np.full((2, d, f), 9, np.uint8)
    dn[0] = 14
    pack = lambda c: (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)
    weights = {
        "gate_up_q": pack(gu), "gate_up_scale": _half(np.full((2, 2 * f, 1), 2.0 ** -6)),
        "gate_up_zero": _half(np.full((2, 2 * f, 1), 8.0)), "down_q": pack(dn),
        "down_scale": _half(np.full((2, d, 1), 2.0 ** -6)), "down_zero": _half(np.full((2, d, 1), 8.0)),
    }
    idx, w = oracle.route(np.array([[0.0, 1.0]], np.float32), 1)
    assert idx[0, 0] == 1 and w[0, 0] == 1.0
    out = oracle.forward(_half(np.ones((1, d))), idx, w, weights, group_gate_up=g, group_down=g)
    want = 2 * 0.5 * (1 + math.tanh(math.sqrt(2 / math.pi) * 1.044715))
    assert np.allclose(out, want, rtol=1e-14, atol=0)   # 64-term fp64 sums round at ~1e-16


def test_dense_form_equals_sparse_form():
    wl = synth.WORKLOADS["tiny"]
    x = synth.make_x(wl, seed=3)[:6]
    lg = synth.make_logits(wl, seed=3)[:6]
    wts = synth.make_weights(wl, seed=3)
    idx, w = oracle.route(lg, wl.top_k)
    sparse = oracle.forward(x, idx, w, wts, group_gate_up=64, group_down=64, nthreads=3)
    dense = oracle.forward_dense(x, idx, w, wts, group_gate_up=64, group_down=64)
    assert np.allclose(sparse, dense, rtol=1e-12, atol=1e-12)


def test_identical_experts_reproduce_one_expert():
    wl = synth.WORKLOADS["tiny"]
    one = {k: v[:1] for k, v in synth.make_weights(wl, seed=5).items()}
    E = 4
    same = {k: np.ascontiguousarray(np.repeat(v, E, axis=0)) for k, v in one.items()}
    x = synth.make_x(wl, seed=5)[:3]
    lg = synth.make_logits(wl, seed=5)[:3, :E]
    idx, w = oracle.route(lg, 3)
    got = oracle.forward(x, idx, w, same, group_gate_up=64, group_down=64)
    single = oracle.forward(x, np.zeros((3, 1), np.int32), np.ones((3, 1)), one, group_gate_up=64, group_down=64)
    assert np.allclose(got, single, rtol=1e-12, atol=1e-13)


def test_token_selection_and_threads_do_not_change_rows():
    wl = synth.WORKLOADS["tiny"]
    x, lg, wts = synth.make_x(wl), synth.make_logits(wl), synth.make_weights(wl)
    idx, w = oracle.route(lg, wl.top_k)
    full = oracle.forward(x, idx, w, wts, group_gate_up=64, group_down=64, nthreads=1)
    sel = np.zeros(wl.tokens, np.uint8)
    sel[[0, 7, 15]] = 1
    part = oracle.forward(x, idx, w, wts, group_gate_up=64, group_down=64, token_sel=sel, nthreads=4)
    assert np.array_equal(part[sel == 1], full[sel == 1])
    assert np.all(np.isnan(part[sel == 0]))


def test_rmsnorm_closed_forms():
    d = 64
    gamma = np.linspace(0.5, 1.5, d).astype(np.float32)
    u = np.full(d, -3.0)
    eps = 1e-6
    assert np.allclose(oracle.rmsnorm(u, gamma, eps), gamma.astype(np.float64) * -3.0 / math.sqrt(9.0 + eps),
                       rtol=1e-15)
    rng = np.random.default_rng(2)
    v = rng.standard_normal(d)
    assert np.allclose(oracle.rmsnorm(7.0 * v, gamma, 0.0), oracle.rmsnorm(v, gamma, 0.0), rtol=1e-14)
    n = oracle.rmsnorm(v, np.ones(d, np.float32), 0.0)
    assert np.mean(n ** 2) == pytest.approx(1.0, rel=1e-14)


def test_layer_rmsnorm_applies_to_combined_row():
    wl = synth.WORKLOADS["tiny"]
    x, lg, wts = synth.make_x(wl), synth.make_logits(wl), synth.make_weights(wl)
    gamma = synth.make_gamma(wl)
    idx, w = oracle.route(lg, wl.top_k)
    u = oracle.forward(x, idx, w, wts, group_gate_up=64, group_down=64)
    normed = oracle.forward(x, idx, w, wts, group_gate_up=64, group_down=64, gamma=gamma, eps=1e-6)
    for t in (0, 5):
        assert np.allclose(normed[t], oracle.rmsnorm(u[t], gamma, 1e-6), rtol=1e-14, atol=1e-15)


def test_fp16_diagnostic_mode_stays_within_rounding():
    wl = synth.WORKLOADS["tiny"]
    x, lg, wts = synth.make_x(wl), synth.make_logits(wl), synth.make_weights(wl)
    idx, w = oracle.route(lg, wl.top_k)
    exact = oracle.forward(x, idx, w, wts, group_gate_up=64, group_down=64)
    rounded = oracle.forward(x, idx, w, wts, group_gate_up=64, group_down=64, round_fp16=True)
    rel = np.linalg.norm(rounded - exact) / np.linalg.norm(exact)
    assert 0 < rel < 2e-3


# ---------------------------------------------------------------- formats
# "ashhart/TensorFold pull 802", "Summary": symmetric GPTQ 4/128 and MLX affine 4/64
# checkpoints next to the model card's asymmetric uint4 (format 0).

def test_format_triples_worked_by_hand():
    """Affine (negative and positive biases) and symmetric (including a negative scale
    and an ignored second value) values worked by hand from the format definitions."""
    rows = _rows("format_triples.txt")
    assert {r[0] for r in rows} == {"1", "2"} and len(rows) >= 10
    for fmt, q, sb, scb, want in rows:
        assert oracle.dequant_format(int(q), int(sb, 16), int(scb, 16), int(fmt)) == float(want)


def test_format_dequant_values():
    s, z, b = 0x211F, 0x47C0, 0xAC00  # fp16 0.0100021..., 7.75, -0.0625
    sv, zv, bv = (float(np.array([v], np.uint16).view(np.float16)[0]) for v in (s, z, b))
    for q in (0, 7, 8, 15):
        assert oracle.dequant_format(q, z, s, 0) == (q - zv) * sv
        assert oracle.dequant_format(q, b, s, 1) == q * sv + bv
        assert oracle.dequant_format(q, z, s, 2) == (q - 8) * sv


def test_format_identities_through_the_layer():
    """Affine with b = 0 is asymmetric with z = 0, and symmetric is asymmetric with
    z = 8, bit for bit through the whole fp64 layer; a swapped or miswired format fails."""
    wl = synth.Workload("fmt", 9, 256, 64, 4, 2, 64, 32)
    x, lg = synth.make_x(wl, 3), synth.make_logits(wl, 3)
    w = synth.make_weights(wl, 3)
    idx, tw = oracle.route(lg, wl.top_k)
    zero = {k: (np.zeros_like(v) if k.endswith("zero") else v) for k, v in w.items()}
    eight = {k: (np.full_like(v, 0x4800) if k.endswith("zero") else v) for k, v in w.items()}
    run = lambda ww, fmt: oracle.forward(x, idx, tw, ww, group_gate_up=64, group_down=32, fmt=fmt)
    assert np.array_equal(run(zero, 1), run(zero, 0))
    assert np.array_equal(run(w, 2), run(eight, 0))
    assert not np.array_equal(run(w, 2), run(w, 0))
    assert not np.array_equal(run(w, 1), run(w, 0))


# ------------------------------------------------------------ MoE block
# The block around the layer: pre-norm u = fp16(gamma * x / sqrt(mean(x^2) + eps)),
# router logits = u . Wr (model card "srswti/axe-diffusion-ksl-xe", "the kernels we
# built": one-launch RMSNorm; "what the model is": top-8 of 128 experts), computed
# in fp32 in a fixed order so that the routing they decide is reproducible.

def _block_inputs(T, d, E, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d)).astype(np.float16).view(np.uint16)
    gamma = (1.0 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    wr = (rng.standard_normal((E, d)) / np.sqrt(d)).astype(np.float16).view(np.uint16)
    return x, gamma, wr


def test_block_front_u_is_the_fp16_rmsnorm():
    """u against the fp64 RMSNorm rounded to fp16: equal except where the fp32
    evaluation lands on the other side of an fp16 rounding boundary (one ulp)."""
    x, gamma, wr = _block_inputs(32, 512, 8, 1)
    u, _ = oracle.block_front(x, gamma, 1e-6, wr)
    xf = x.view(np.float16).astype(np.float64)
    ref = (gamma * xf / np.sqrt((xf * xf).mean(1, keepdims=True) + 1e-6)).astype(np.float16)
    got = u.view(np.float16)
    assert (got == ref).mean() > 0.999
    ulp = np.abs(np.spacing(ref.astype(np.float16))).astype(np.float64)
    assert np.all(np.abs(got.astype(np.float64) - ref.astype(np.float64)) <= ulp)


def test_block_front_logits_within_the_fp32_bound():
    """logits against the fp64 dot product of the same u and Wr, inside the classical
    bound for a sum of n fp32 terms: |err| <= n eps / (1 - n eps) * sum |u_k w_k|, with
    n = d / 256 * 8 sequential terms per lane plus 5 butterfly levels."""
    T, d, E = 16, 2048, 128
    x, gamma, wr = _block_inputs(T, d, E, 2)
    u, logits = oracle.block_front(x, gamma, 1e-6, wr)
    uf = u.view(np.float16).astype(np.float64)
    wf = wr.view(np.float16).astype(np.float64)
    ref = uf @ wf.T
    n = d // 256 * 8 + 5
    eps = 2.0 ** -24
    bound = n * eps / (1 - n * eps) * (np.abs(uf) @ np.abs(wf).T)
    assert np.all(np.abs(logits.astype(np.float64) - ref) <= bound)
    # a wrong row of Wr, a transposed operand or a dropped chunk is far outside the bound
    assert np.abs(logits.astype(np.float64) - uf @ np.roll(wf, 1, axis=0).T).max() > 100 * bound.max()


def test_block_front_one_hot_router_copies_u():
    """A router whose row e is 1 at column c_e and 0 elsewhere gives logits[t][e] = u[t][c_e]
    exactly (one exact product, the rest exact zeros)."""
    T, d, E = 8, 256, 16
    x, gamma, _ = _block_inputs(T, d, E, 3)
    cols = np.array([0, 7, 8, 255, 31, 32, 100, 200, 63, 64, 1, 2, 250, 17, 128, 129])
    wr = np.zeros((E, d), np.float16)
    wr[np.arange(E), cols] = 1.0
    u, logits = oracle.block_front(x, gamma, 1e-6, wr.view(np.uint16))
    assert np.array_equal(logits, u.view(np.float16)[:, cols].astype(np.float32))


def test_block_front_constant_rows_closed_form():
    """x = 2 everywhere, gamma = 1, eps = 0: ss = 4 d exactly, r = 1/2, u = 1.0 exactly;
    x = c with eps: u = fp16(c / sqrt(c^2 + eps)) for every column."""
    d = 512
    x = np.full((2, d), 2.0, np.float16).view(np.uint16)
    u, _ = oracle.block_front(x, np.ones(d, np.float32), 0.0, np.zeros((1, d), np.uint16))
    assert np.all(u == 0x3C00)
    x = np.full((1, d), 0.5, np.float16).view(np.uint16)
    u, _ = oracle.block_front(x, np.ones(d, np.float32), 1.0, np.zeros((1, d), np.uint16))
    assert np.all(u.view(np.float16) == np.float16(0.5 / np.sqrt(1.25)))
