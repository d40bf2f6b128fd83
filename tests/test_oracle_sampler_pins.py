"""Pins of the sampler oracle (oracle/sampler_oracle.c) to things other than itself:
libm's logarithm and exponential, closed forms of the entropy and of the group keys,
the distribution Gumbel-max must sample (per token and per group of four), the
generator's published known-answer vectors and statistics, and the page's own
formula of the entropy-bound rule.

Sources: "srswti/axe-diffusion-ksl-xe" model card ("the kernels we built": entropy in
one streaming pass, Gumbel-max instead of softmax + multinomial); "lablup/mlxcel
block-diffusion docs" ("Samplers": the entropy-bound rule, the mlx-vlm formula
(cumsum - cummax) <= bound, at least one accepted; the confidence-threshold rule);
Salmon et al., SC'11 (Philox4x32-10); the max-stability of the Gumbel law (the maximum
of independent Gumbel(mu_i) variables is Gumbel(ln sum_i e^mu_i), attained at i with
probability proportional to e^mu_i), which the per-group form rests on.
"""
import math

import os

import numpy as np
import pytest

import oracle


def _ulp(v: float) -> float:
    return float(np.spacing(np.float32(abs(v))))


# ------------------------------------------------------------------ log_f32

def test_log_f32_against_libm_over_the_noise_domain():
    """Within 2.5 fp32 ulps of the exact logarithm on the two ranges the Gumbel noise
    uses (U in [2^-24, 1), E = -ln U in (0, 17]) and across the exponent range (the
    roundings of the quotient, the Horner steps and the product give ~2 ulps near
    x = 1; a wrong series coefficient costs 5 or more)."""
    rng = np.random.default_rng(0)
    xs = np.concatenate([
        ((np.arange(0, 1 << 23, 97) + 0.5) * 2.0 ** -23),          # the U grid itself
        1.0 - np.arange(1, 4096) * 2.0 ** -24,                      # just below 1
        1.0 + np.arange(1, 4096) * 2.0 ** -23,                      # just above 1
        rng.uniform(1e-7, 17.0, 20000),
        2.0 ** rng.uniform(-120, 120, 20000),
    ]).astype(np.float32)
    worst = 0.0
    for x in xs[:: 7]:
        got = oracle.log_f32(float(x))
        want = math.log(float(x))
        if want == 0.0:
            assert got == 0.0
            continue
        worst = max(worst, abs(got - want) / _ulp(want))
    assert worst <= 2.5, worst


def test_log_f32_special_values():
    assert oracle.log_f32(1.0) == 0.0
    for k in range(-30, 31):
        want = k * math.log(2.0)
        got = oracle.log_f32(2.0 ** k)
        assert abs(got - want) <= (_ulp(want) if k else 0.0)


# ------------------------------------------------------------------ Philox

def test_philox_known_answer_vectors():
    """The generator's published known-answer vectors (golden file, with its citation):
    a swapped output word, a wrong key schedule, a wrong multiplier or a mis-ordered
    counter changes every one of them."""
    path = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")
    with open(path) as fh:
        rows = [ln.split() for ln in fh if ln.strip() and not ln.startswith("#")]
    assert len(rows) >= 3
    for r in rows:
        v = [int(x, 16) for x in r]
        got = oracle.philox4x32_10(np.array(v[0:4], np.uint32), np.array(v[4:6], np.uint32))
        assert [int(w) for w in got] == v[6:10]


def test_philox_words_are_uniform_and_counters_avalanche():
    """Counter-based: the same (counter, key) gives the same words; across counters the
    words are uniform (chi-square on the top 4 bits) and flipping one counter or key
    bit flips about half of the 128 output bits."""
    key = np.array([0x12345678, 0x9abcdef0], np.uint32)
    a = oracle.philox4x32_10([5, 6, 7, 8], key)
    assert np.array_equal(a, oracle.philox4x32_10([5, 6, 7, 8], key))
    words = np.concatenate([oracle.philox4x32_10([i, 3, 1, 0], key) for i in range(4096)])
    counts = np.bincount(words >> 28, minlength=16)
    exp = len(words) / 16
    chi2 = float(((counts - exp) ** 2 / exp).sum())
    assert chi2 < 37.7  # chi-square, 15 degrees of freedom, p = 0.001
    rng = np.random.default_rng(1)
    flips = []
    for _ in range(200):
        c = rng.integers(0, 2 ** 32, 4, dtype=np.uint64).astype(np.uint32)
        k = rng.integers(0, 2 ** 32, 2, dtype=np.uint64).astype(np.uint32)
        base = oracle.philox4x32_10(c, k)
        bit = int(rng.integers(0, 192))
        c2, k2 = c.copy(), k.copy()
        if bit < 128:
            c2[bit // 32] ^= np.uint32(1 << (bit % 32))
        else:
            k2[(bit - 128) // 32] ^= np.uint32(1 << (bit % 32))
        d = oracle.philox4x32_10(c2, k2) ^ base
        flips.append(sum(bin(int(w)).count("1") for w in d))
    assert 60 <= np.mean(flips) <= 68


# ------------------------------------------------------------------ entropy

def test_entropy_of_uniform_logits_is_log_v():
    V = 4096
    lg = np.full((3, V), 0.25, np.float32)
    _, ent, pm = oracle.sample(lg, 1.0, 7, 0)
    assert np.allclose(ent, math.log(V), rtol=0, atol=1e-12)
    assert np.allclose(pm, 1.0 / V, rtol=1e-14)


def test_entropy_of_a_two_point_distribution():
    """Two logits a, b and the rest so low that exp underflows: H is the binary entropy of sigmoid(a - b)."""
    V = 64
    lg = np.full((1, V), -1e5, np.float32)
    lg[0, 10], lg[0, 40] = 1.5, -0.25
    _, ent, pm = oracle.sample(lg, 1.0, 1, 0)
    p = 1.0 / (1.0 + math.exp(-(1.5 + 0.25)))
    assert abs(ent[0] - (-p * math.log(p) - (1 - p) * math.log(1 - p))) < 1e-12
    assert abs(pm[0] - p) < 1e-12


def test_entropy_and_confidence_against_scipy():
    scipy_special = pytest.importorskip("scipy.special")
    scipy_stats = pytest.importorskip("scipy.stats")
    rng = np.random.default_rng(6)
    lg = (rng.standard_normal((5, 3000)) * 3).astype(np.float32)
    _, ent, pm = oracle.sample(lg, 0.7, 1, 0)
    p = scipy_special.softmax(lg.astype(np.float64) * np.float64(np.float32(0.7)), axis=1)
    assert np.allclose(ent, scipy_stats.entropy(p, axis=1), rtol=1e-12, atol=1e-12)
    assert np.allclose(pm, p.max(1), rtol=1e-12)


def test_temperature_scales_the_logits():
    rng = np.random.default_rng(2)
    lg = rng.standard_normal((2, 512)).astype(np.float32)
    _, e1, p1 = oracle.sample(lg, 2.0, 3, 0)
    _, e2, p2 = oracle.sample((lg * 2).astype(np.float32), 1.0, 3, 0)
    assert np.allclose(e1, e2, rtol=0, atol=1e-12) and np.allclose(p1, p2, rtol=1e-12)


# ------------------------------------------------------------------ Gumbel-max

@pytest.mark.parametrize("noise", [0, 1])
@pytest.mark.parametrize("inv_temp", [1.0, 0.5])
def test_gumbel_max_samples_the_softmax(inv_temp, noise):
    """The tokens of 40000 positions with the same logits (each position its own
    counters) follow softmax(logits * inv_temp): chi-square at p = 1e-4.  Per group,
    a wrong group sum, a missing ln S, a pick from the wrong end of the CDF or a group's
    noise taken from another group's word skews it far past the bound."""
    base = np.array([0.0, 1.0, 2.0, -1.0, 0.5, 3.0, -2.0, 1.5], np.float32)
    P = 40000
    tok, _, _ = oracle.sample(np.tile(base, (P, 1)), inv_temp, 11, 4, nthreads=8, noise=noise)
    p = np.exp(base.astype(np.float64) * inv_temp)
    p /= p.sum()
    counts = np.bincount(tok, minlength=8)
    chi2 = float(((counts - P * p) ** 2 / (P * p)).sum())
    assert chi2 < 29.9  # chi-square, 7 degrees of freedom, p = 1e-4


def test_grouped_gumbel_max_over_many_groups():
    """24 entries (six groups, one of them far ahead, one far behind) over 30000
    positions and two steps: the per-group form samples softmax, chi-square at
    p = 1e-4 over the entries with an expected count of at least 5."""
    rng = np.random.default_rng(12)
    base = rng.normal(0.0, 1.5, 24).astype(np.float32)
    base[8:12] += 2.5
    base[16:20] -= 4.0
    P = 30000
    p = np.exp(base.astype(np.float64))
    p /= p.sum()
    counts = np.zeros(24)
    for step in (0, 1):
        tok, _, _ = oracle.sample(np.tile(base, (P, 1)), 1.0, 99, step, nthreads=8, noise=0)
        counts += np.bincount(tok, minlength=24)
    n = 2 * P
    keep = n * p >= 5
    other = counts[~keep].sum(), n * p[~keep].sum()
    chi2 = float(((counts[keep] - n * p[keep]) ** 2 / (n * p[keep])).sum())
    if other[1] > 0:
        chi2 += (other[0] - other[1]) ** 2 / other[1]
    dof = int(keep.sum()) - (0 if other[1] > 0 else 1)
    scipy_stats = pytest.importorskip("scipy.stats")
    assert chi2 < scipy_stats.chi2.ppf(1 - 1e-4, dof), (chi2, dof)


def test_gumbel_key_matches_the_definition_in_fp64():
    """key = t + G with G = -ln(-ln U): the fp32 definition stays within a few ulps of
    the same steps taken in fp64."""
    rng = np.random.default_rng(3)
    for w in rng.integers(0, 2 ** 32, 2000, dtype=np.uint64):
        w = int(w)
        u = ((w & 0x7FFFFF) + 0.5) * 2.0 ** -23
        want = 0.75 * 1.25 - math.log(-math.log(u))
        got = oracle.gumbel_key(0.75, 1.25, w)
        assert abs(got - want) <= 8 * _ulp(want) + 1e-6


@pytest.mark.parametrize("noise", [0, 1])
def test_dominant_logit_wins_and_seeds_change_draws(noise):
    lg = np.zeros((4, 256), np.float32)
    lg[:, 77] = 60.0  # exp(60) outweighs any Gumbel noise the 23-bit uniforms can give (G <= 16.7)
    tok, _, _ = oracle.sample(lg, 1.0, 5, 9, noise=noise)
    assert np.all(tok == 77)
    rng = np.random.default_rng(4)
    lg = rng.standard_normal((64, 1024)).astype(np.float32)
    t1, _, _ = oracle.sample(lg, 1.0, 1, 0, noise=noise)
    t2, _, _ = oracle.sample(lg, 1.0, 2, 0, noise=noise)
    t3, _, _ = oracle.sample(lg, 1.0, 1, 1, noise=noise)
    assert np.array_equal(t1, oracle.sample(lg, 1.0, 1, 0, noise=noise)[0])
    assert (t1 != t2).mean() > 0.5 and (t1 != t3).mean() > 0.5


# ------------------------------------------------------------------ groups of four

def test_exp_f32_against_libm():
    """Within 1 fp32 ulp of the exact exponential over [-87, 0] (measured worst 0.9),
    exactly 1 at 0 and 0 below -87; dropping the r^7 term costs 2.5 ulps, dropping the
    low part of ln 2 thousands, a wrong coefficient more."""
    rng = np.random.default_rng(8)
    xs = np.concatenate([-rng.uniform(0, 87, 60000), -np.arange(0, 2000) * 2.0 ** -20,
                         -87 + np.arange(0, 2000) * 1e-4, -(2.0 ** rng.uniform(-40, 6.4, 20000))]).astype(np.float32)
    worst = 0.0
    prev = None
    for x in np.sort(xs)[::3]:
        got = oracle.exp_f32(float(x))
        want = math.exp(float(x))
        worst = max(worst, abs(got - want) / _ulp(want))
        if prev is not None:
            assert got >= prev  # monotone on the sorted grid
        prev = got
    assert worst <= 1.0, worst
    assert oracle.exp_f32(0.0) == 1.0 and oracle.exp_f32(-0.0) == 1.0
    assert oracle.exp_f32(-87.0001) == 0.0 and oracle.exp_f32(-1000.0) == 0.0


def test_group_counter_word_is_a_bijection_onto_the_blocks_counters():
    """Every (counter, word) pair is used by exactly one group, and the groups of
    4,096-entry block b use exactly counters 256 b .. 256 b + 255."""
    G = 1024 * 5
    pairs = [oracle.group_counter_word(g) for g in range(G)]
    assert len(set(pairs)) == G
    for b in range(5):
        cs = {c for c, _ in pairs[1024 * b:1024 * (b + 1)]}
        assert cs == set(range(256 * b, 256 * b + 256))
    assert {w for _, w in pairs} == {0, 1, 2, 3}


def _g_of(word: int) -> float:
    u = ((word & 0x7FFFFF) + 0.5) * 2.0 ** -23
    return -math.log(-math.log(u))


def test_group_key_closed_forms():
    """Four equal logits: key = a + ln 4 + G.  One logit far ahead of the others
    (their e^(t - m) underflows to 0): the key is that entry's per-token key, bit for
    bit (inv_temp 1, so both are fl(a + G)).  Random groups: key - G = ln sum e^t
    within fp32 rounding (a dropped term of the sum, a missing ln or a max taken
    wrongly all fail)."""
    rng = np.random.default_rng(9)
    for w in rng.integers(0, 2 ** 32, 300, dtype=np.uint64):
        w = int(w)
        a = float(np.float32(rng.uniform(-20, 20)))
        got = oracle.group_key([a] * 4, 1.0, w)
        want = a + math.log(4.0) + _g_of(w)
        assert abs(got - want) <= 8 * _ulp(want) + 1e-6
        l4 = np.full(4, a - 200.0, np.float32)
        i = int(rng.integers(0, 4))
        l4[i] = a
        assert oracle.group_key(l4, 1.0, w) == oracle.gumbel_key(a, 1.0, w)
        l4 = rng.normal(0, 3, 4).astype(np.float32)
        it = float(np.float32(rng.uniform(0.3, 2.0)))
        t = l4.astype(np.float64) * it
        want = float(np.log(np.exp(t).sum())) + _g_of(w)
        got = oracle.group_key(l4, it, w)
        assert abs(got - want) <= 16 * _ulp(want) + 2e-6, (got, want)


def test_group_pick_is_the_inverse_cdf():
    """Logits ln 1 .. ln 4 give probabilities 0.1 .. 0.4: the pick is the first i whose
    cumulative probability exceeds U' (checked away from the boundaries); equal logits
    give floor(4 U'); a dominant entry is always picked."""
    rng = np.random.default_rng(10)
    l4 = np.log(np.array([1.0, 2.0, 3.0, 4.0])).astype(np.float32)
    cdf = np.array([0.1, 0.3, 0.6, 1.0])
    seen = set()
    for w in rng.integers(0, 2 ** 32, 3000, dtype=np.uint64):
        w = int(w)
        u = ((w & 0x7FFFFF) + 0.5) * 2.0 ** -23
        if np.min(np.abs(cdf - u)) < 1e-5 or min(abs(u - k / 4) for k in range(5)) < 1e-5:
            continue
        want = int(np.argmax(cdf > u))
        assert oracle.group_pick(l4, 1.0, w) == want
        assert oracle.group_pick([1.5] * 4, 1.0, w) == int(4 * u)
        seen.add(want)
        assert oracle.group_pick([-3.0, 9.0, -80.0, -3.0], 1.0, w) == 1
    assert seen == {0, 1, 2, 3}


def test_one_group_vocabulary_is_the_pick_of_its_second_stream():
    """V = 4: the group wins trivially, so the token is the inverse-CDF pick under word 0
    of counter (0, position, step, 1) of the published generator."""
    rng = np.random.default_rng(11)
    lg = rng.normal(0, 1, (200, 4)).astype(np.float32)
    seed, step = 0x0123_4567_89AB_CDEF, 7
    tok, _, _ = oracle.sample(lg, 0.8, seed, step, noise=0)
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint32)
    for p in range(200):
        w = oracle.philox4x32_10([0, p, step, 1], key)[0]
        assert tok[p] == oracle.group_pick(lg[p], 0.8, int(w))


# ------------------------------------------------------------------ acceptance

def _mlx_vlm_rule(ent, revealed, bound):
    """The page's formula, restated with numpy: sort the unrevealed entropies ascending
    (stable, so ties keep position order), mask = (cumsum - cummax) <= bound in fp32,
    and the first sorted position always."""
    idx = np.nonzero(revealed == 0)[0]
    order = idx[np.argsort(ent[idx], kind="stable")]
    h = ent[order].astype(np.float32)
    cs = np.cumsum(h, dtype=np.float32)
    cm = np.maximum.accumulate(h)
    mask = (cs - cm) <= np.float32(bound)
    if len(mask):
        mask[0] = True
    out = np.zeros(len(ent), np.uint8)
    out[order[mask]] = 1
    return out


def test_entropy_bound_worked_example():
    ent = np.array([0.5, 0.1, 0.3, 0.2], np.float32)
    acc = oracle.accept_entropy(ent, np.zeros(4, np.uint8), 0.35)
    # sorted 0.1 (1), 0.2 (3), 0.3 (2), 0.5 (0): sums before each 0, 0.1, 0.3, 0.6
    assert acc.tolist() == [0, 1, 1, 1]
    assert oracle.accept_entropy(ent, np.zeros(4, np.uint8), -1.0).tolist() == [0, 1, 0, 0]
    assert oracle.accept_entropy(ent, np.array([0, 1, 0, 0], np.uint8), 0.25).tolist() == [0, 0, 1, 1]
    assert oracle.accept_entropy(ent, np.ones(4, np.uint8), 10.0).tolist() == [0, 0, 0, 0]


def test_entropy_bound_equals_the_mlx_vlm_formula():
    rng = np.random.default_rng(5)
    for trial in range(50):
        P = int(rng.integers(1, 400))
        ent = (rng.gamma(1.0, 1.0, P) * rng.choice([1.0, 0.01])).astype(np.float32)
        ent[rng.random(P) < 0.1] = ent[0]  # ties
        revealed = (rng.random(P) < 0.3).astype(np.uint8)
        bound = float(rng.uniform(-0.5, 5.0))
        assert np.array_equal(oracle.accept_entropy(ent, revealed, bound), _mlx_vlm_rule(ent, revealed, bound))


def test_confidence_threshold_rule():
    pm = np.array([0.95, 0.5, 0.91, 0.99, 0.2], np.float32)
    rv = np.array([0, 0, 0, 1, 0], np.uint8)
    assert oracle.accept_confidence(pm, rv, 0.9).tolist() == [1, 0, 1, 0, 0]
    # none above: the most confident unrevealed position, ties to the lower position
    assert oracle.accept_confidence(np.array([0.3, 0.6, 0.6, 0.99], np.float32), np.array([0, 0, 0, 1], np.uint8),
                                    0.9).tolist() == [0, 1, 0, 0]
    assert oracle.accept_confidence(pm, np.ones(5, np.uint8), 0.9).tolist() == [0, 0, 0, 0, 0]
