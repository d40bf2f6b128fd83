"""The per-step sampler through the C ABI against the CPU oracle (sampler_oracle.c).

Both noise forms (0: one Gumbel per group of four entries, 1: one per token) are
checked on every shape.  Bars:
  token     equal element for element (the Gumbel keys are defined in fp32 operation
            by operation, so the argmax and the pick inside a group are the same
            integers on both sides);
  entropy   |gpu - oracle| <= 2e-5 + 2e-5 |oracle| (fp32 streaming sums against fp64);
  pmax      relative 2e-5;
  accept    equal to the oracle's rule applied to the GPU's own fp32 entropy / pmax
            (the rule is decided in fp32; the values themselves are checked above);
  determinism  repeated calls bit-identical.
Inputs: fp32 logits sigma * N(0, 1) (sigma 1 or 3) with a few peaked positions, as an
LM head's logits over a 262,144-token vocabulary look at the scale the model card
gives (268 MB of fp32 logits for a 256-token canvas).
"""
import os

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

NCPU = os.cpu_count() or 1


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a16_moe_expert_router_gb300 import build as libbuild
    libbuild.build()
    from w4a16_moe_expert_router_gb300 import binding
    return binding


def _logits(P, V, sigma, seed):
    rng = np.random.default_rng(seed)
    lg = (rng.standard_normal((P, V), dtype=np.float32) * sigma).astype(np.float32)
    for p in range(0, P, 5):  # peaked positions: low entropy, confident
        lg[p, rng.integers(0, V)] += 12.0
    return lg


def _gpu_sample(B, lg, revealed, inv_temp, rule, bound, seed, step, noise, repeats=1):
    P, V = lg.shape
    cfg = B.make_sampler(P, V, inv_temp, rule, bound, step, seed, noise)
    ws = torch.empty(B.moe_w4a16_sampler_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")
    d_lg = torch.from_numpy(lg).cuda()
    d_rev = torch.from_numpy(revealed).cuda()
    outs = []
    for _ in range(repeats):
        tok = torch.empty(P, dtype=torch.int32, device="cuda")
        ent = torch.empty(P, dtype=torch.float32, device="cuda")
        pm = torch.empty(P, dtype=torch.float32, device="cuda")
        acc = torch.empty(P, dtype=torch.uint8, device="cuda")
        B.moe_w4a16_sample(cfg, d_lg, d_rev, tok, ent, pm, acc, ws)
        outs.append((tok, ent, pm, acc))
    torch.cuda.synchronize()
    return [tuple(t.cpu().numpy() for t in o) for o in outs]


def _check(lg, revealed, inv_temp, rule, bound, seed, step, noise, got):
    tok, ent, pm, acc = got
    o_tok, o_ent, o_pm = oracle.sample(lg, inv_temp, seed, step, nthreads=NCPU, noise=noise)
    assert np.array_equal(tok, o_tok), np.nonzero(tok != o_tok)[0][:10]
    assert np.all(np.abs(ent.astype(np.float64) - o_ent) <= 2e-5 + 2e-5 * np.abs(o_ent)), \
        float(np.abs(ent - o_ent).max())
    assert np.all(np.abs(pm.astype(np.float64) - o_pm) <= 2e-5 * o_pm), float(np.abs(pm / o_pm - 1).max())
    want = (oracle.accept_entropy(ent, revealed, bound) if rule == 0
            else oracle.accept_confidence(pm, revealed, bound))
    assert np.array_equal(acc, want)


NOISE = pytest.mark.parametrize("noise", [0, 1], ids=["group", "token"])


@NOISE
@pytest.mark.parametrize("P,V,sigma,inv_temp,rule,bound", [
    (8, 4096, 1.0, 1.0, 0, 5.0),
    (3, 4100, 3.0, 0.7, 1, 0.5),          # splits of 4,096: one full one and a split of one float4
    (5, 70000, 1.0, 1.0, 0, 30.0),        # 17 splits of one block each (an odd block count), a ragged last split
    (1, 4, 2.0, 1.3, 0, 0.0),             # smallest vocabulary: one split of one float4 (one group)
    (17, 65544, 3.0, 1.0, 1, 0.9),        # 16 full splits of 4,096 and one of 8 elements
    (64, 32768, 1.0, 2.0, 0, 1.0),
    (6, 32772, 1.0, 1.0, 0, 2.0),
    (9, 2060, 3.0, 1.0, 0, 3.0),          # one split of 515 float4s: a full per-token iteration and 3 more; a partial block
    (1, 1000000, 1.0, 1.0, 0, 2.0),       # one position cut into 245 splits: many partials to merge
    (3, 999996, 3.0, 1.0, 1, 0.5),        # 245 splits of 4,096 per position, the last one ragged
    (600, 12300, 3.0, 1.0, 0, 20.0),      # splits of 8,192 (two blocks) and 4,108 (one block and 3 float4s)
    (1000, 13000, 1.0, 0.9, 1, 0.3),      # one split: three full blocks and a partial one
], ids=lambda v: str(v))
def test_sampler_matches_oracle(B, P, V, sigma, inv_temp, rule, bound, noise):
    lg = _logits(P, V, sigma, seed=P * 1000 + V)
    revealed = (np.arange(P) % 3 == 1).astype(np.uint8)
    (got,) = _gpu_sample(B, lg, revealed, inv_temp, rule, bound, seed=0x1234_5678_9abc_def0 + P, step=V % 97,
                         noise=noise)
    _check(lg, revealed, inv_temp, rule, bound, 0x1234_5678_9abc_def0 + P, V % 97, noise, got)


@NOISE
def test_sampler_ties_and_dominant_logits(B, noise):
    """Equal logits (the noise alone decides) and one overwhelming logit per position."""
    P, V = 6, 8192
    lg = np.zeros((P, V), np.float32)
    lg[3:, 100] = 60.0
    revealed = np.zeros(P, np.uint8)
    (got,) = _gpu_sample(B, lg, revealed, 1.0, 0, 2.0, seed=9, step=3, noise=noise)
    _check(lg, revealed, 1.0, 0, 2.0, 9, 3, noise, got)
    assert np.all(got[0][3:] == 100)


@NOISE
@pytest.mark.parametrize("rule,bound", [(0, 40.0), (1, 0.5)])
def test_sampler_full_canvas_step(B, rule, bound, noise):
    """256 positions x 262,144 vocabulary (268 MB of fp32 logits), every position checked;
    three repeated calls bit-identical."""
    P, V = 256, 262144
    lg = _logits(P, V, 3.0, seed=rule)
    revealed = np.zeros(P, np.uint8)
    revealed[::4] = 1
    outs = _gpu_sample(B, lg, revealed, 1.0, rule, bound, seed=77, step=5, noise=noise, repeats=3)
    for o in outs[1:]:
        for a, b in zip(o, outs[0]):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    _check(lg, revealed, 1.0, rule, bound, 77, 5, noise, outs[0])
    assert outs[0][3].sum() >= 1


@NOISE
@pytest.mark.parametrize("rule,bound", [(0, 60.0), (1, 0.4)])
def test_sampler_max_positions(B, rule, bound, noise):
    """P = 1024, the most positions one call takes (the final CTA holds one position
    per thread), over 16,384 tokens; every position checked."""
    P, V = 1024, 16384
    lg = _logits(P, V, 3.0, seed=1024 + rule)
    revealed = (np.arange(P) % 7 == 2).astype(np.uint8)
    (got,) = _gpu_sample(B, lg, revealed, 1.0, rule, bound, seed=4242, step=11, noise=noise)
    _check(lg, revealed, 1.0, rule, bound, 4242, 11, noise, got)


@NOISE
def test_sampler_all_revealed_accepts_nothing(B, noise):
    P, V = 4, 4096
    lg = _logits(P, V, 1.0, 5)
    (got,) = _gpu_sample(B, lg, np.ones(P, np.uint8), 1.0, 0, 10.0, seed=1, step=0, noise=noise)
    assert got[3].sum() == 0


def test_sampler_forms_sample_the_same_distribution(B):
    """Both forms draw from softmax: over 8,192 positions with the same 64 logits (each
    position its own counters), the token frequencies of each form pass a chi-square
    test at p = 1e-4 against softmax, over the tokens with an expected count >= 5."""
    scipy_stats = pytest.importorskip("scipy.stats")
    rng = np.random.default_rng(21)
    base = (rng.standard_normal(64) * 1.2).astype(np.float32)
    P = 1024
    p = np.exp(base.astype(np.float64))
    p /= p.sum()
    for noise in (0, 1):
        counts = np.zeros(64)
        for step in range(8):
            (got,) = _gpu_sample(B, np.tile(base, (P, 1)), np.zeros(P, np.uint8), 1.0, 1, 0.99, seed=5, step=step,
                                 noise=noise)
            counts += np.bincount(got[0], minlength=64)
        n = counts.sum()
        keep = n * p >= 5
        chi2 = float(((counts[keep] - n * p[keep]) ** 2 / (n * p[keep])).sum())
        rest_o, rest_e = counts[~keep].sum(), n * p[~keep].sum()
        dof = int(keep.sum()) - 1
        if rest_e > 0:
            chi2 += (rest_o - rest_e) ** 2 / rest_e
            dof += 1
        assert chi2 < scipy_stats.chi2.ppf(1 - 1e-4, dof), (noise, chi2, dof)


def test_sampler_random_shapes(B):
    """Twelve seeded random configurations (positions 1..1024, vocabularies of 4..300,000
    entries not aligned to any split, logits of scale 0.5..8, both rules, both noise
    forms), every output checked against the oracle."""
    rng = np.random.default_rng(2026)
    for trial in range(12):
        P = int(rng.choice([1, 2, 7, 33, 100, 257, 640, 1024]))
        V = 4 * int(rng.integers(1, 75000 if P < 300 else 4000))
        sigma = float(rng.choice([0.5, 1.0, 3.0, 8.0]))
        inv_temp = float(np.float32(rng.uniform(0.4, 2.5)))
        rule = int(rng.integers(0, 2))
        bound = float(rng.uniform(0.0, 50.0)) if rule == 0 else float(rng.uniform(0.05, 0.95))
        noise = trial % 2
        seed, step = int(rng.integers(0, 2 ** 63)), int(rng.integers(0, 2 ** 32))
        lg = _logits(P, V, sigma, seed=trial)
        revealed = (rng.random(P) < 0.3).astype(np.uint8)
        (got,) = _gpu_sample(B, lg, revealed, inv_temp, rule, bound, seed=seed, step=step, noise=noise)
        _check(lg, revealed, inv_temp, rule, bound, seed, step, noise, got)


@NOISE
@pytest.mark.parametrize("sigma,inv_temp", [(50.0, 0.02), (50.0, 20.0), (0.01, 1.0), (0.5, 300.0)])
def test_sampler_extreme_scales(B, sigma, inv_temp, noise):
    """Logit scales and temperatures far from the workload's (t = logit * inv_temp from
    ~1e-2 to ~1e4).  Tokens exact (the screen's margin scales with |m2| and |K| and must
    never drop the winning token) and acceptance equal to the rule on the GPU's values.
    Entropy and confidence get a bar derived from the fp32 arithmetic: t2 = fl(logit *
    fl(inv_temp log2 e)) is off by up to 2^-23 |t2|, so with T = max |t2| every
    probability is off by a relative ~2^-22 T; pmax within 2e-5 + 2^-22 T relative,
    the entropy within (2e-5 + 2^-22 T)(H + 1)."""
    P, V = 12, 50000
    lg = _logits(P, V, sigma, seed=int(sigma * 100) + int(inv_temp))
    revealed = (np.arange(P) % 4 == 0).astype(np.uint8)
    (got,) = _gpu_sample(B, lg, revealed, inv_temp, 0, 5.0, seed=31, step=2, noise=noise)
    tok, ent, pm, acc = got
    o_tok, o_ent, o_pm = oracle.sample(lg, inv_temp, 31, 2, nthreads=NCPU, noise=noise)
    assert np.array_equal(tok, o_tok), np.nonzero(tok != o_tok)[0][:10]
    T = float(np.abs(lg.astype(np.float64)).max()) * inv_temp * 1.4426950408889634
    rel = 2e-5 + 2.0 ** -22 * T
    assert np.all(np.abs(pm.astype(np.float64) - o_pm) <= rel * o_pm), float(np.abs(pm / o_pm - 1).max())
    assert np.all(np.abs(ent.astype(np.float64) - o_ent) <= rel * (np.abs(o_ent) + 1)), float(np.abs(ent - o_ent).max())
    assert np.array_equal(acc, oracle.accept_entropy(ent, revealed, 5.0))
