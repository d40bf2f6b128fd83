"""Routing edge cases through the C ABI (moe_w4a16_route) against the oracle.

The router takes the top-k of each token's fp32 logits in descending order with
ties to the lower expert index, compared as fp32 values (so -0 ties +0), then the
softmax over the k selected logits (model card "srswti/axe-diffusion-ksl-xe",
"what the model is": top-8 of 128 experts).  N(0, 1) logits practically never tie,
so these inputs are built to: all-equal rows, +-0 mixtures, duplicated values
straddling the k-th place, 256 experts drawn from a handful of values, and a
single token.  topk_idx, expert_offsets and pair_list must equal the oracle's
element for element; topk_w within 1e-6 relative.
"""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

W_REL = 1e-6


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a16_moe_expert_router_gb300 import build as libbuild
    libbuild.build()
    from w4a16_moe_expert_router_gb300 import binding
    return binding


def _route(B, lg, k, repeats=1):
    T, E = lg.shape
    sh = B.make_shape(T, 128, 64, E, k, 64, 64)
    routing = B.RoutingBuffers(
        topk_idx=torch.empty((T, k), dtype=torch.int32, device="cuda"),
        topk_w=torch.empty((T, k), dtype=torch.float32, device="cuda"),
        expert_offsets=torch.empty((E + 1,), dtype=torch.int32, device="cuda"),
        pair_list=torch.empty((T * k,), dtype=torch.int32, device="cuda"),
    )
    ws = torch.empty((B.moe_w4a16_workspace_bytes(sh),), dtype=torch.uint8, device="cuda")
    B.moe_w4a16_workspace_init(ws)
    d_lg = torch.from_numpy(np.ascontiguousarray(lg, np.float32)).cuda()
    runs = []
    for _ in range(repeats):  # the same workspace: the one-launch routing's ticket must come back to 0
        for t in (routing.topk_idx, routing.expert_offsets, routing.pair_list):
            t.fill_(-1)
        B.moe_w4a16_route(sh, d_lg, routing, ws)
        torch.cuda.synchronize()
        runs.append(tuple(t.cpu().numpy() for t in (routing.topk_idx, routing.topk_w, routing.expert_offsets,
                                                    routing.pair_list)))
    for r in runs[1:]:
        assert all(np.array_equal(a, b) for a, b in zip(r, runs[0]))
    return runs[0]


def _check(B, lg, k, repeats=1):
    idx_g, w_g, off_g, pl_g = _route(B, lg, k, repeats)
    idx_o, w_o = oracle.route(lg, k)
    off_o, pl_o = oracle.permute(idx_o, lg.shape[1])
    assert np.array_equal(idx_g, idx_o), np.argwhere(idx_g != idx_o)[:5]
    assert np.array_equal(off_g, off_o)
    assert np.array_equal(pl_g, pl_o)
    assert np.all(np.abs(w_g.astype(np.float64) - w_o) <= W_REL * np.abs(w_o))
    return idx_g, w_g


def test_all_equal_logits_pick_the_lowest_experts(B):
    lg = np.full((16, 128), 0.375, np.float32)
    idx, w = _check(B, lg, 8)
    assert np.array_equal(idx, np.tile(np.arange(8, dtype=np.int32), (16, 1)))
    assert np.allclose(w, 1.0 / 8, rtol=0, atol=1e-7)


def test_signed_zeros_tie(B):
    """Rows of +0 and -0 only (all tied: lowest indices win whatever the signs),
    then rows with a few positive values among signed zeros."""
    rng = np.random.default_rng(11)
    lg = np.where(rng.random((24, 128)) < 0.5, np.float32(-0.0), np.float32(0.0)).astype(np.float32)
    for t in range(12, 24):
        lg[t, rng.choice(128, 3, replace=False)] = rng.uniform(0.5, 1.0, 3).astype(np.float32)
    idx, _ = _check(B, lg, 8)
    assert np.array_equal(idx[:12], np.tile(np.arange(8, dtype=np.int32), (12, 1)))


def test_duplicates_straddle_the_kth_place(B):
    """Each row has its k-th largest value repeated at several experts, some inside the
    top-k and some beyond it: the lower indices among the duplicates are selected."""
    rng = np.random.default_rng(12)
    T, E, k = 40, 128, 8
    lg = rng.uniform(-3.0, -1.0, (T, E)).astype(np.float32)
    for t in range(T):
        top = rng.choice(E, 5, replace=False)
        lg[t, top] = np.float32(2.0) + np.arange(5, dtype=np.float32)
        dup = rng.choice(np.setdiff1d(np.arange(E), top), 3 + t % 6, replace=False)
        lg[t, dup] = np.float32(1.25)
    idx, _ = _check(B, lg, k)
    for t in range(T):
        ties = np.nonzero(lg[t] == np.float32(1.25))[0]
        assert np.array_equal(np.sort(idx[t, 5:]), np.sort(ties)[:3])


def test_256_experts_many_ties(B):
    """E = 256, k = 8, logits drawn from six values: ties at and across the k-th place."""
    rng = np.random.default_rng(13)
    lg = rng.choice(np.array([-1.0, -0.0, 0.0, 0.5, 1.0, 1.5], np.float32), (64, 256)).astype(np.float32)
    _check(B, lg, 8)


def test_one_token(B):
    rng = np.random.default_rng(14)
    _check(B, rng.standard_normal((1, 128), dtype=np.float32), 8)


@pytest.mark.parametrize("T,E,k", [(1, 256, 8), (7, 3, 3), (9, 256, 1), (129, 64, 4)])
def test_ragged_shapes_with_ties(B, T, E, k):
    rng = np.random.default_rng(T * 1000 + E)
    lg = rng.integers(-2, 3, (T, E)).astype(np.float32)
    _check(B, lg, k)


@pytest.mark.parametrize("T,E,k", [(512, 128, 8), (513, 128, 8), (504, 256, 8), (1024, 128, 8), (4097, 256, 3),
                                   (20000, 128, 8)])
def test_one_launch_and_three_launch_routing(B, T, E, k):
    """Up to 64 top-k CTAs (512 tokens) routing is one launch, whose last CTA groups
    every pair; above that it takes three launches (top-k, per-expert prefix over
    CTAs, placement).  Both sides of the boundary, and sizes far above it, against
    the oracle, three calls each on one workspace."""
    rng = np.random.default_rng(T + E + k)
    lg = rng.standard_normal((T, E), dtype=np.float32)
    lg[::7] = np.round(lg[::7])  # ties on some rows
    _check(B, lg, k, repeats=3)
