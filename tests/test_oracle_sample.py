"""Pins for the oracle's temperature sampling (oracle.tree_sample) against what
the mathematics fixes: closed forms (uniform and two-point distributions),
numpy's argmax for the greedy limit, scipy's softmax for the node
probabilities, and the defining property of inverse-transform sampling (on an
evenly spaced grid of uniforms each token's share of the grid is its
probability, up to one grid point)."""
import math

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from mla_tree_verify_ddt_gb300 import synth

BAD = oracle.BADINPUT


def star_tree(B, Qc, tokens=None):
    """Every node 1..Qc-1 a child of the root; node tokens 0, 1, 2, ..."""
    tok = np.tile(np.arange(Qc, dtype=np.int32), (B, 1)) if tokens is None else np.asarray(tokens, np.int32)
    par = np.zeros((B, Qc), np.int32)
    par[:, 0] = -1
    return oracle.Tree(token=tok, parent=par, n_nodes=np.full(B, Qc, np.int32))


def one_row(logits_row, tau, u):
    """Sample one logit row with each uniform in ``u`` (a column of root-only trees)."""
    u = np.asarray(u, np.float32).reshape(-1, 1)
    n = u.shape[0]
    lg = np.broadcast_to(np.asarray(logits_row, np.float32), (n, 1, len(logits_row))).copy()
    t = oracle.Tree(token=np.zeros((n, 1), np.int32), parent=np.full((n, 1), -1, np.int32),
                    n_nodes=np.ones(n, np.int32))
    tok, _, st = oracle.tree_sample(t, lg, tau, u)
    return tok[:, 0], st


@pytest.mark.parametrize("tau", [0.5, 1.0, 3.0])
def test_equal_logits_sample_is_floor_u_times_v(tau):
    V = 1000
    k = np.arange(0, V, 7)
    u = ((k + 0.5) / V).astype(np.float32)
    tok, st = one_row(np.full(V, 2.5, np.float32), tau, u)
    np.testing.assert_array_equal(tok, np.floor(u.astype(np.float64) * V).astype(np.int32))
    assert (st == 0).all()


def test_uniform_on_a_cdf_boundary_takes_the_upper_token():
    """u exactly equal to C_{k-1} = k/V draws token k (the cumulative sum must
    EXCEED u), checked where every value is exact in binary."""
    V = 64
    k = np.arange(V)
    tok, _ = one_row(np.zeros(V, np.float32), 1.0, (k / V).astype(np.float32))
    np.testing.assert_array_equal(tok, k)


def test_equal_logits_node_probability_is_one_over_v():
    V, Qc = 400, 5
    t = star_tree(1, Qc, [[7, 11, 13, 17, 19]])
    lg = np.full((1, Qc, V), -3.0, np.float32)
    _, p, _ = oracle.tree_sample(t, lg, 0.8, np.full((1, Qc), 0.3, np.float32))
    assert p[0, 0] == 1.0
    np.testing.assert_allclose(p[0, 1:], 1.0 / V, rtol=1e-13)


@pytest.mark.parametrize("tau", [0.25, 1.0, 4.0])
def test_two_point_distribution_threshold(tau):
    V = 64
    row = np.full(V, -np.inf, np.float32)
    a, b = 1.25, -0.5
    row[9], row[40] = a, b
    p9 = 1.0 / (1.0 + math.exp((b - a) / tau))
    eps = 1e-6
    tok, _ = one_row(row, tau, [0.0, p9 - eps, p9 + eps, 0.999999])
    np.testing.assert_array_equal(tok, [9, 9, 40, 40])


@pytest.mark.parametrize("tau", [0.0, -1.0])
def test_greedy_limit_is_first_argmax(tau):
    rng = np.random.default_rng(5)
    B, Qc, V = 3, 6, 300
    lg = rng.standard_normal((B, Qc, V)).astype(np.float32)
    lg[1, 2, 17] = lg[1, 2, 250] = 9.0      # a tie: the lower index wins
    lg[2, 4, :] = -np.inf                   # every logit -inf: index 0
    lg[2, 4, 3] = -np.inf
    tok, _, st = oracle.tree_sample(star_tree(B, Qc), lg, tau, np.zeros((B, Qc), np.float32))
    want = lg.argmax(axis=2)
    np.testing.assert_array_equal(tok, want)
    assert tok[1, 2] == 17 and tok[2, 4] == 0
    assert (st == 0).all()


def test_greedy_node_probability_is_indicator():
    rng = np.random.default_rng(6)
    V, Qc = 50, 4
    lg = rng.standard_normal((1, Qc, V)).astype(np.float32)
    am = int(lg[0, 0].argmax())
    t = star_tree(1, Qc, [[1, am, (am + 1) % V, am]])
    _, p, _ = oracle.tree_sample(t, lg, 0.0, np.zeros((1, Qc), np.float32))
    np.testing.assert_array_equal(p[0], [1.0, 1.0, 0.0, 1.0])


@pytest.mark.parametrize("tau", [0.7, 1.0, 2.5])
def test_inverse_transform_frequencies_on_a_uniform_grid(tau):
    """On N evenly spaced uniforms, token j is drawn for N*p_j points +-1."""
    rng = np.random.default_rng(7)
    V, N = 50, 20000
    row = (rng.standard_normal(V) * 2.0).astype(np.float32)
    row[rng.choice(V, 5, replace=False)] = -np.inf      # zero-probability tokens
    u = ((np.arange(N) + 0.5) / N).astype(np.float32)
    tok, _ = one_row(row, tau, u)
    counts = np.bincount(tok, minlength=V)
    p = softmax(row.astype(np.float64) / tau)
    assert np.all(np.abs(counts - N * p) <= 1.0 + 1e-9), np.abs(counts - N * p).max()
    assert counts[np.isneginf(row)].sum() == 0
    # and the draws are monotone in u (an inverse transform)
    assert np.all(np.diff(tok) >= 0)


def test_node_probabilities_match_softmax_of_parent_row():
    rng = synth.rng_for(0)
    wl = synth.WORKLOADS[0]
    inp = synth.make_inputs(0, attention=False)
    t = oracle.tree_build(inp.draft_tok, inp.draft_lp, inp.root_tok, wl.budget, wl.vocab)
    lg = synth.target_logits(rng, t.depth, t.n_nodes, inp.draft_tok, wl.vocab)
    for tau in (0.6, 1.0, 1.7):
        _, p, st = oracle.tree_sample(t, lg, tau, synth.sample_uniforms(rng, 1, wl.Qc))
        assert (st == 0).all()
        for c in range(1, int(t.n_nodes[0])):
            par = int(t.parent[0, c])
            want = softmax(lg[0, par].astype(np.float64) / tau)[t.token[0, c]]
            assert p[0, c] == pytest.approx(want, rel=1e-12)
        # the children of one node are distinct tokens: their probabilities
        # add up to at most 1
        for i in range(int(t.n_nodes[0])):
            kids = [c for c in range(1, int(t.n_nodes[0])) if t.parent[0, c] == i]
            assert sum(p[0, c] for c in kids) <= 1.0 + 1e-12


def test_rows_without_a_distribution_are_flagged():
    V, Qc = 40, 4
    t = star_tree(4, Qc)
    lg = np.zeros((4, Qc, V), np.float32)
    lg[0, 0, 5] = np.nan                 # NaN in the root row
    lg[1, 2, :] = -np.inf                # no finite logit (tau > 0)
    lg[2, 1, 7] = np.inf                 # +inf (tau > 0)
    u = np.full((4, Qc), 0.5, np.float32)
    tok, p, st = oracle.tree_sample(t, lg, 1.0, u)
    assert tok[0, 0] == -1 and tok[1, 2] == -1 and tok[2, 1] == -1
    assert list(st) == [BAD, BAD, BAD, 0]
    assert (p[0, 1:] == 0).all()         # children of the NaN root row
    assert (tok[3] >= 0).all()
    # greedy: only the NaN row has no answer; +inf and all -inf rows are fine
    tok, p, st = oracle.tree_sample(t, lg, 0.0, u)
    assert tok[0, 0] == -1 and tok[1, 2] == 0 and tok[2, 1] == 7
    assert list(st) == [BAD, 0, 0, 0]


def test_child_token_outside_vocab_is_flagged():
    V, Qc = 16, 3
    t = star_tree(1, Qc, [[0, 5, 16]])
    _, p, st = oracle.tree_sample(t, np.zeros((1, Qc, V), np.float32), 1.0,
                                  np.full((1, Qc), 0.5, np.float32))
    assert st[0] == BAD and p[0, 2] == 0.0 and p[0, 1] == pytest.approx(1.0 / V)


def test_uniforms_outside_zero_one_clamp_to_nonzero_tokens():
    V = 20
    row = np.full(V, -np.inf, np.float32)
    row[3:15] = np.linspace(-1, 1, 12, dtype=np.float32)
    tok, st = one_row(row, 1.0, [-0.5, 0.0, 1.0, 2.0, np.nan])
    np.testing.assert_array_equal(tok, [3, 3, 14, 14, 14])
    assert (st == 0).all()


def test_padding_slots():
    V, Qc = 12, 5
    t = star_tree(2, Qc)
    t["n_nodes"] = np.array([2, 5], np.int32)
    tok, p, _ = oracle.tree_sample(t, np.zeros((2, Qc, V), np.float32), 1.0,
                                   np.full((2, Qc), 0.1, np.float32))
    assert list(tok[0, 2:]) == [-1, -1, -1] and list(p[0, 2:]) == [0, 0, 0]
    assert (tok[1] >= 0).all()


def test_sampled_accept_probability_equals_children_mass():
    """Chained with the greedy walk: over a uniform grid for the root, the share
    of draws that accept a child equals the children's total probability."""
    V, Qc, N = 30, 4, 6000
    rng = np.random.default_rng(11)
    base = rng.standard_normal((1, Qc, V)).astype(np.float32)
    t1 = star_tree(1, Qc, [[0, 4, 9, 21]])
    _, p, _ = oracle.tree_sample(t1, base, 0.9, np.full((1, Qc), 0.5, np.float32))
    lg = np.repeat(base, N, axis=0)
    t = star_tree(N, Qc, np.repeat([[0, 4, 9, 21]], N, axis=0))
    u = np.repeat(rng.random((1, Qc), dtype=np.float32), N, axis=0)
    u[:, 0] = ((np.arange(N) + 0.5) / N).astype(np.float32)
    tok, _, _ = oracle.tree_sample(t, lg, 0.9, u)
    acc = oracle.tree_accept(t, tok, D=1)
    share = float((acc["accept_len"] == 2).mean())
    assert abs(share - p[0, 1:].sum()) <= 3.0 / N
    # the first committed token is always the root's sample
    np.testing.assert_array_equal(acc["commit_tok"][:, 0], tok[:, 0])
