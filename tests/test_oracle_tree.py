"""Pins for the oracle's draft-tree build (CPU only).

The oracle's heap expansion is checked against things fixed independently of
it: brute-force enumeration of every path on tiny inputs, hand-derived
fixtures, structural invariants, and special cases with known answers.
"""
import os

import numpy as np
import pytest

import oracle
from mla_tree_verify_ddt_gb300 import synth
from tests.brute import brute_tree, enumerate_paths

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            vals[k] = v
    return vals


def _ints(v):
    return np.array([int(x) for x in v], np.int64)


def _lp(v):
    return np.array([float(x) for x in v], np.float32)


def random_rows(rng, B, D, K, vocab=1000, mode="normal"):
    tok = np.empty((B, D, K), np.int32)
    for b in range(B):
        for d in range(D):
            tok[b, d] = rng.choice(vocab, K, replace=False)
    if mode == "normal":
        lp = -np.abs(rng.normal(0, 2, (B, D, K))).astype(np.float32)
    elif mode == "ties":  # few distinct values: many equal scores
        lp = -rng.integers(0, 3, (B, D, K)).astype(np.float32) * np.float32(0.5)
    elif mode == "neginf":
        lp = -np.abs(rng.normal(0, 2, (B, D, K))).astype(np.float32)
        lp[rng.random((B, D, K)) < 0.3] = -np.inf
    elif mode == "zeros":
        lp = np.zeros((B, D, K), np.float32)
    lp = -np.sort(-lp, axis=2)
    return tok, lp.astype(np.float32)


def check_against_brute(tok, lp, root, budget):
    B = tok.shape[0]
    t = oracle.tree_build(tok, lp, root, budget, vocab=1000)
    for b in range(B):
        token, parent, depth, rank, score = brute_tree(tok[b], lp[b], int(root[b]), budget)
        n = len(token)
        assert t.n_nodes[b] == n
        assert t.status[b] == oracle.OK
        np.testing.assert_array_equal(t.token[b, :n], token)
        np.testing.assert_array_equal(t.parent[b, :n], parent)
        np.testing.assert_array_equal(t.depth[b, :n], depth)
        np.testing.assert_array_equal(t.rank[b, :n], rank)
        np.testing.assert_array_equal(t.score[b, :n].view(np.uint32),
                                      np.array(score, np.float32).view(np.uint32))
    return t


@pytest.mark.parametrize("mode", ["normal", "ties", "neginf", "zeros"])
@pytest.mark.parametrize("D,K", [(1, 1), (1, 4), (2, 3), (3, 3), (4, 4), (3, 5), (5, 2)])
def test_heap_equals_brute_force(mode, D, K):
    rng = np.random.default_rng(1000 * D + K + {"normal": 0, "ties": 1, "neginf": 2, "zeros": 3}[mode])
    B = 6
    tok, lp = random_rows(rng, B, D, K, mode=mode)
    root = rng.integers(0, 1000, B).astype(np.int32)
    total = sum(K ** d for d in range(1, D + 1))
    for budget in sorted({1, 2, 3, min(8, total), min(64, total), min(64, total + 3)}):
        check_against_brute(tok, lp, root, budget)


def test_tiny_workload_against_brute_force():
    inp = synth.make_inputs(0, attention=False)
    wl = inp.wl
    t = oracle.tree_build(inp.draft_tok, inp.draft_lp, inp.root_tok, wl.budget, wl.vocab)
    token, parent, depth, rank, score = brute_tree(inp.draft_tok[0], inp.draft_lp[0],
                                                   int(inp.root_tok[0]), wl.budget)
    assert t.n_nodes[0] == len(token) == wl.Qc
    np.testing.assert_array_equal(t.token[0], token)
    np.testing.assert_array_equal(t.parent[0], parent)
    assert len(enumerate_paths(inp.draft_lp[0])) == 340


@pytest.mark.parametrize("name", ["tree_hand_d2k2.txt", "tree_tie_depth.txt"])
def test_hand_fixtures(name):
    g = read_golden(name)
    D, K, budget = int(g["D"][0]), int(g["K"][0]), int(g["budget"][0])
    tok = _ints(g["tok"]).reshape(1, D, K).astype(np.int32)
    lp = _lp(g["lp"]).reshape(1, D, K)
    root = np.array([int(g["root"][0])], np.int32)
    t = oracle.tree_build(tok, lp, root, budget, vocab=1000)
    n = int(g["n_nodes"][0])
    assert t.n_nodes[0] == n
    for key in ("token", "parent", "depth", "rank", "first_child", "next_sibling"):
        np.testing.assert_array_equal(t[key][0, :n], _ints(g[key]), err_msg=key)
    np.testing.assert_array_equal(t.mask[0, :n, 0], _ints(g["mask"]).astype(np.uint64))


def test_hand_fixture_scores():
    g = read_golden("tree_hand_d2k2.txt")
    lp = _lp(g["lp"]).reshape(2, 2)
    t = oracle.tree_build(_ints(g["tok"]).reshape(1, 2, 2).astype(np.int32), lp[None],
                          np.array([5], np.int32), 3, vocab=1000)
    exp = [np.float32(0), lp[0, 0], np.float32(lp[0, 0] + lp[1, 0]), np.float32(lp[0, 0] + lp[1, 1])]
    np.testing.assert_array_equal(t.score[0, :4], np.array(exp, np.float32))


def tree_invariants(t, tok, lp, budget, D, K):
    B, Qc = t.token.shape
    W = t.mask.shape[2]
    for b in range(B):
        n = int(t.n_nodes[b])
        assert 1 <= n <= budget + 1
        finite = sum(1 for _, s in enumerate_paths(lp[b]) if np.isfinite(s)) \
            if sum(K ** d for d in range(1, D + 1)) <= 5000 else None
        if finite is not None and t.status[b] == oracle.OK:
            assert n == 1 + min(budget, finite)
        assert t.parent[b, 0] == -1 and t.depth[b, 0] == 0 and t.score[b, 0] == 0
        for i in range(1, n):
            p = t.parent[b, i]
            assert 0 <= p < i
            assert t.depth[b, i] == t.depth[b, p] + 1 <= D
            assert t.score[b, i] <= t.score[b, i - 1]
            assert t.score[b, i] <= t.score[b, p]
            d, r = t.depth[b, i], t.rank[b, i]
            assert t.token[b, i] == tok[b, d - 1, r]
            # score is the float32 sum of the parent score and this rank's log-prob
            assert np.float32(t.score[b, p] + lp[b, d - 1, r]) == t.score[b, i]
        for i in range(n):
            bits = 0
            j = i
            while j >= 0:
                bits |= 1 << j
                j = int(t.parent[b, j])
            words = [(bits >> (64 * w)) & ((1 << 64) - 1) for w in range(W)]
            assert [int(x) for x in t.mask[b, i]] == words
            assert bin(bits).count("1") == t.depth[b, i] + 1
            kids = [j for j in range(n) if t.parent[b, j] == i]
            assert t.first_child[b, i] == (kids[0] if kids else -1)
            ranks = [t.rank[b, j] for j in kids]
            assert ranks == sorted(ranks) and len(set(ranks)) == len(ranks)
            toks = [t.token[b, j] for j in kids]
            assert len(set(toks)) == len(toks)
            for a, c in zip(kids, kids[1:] + [-1]):
                assert t.next_sibling[b, a] == c
        for i in range(n, Qc):
            assert t.token[b, i] == -1 and t.parent[b, i] == -1 and t.depth[b, i] == -1
            assert t.score[b, i] == -np.inf and not t.mask[b, i].any()


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_workload_invariants(idx):
    inp = synth.make_inputs(idx, attention=False)
    wl = inp.wl
    t = oracle.tree_build(inp.draft_tok, inp.draft_lp, inp.root_tok, wl.budget, wl.vocab)
    tree_invariants(t, inp.draft_tok, inp.draft_lp, wl.budget, wl.D, wl.K)
    assert (t.status == oracle.OK).all()
    if wl.underfull:
        for b in range(wl.underfull):
            assert t.n_nodes[b] == 1 + min(wl.budget, wl.D)
            assert list(t.depth[b, :t.n_nodes[b]]) == list(range(t.n_nodes[b]))
        assert (t.n_nodes[wl.underfull:] == wl.Qc).all()
    else:
        assert (t.n_nodes == wl.Qc).all()


def test_k1_is_a_chain():
    rng = np.random.default_rng(5)
    tok, lp = random_rows(rng, 3, 7, 1)
    root = np.array([1, 2, 3], np.int32)
    for budget in (1, 3, 7, 20):
        t = oracle.tree_build(tok, lp, root, budget, vocab=1000)
        n = 1 + min(budget, 7)
        assert (t.n_nodes == n).all()
        assert (t.parent[:, 1:n] == np.arange(n - 1)).all()


def test_deterministic_rows_give_a_chain():
    rng = np.random.default_rng(6)
    tok, _ = random_rows(rng, 2, 6, 5)
    lp = np.full((2, 6, 5), -np.inf, np.float32)
    lp[:, :, 0] = 0.0
    t = oracle.tree_build(tok, lp, np.array([0, 1], np.int32), 32, vocab=1000)
    assert (t.n_nodes == 7).all()
    assert (t.token[:, 1:7] == tok[:, :, 0]).all()


def test_budget_covers_all_paths():
    rng = np.random.default_rng(7)
    tok, lp = random_rows(rng, 2, 3, 3)
    t = oracle.tree_build(tok, lp, np.array([0, 1], np.int32), 64, vocab=1000)
    assert (t.n_nodes == 1 + 3 + 9 + 27).all()


def test_equal_logprobs_give_breadth_first_order():
    D, K, budget = 3, 3, 30
    tok = np.arange(D * K, dtype=np.int32).reshape(1, D, K)
    lp = np.full((1, D, K), -0.25, np.float32)
    t = oracle.tree_build(tok, lp, np.array([99], np.int32), budget, vocab=1000)
    # breadth-first, children in rank order = depth then lexicographic path
    order = []
    frontier = [()]
    while frontier and len(order) < budget:
        nxt = []
        for p in frontier:
            for r in range(K):
                if len(p) < D:
                    nxt.append(p + (r,))
        order += nxt
        frontier = nxt
    order = order[:budget]
    exp_tok = [99] + [int(tok[0, len(p) - 1, p[-1]]) for p in order]
    assert list(t.token[0, :budget + 1]) == exp_tok


@pytest.mark.parametrize("bad", ["nan", "positive", "unsorted", "token", "root", "posinf"])
def test_bad_rows_are_flagged(bad):
    rng = np.random.default_rng(8)
    tok, lp = random_rows(rng, 3, 3, 3)
    root = np.array([1, 2, 3], np.int32)
    if bad == "nan":
        lp[1, 1, 1] = np.nan
    elif bad == "positive":
        lp[1, 0, 0] = 0.5
    elif bad == "unsorted":
        lp[1, 2] = [-3.0, -1.0, -2.0]
    elif bad == "token":
        tok[1, 2, 2] = 1000
    elif bad == "root":
        root[1] = -1
    elif bad == "posinf":
        lp[1, 0, 0] = np.inf
    t = oracle.tree_build(tok, lp, root, 8, vocab=1000)
    assert list(t.status) == [oracle.OK, oracle.BADINPUT, oracle.OK]
    assert t.n_nodes[1] == 1
    assert t.n_nodes[0] == 9 and t.n_nodes[2] == 9
