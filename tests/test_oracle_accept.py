"""Pins for the oracle's greedy accept (CPU only).

The walk is checked against a second formulation (a node is matched when its
parent is matched and its token equals the target's argmax after the parent;
the accept length is one plus the deepest matched depth), against the
hand-derived fixture, and against the extremes: no match at all, and a
target that follows the whole rank-0 chain.
"""
import numpy as np
import pytest

import oracle
from mla_tree_verify_ddt_gb300 import synth
from tests.test_oracle_tree import read_golden, _ints, _lp


def second_formulation(tree, target, b):
    n = int(tree.n_nodes[b])
    matched = [False] * n
    matched[0] = True
    best = 0
    for i in range(1, n):
        p = tree.parent[b, i]
        matched[i] = matched[p] and tree.token[b, i] == target[b, p]
        if matched[i]:
            best = max(best, int(tree.depth[b, i]))
    return 1 + best


def check(tree, target, acc, D):
    B = tree.token.shape[0]
    for b in range(B):
        L = int(acc["accept_len"][b])
        assert L == second_formulation(tree, target, b)
        n = int(tree.n_nodes[b])
        maxdepth = int(tree.depth[b, :n].max())
        assert 1 <= L <= maxdepth + 1 <= D + 1
        idx = acc["accept_idx"][b]
        assert idx[0] == 0 and (idx[L:] == -1).all()
        for k in range(1, L):
            assert tree.parent[b, idx[k]] == idx[k - 1]
            assert tree.token[b, idx[k]] == target[b, idx[k - 1]]
        ct = acc["commit_tok"][b]
        assert list(ct[:L - 1]) == [tree.token[b, idx[k]] for k in range(1, L)]
        assert ct[L - 1] == target[b, idx[L - 1]] == acc["next_root"][b]
        assert (ct[L:] == -1).all()


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_workloads(idx):
    inp = synth.make_inputs(idx, attention=False)
    wl = inp.wl
    t = oracle.tree_build(inp.draft_tok, inp.draft_lp, inp.root_tok, wl.budget, wl.vocab)
    tg = synth.synth_target_argmax(t.depth, t.n_nodes, inp.draft_tok, inp.target_u,
                                   inp.target_alt, wl.p_match)
    acc = oracle.tree_accept(t, tg, wl.D)
    check(t, tg, acc, wl.D)


def test_hand_fixture():
    g = read_golden("tree_hand_d2k2.txt")
    t = oracle.tree_build(_ints(g["tok"]).reshape(1, 2, 2).astype(np.int32),
                          _lp(g["lp"]).reshape(1, 2, 2), np.array([5], np.int32), 3, vocab=1000)
    tg = _ints(g["target"]).astype(np.int32)[None]
    acc = oracle.tree_accept(t, tg, 2)
    assert acc["accept_len"][0] == int(g["accept_len"][0])
    L = int(g["accept_len"][0])
    assert list(acc["accept_idx"][0, :L]) == list(_ints(g["accept_idx"]))
    assert list(acc["commit_tok"][0, :L]) == list(_ints(g["commit_tok"]))
    assert acc["next_root"][0] == int(g["next_root"][0])


def test_never_matching_accepts_only_the_root():
    inp = synth.make_inputs(1, attention=False)
    t = oracle.tree_build(inp.draft_tok, inp.draft_lp, inp.root_tok, 8, 163840)
    tg = np.full((1, 9), -5, np.int32)
    acc = oracle.tree_accept(t, tg, 8)
    assert acc["accept_len"][0] == 1 and acc["next_root"][0] == -5
    check(t, tg, acc, 8)


@pytest.mark.parametrize("D", [1, 4, 8, 16])
def test_full_chain_is_accepted(D):
    rng = np.random.default_rng(D)
    K = 4
    tok = np.stack([rng.choice(1000, K, replace=False) for _ in range(D)])[None].astype(np.int32)
    lp = np.full((1, D, K), -np.inf, np.float32)
    lp[0, :, 0] = -0.01
    lp[0, :, 1] = -5.0  # a second rank keeps the tree branchy
    t = oracle.tree_build(tok, lp, np.array([7], np.int32), 64, 1000)
    tg = np.full((1, 65), 12345, np.int32)
    for i in range(int(t.n_nodes[0])):
        d = int(t.depth[0, i])
        if d < D:
            tg[0, i] = tok[0, d, 0]
    acc = oracle.tree_accept(t, tg, D)
    assert acc["accept_len"][0] == D + 1
    assert list(acc["commit_tok"][0, :D]) == list(tok[0, :, 0])
    assert acc["next_root"][0] == 12345
    check(t, tg, acc, D)


def test_random_targets_cover_lengths():
    rng = np.random.default_rng(3)
    seen = set()
    for trial in range(60):
        D, K = 8, 3
        tok = np.stack([rng.choice(50, K, replace=False) for _ in range(D)])[None].astype(np.int32)
        lp = -np.sort(np.abs(rng.normal(0, 1, (1, D, K))), axis=2).astype(np.float32)
        t = oracle.tree_build(tok, lp, np.array([1], np.int32), 32, 50)
        tg = np.where(rng.random((1, 33)) < 0.85,
                      tok[0, np.clip(t.depth[0], 0, D - 1), 0], rng.integers(0, 50, (1, 33)))
        tg = tg.astype(np.int32)
        acc = oracle.tree_accept(t, tg, D)
        check(t, tg, acc, D)
        seen.add(int(acc["accept_len"][0]))
    assert {1, 2, 3, 4, 5} <= seen
