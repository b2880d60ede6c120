"""Pins for the oracle's KV commit (the append after accept).

The committed rows are checked against the accepted path rebuilt a second
way: by walking the tree's parent pointers up from the deepest accepted node,
not by reading accept_idx. Every KV row carries a marker (its own row number)
so a row that moved can be told from one that did not."""
import numpy as np
import pytest

import oracle
from mla_tree_verify_ddt_gb300 import synth


def marked_cache(B, Tcap, seed=0):
    """c_kv / k_rope whose every row starts with its (b, row) marker."""
    rng = np.random.default_rng(seed)
    kv = rng.integers(0, 1 << 16, size=(B, Tcap, 512), dtype=np.uint16)
    kr = rng.integers(0, 1 << 16, size=(B, Tcap, 64), dtype=np.uint16)
    for b in range(B):
        kv[b, :, 0] = np.arange(Tcap, dtype=np.uint16)
        kv[b, :, 1] = b
        kr[b, :, 0] = np.arange(Tcap, dtype=np.uint16)
    return kv, kr


def path_by_parents(tree, b, deepest):
    """Root-to-node path of `deepest`, from the parent pointers."""
    path = [deepest]
    while path[-1] != 0:
        path.append(int(tree.parent[b, path[-1]]))
    return path[::-1]


@pytest.mark.parametrize("idx", [0, 1, 2, 3])
def test_commit_matches_the_parent_walk(idx):
    inp = synth.make_inputs(idx, attention=False)
    wl = inp.wl
    tree = oracle.tree_build(inp.draft_tok, inp.draft_lp, inp.root_tok, wl.budget, wl.vocab)
    tgt = synth.synth_target_argmax(tree.depth, tree.n_nodes, inp.draft_tok, inp.target_u, inp.target_alt,
                                    wl.p_match)
    acc = oracle.tree_accept(tree, tgt, wl.D)
    Tcap = int(inp.prefix_len.max()) + wl.budget + 1
    kv, kr = marked_cache(wl.B, Tcap, idx)
    status = np.zeros(wl.B, np.int32)
    nkv, nkr, npl, nst = oracle.kv_commit(acc["accept_len"], acc["accept_idx"], kv, kr, inp.prefix_len, status,
                                          wl.D)
    assert (nst == 0).all()
    for b in range(wl.B):
        T, L = int(inp.prefix_len[b]), int(acc["accept_len"][b])
        assert npl[b] == T + L
        deepest = int(acc["accept_idx"][b, L - 1])
        path = path_by_parents(tree, b, deepest)
        assert len(path) == L
        for k, node in enumerate(path):
            np.testing.assert_array_equal(nkv[b, T + k], kv[b, T + node])
            np.testing.assert_array_equal(nkr[b, T + k], kr[b, T + node])
        # nothing below the prefix end moves
        np.testing.assert_array_equal(nkv[b, :T], kv[b, :T])
        np.testing.assert_array_equal(nkr[b, :T], kr[b, :T])


def test_overlapping_path_hand_example():
    """Path 0 -> 2 -> 3 over T = 5: row 7 goes to row 6 and row 8 to row 7,
    so row 7 is a source and a destination; its old contents must go to 6."""
    kv, kr = marked_cache(1, 16)
    acc_len = np.array([3], np.int32)
    acc_idx = np.array([[0, 2, 3, -1, -1]], np.int32)
    nkv, nkr, npl, nst = oracle.kv_commit(acc_len, acc_idx, kv, kr, np.array([5], np.int32),
                                          np.zeros(1, np.int32), 4)
    assert list(nkv[0, 5:8, 0]) == [5, 7, 8]
    assert list(nkr[0, 5:8, 0]) == [5, 7, 8]
    assert npl[0] == 8 and nst[0] == 0
    np.testing.assert_array_equal(nkv[0, 8:], kv[0, 8:])


def test_root_only_moves_nothing():
    kv, kr = marked_cache(2, 32)
    acc_len = np.array([1, 1], np.int32)
    acc_idx = np.full((2, 9), -1, np.int32)
    acc_idx[:, 0] = 0
    nkv, nkr, npl, nst = oracle.kv_commit(acc_len, acc_idx, kv, kr, np.array([3, 10], np.int32),
                                          np.zeros(2, np.int32), 8)
    np.testing.assert_array_equal(nkv, kv)
    np.testing.assert_array_equal(nkr, kr)
    assert list(npl) == [4, 11]


@pytest.mark.parametrize("case", ["len0", "len_too_long", "not_rising", "past_cap", "bad_root", "neg_prefix"])
def test_bad_sequences_are_flagged_and_untouched(case):
    kv, kr = marked_cache(2, 16)
    D = 4
    acc_len = np.array([3, 2], np.int32)
    acc_idx = np.array([[0, 1, 2, -1, -1], [0, 3, -1, -1, -1]], np.int32)
    pl = np.array([4, 6], np.int32)
    if case == "len0":
        acc_len[0] = 0
    elif case == "len_too_long":
        acc_len[0] = D + 2
    elif case == "not_rising":
        acc_idx[0, 2] = 1
    elif case == "past_cap":
        pl[0] = 14  # rows 14 + 2 = 16 = Tcap
    elif case == "bad_root":
        acc_idx[0, 0] = 1
    elif case == "neg_prefix":
        pl[0] = -1
    nkv, nkr, npl, nst = oracle.kv_commit(acc_len, acc_idx, kv, kr, pl, np.zeros(2, np.int32), D)
    assert nst[0] == oracle.BADINPUT and npl[0] == pl[0]
    np.testing.assert_array_equal(nkv[0], kv[0])
    np.testing.assert_array_equal(nkr[0], kr[0])
    # the other sequence is committed as usual
    assert nst[1] == 0 and npl[1] == 8
    assert list(nkv[1, 6:8, 0]) == [6, 9]
