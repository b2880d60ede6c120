"""GPU draft-tree build and greedy accept vs the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from mla_tree_verify_ddt_gb300 import ddtree, synth
from tests import gpu_util as gu
from tests.test_oracle_tree import random_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ddtree.lib()
    torch.cuda.init()


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_build_matches_oracle_on_workloads(idx):
    inp = synth.make_inputs(idx, attention=False)
    wl = inp.wl
    gt = ddtree.ddt_tree_build(gu.i32_dev(inp.draft_tok), gu.f32_dev(inp.draft_lp),
                               gu.i32_dev(inp.root_tok), wl.budget, wl.vocab)
    torch.cuda.synchronize()
    gu.assert_tree_equal(gt, gu.oracle_tree(inp))


SWEEP = [(D, K, budget) for D, K, budget in [
    (1, 1, 1), (1, 16, 16), (2, 2, 64), (3, 5, 7), (4, 4, 8), (5, 3, 64), (8, 8, 8), (8, 8, 16),
    (15, 4, 32), (16, 8, 64), (16, 16, 64), (16, 1, 64), (6, 16, 33), (12, 2, 63)]]


@pytest.mark.parametrize("mode", ["normal", "ties", "neginf", "zeros"])
@pytest.mark.parametrize("D,K,budget", SWEEP)
def test_build_sweep(mode, D, K, budget):
    rng = np.random.default_rng(D * 1000 + K * 10 + budget)
    B = 9
    tok, lp = random_rows(rng, B, D, K, vocab=5000, mode=mode)
    root = rng.integers(0, 5000, B).astype(np.int32)
    gt = ddtree.ddt_tree_build(gu.i32_dev(tok), gu.f32_dev(lp), gu.i32_dev(root), budget, 5000)
    torch.cuda.synchronize()
    ot = oracle.tree_build(tok, lp, root, budget, 5000)
    gu.assert_tree_equal(gt, ot)


@pytest.mark.parametrize("bad", ["nan", "positive", "unsorted", "token", "root"])
def test_bad_rows_flagged_on_device(bad):
    rng = np.random.default_rng(8)
    tok, lp = random_rows(rng, 3, 3, 3, vocab=1000)
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
        root[1] = 1000
    gt = ddtree.ddt_tree_build(gu.i32_dev(tok), gu.f32_dev(lp), gu.i32_dev(root), 8, 1000)
    st = ddtree.ddt_read_device_status(gt.status)
    assert list(st) == [ddtree.DDT_OK, ddtree.DDT_E_BADINPUT, ddtree.DDT_OK]
    gu.assert_tree_equal(gt, oracle.tree_build(tok, lp, root, 8, 1000))


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_accept_matches_oracle(idx):
    inp = synth.make_inputs(idx, attention=False)
    wl = inp.wl
    ot = gu.oracle_tree(inp)
    tg = gu.target_for(inp, ot)
    gt = ddtree.ddt_tree_build(gu.i32_dev(inp.draft_tok), gu.f32_dev(inp.draft_lp),
                               gu.i32_dev(inp.root_tok), wl.budget, wl.vocab)
    acc = ddtree.ddt_tree_accept(gt, gu.i32_dev(tg))
    torch.cuda.synchronize()
    ref = oracle.tree_accept(ot, tg, wl.D)
    for k in ("accept_len", "accept_idx", "commit_tok", "next_root"):
        np.testing.assert_array_equal(getattr(acc, k).cpu().numpy(), ref[k], err_msg=k)


def test_accept_lengths_cover_the_range():
    """Chained on the device (build -> accept, no host round-trip), with
    targets that accept anything from the root alone to the whole depth."""
    rng = np.random.default_rng(77)
    D, K, budget, B = 8, 4, 64, 48
    tok, lp = random_rows(rng, B, D, K, vocab=3000)
    root = rng.integers(0, 3000, B).astype(np.int32)
    ot = oracle.tree_build(tok, lp, root, budget, 3000)
    tg = np.empty((B, budget + 1), np.int32)
    for b in range(B):
        p = b / (B - 1)
        for i in range(budget + 1):
            d = int(ot.depth[b, i])
            tg[b, i] = tok[b, d, 0] if (0 <= d < D and rng.random() < p) else rng.integers(0, 3000)
    gt = ddtree.ddt_tree_build(gu.i32_dev(tok), gu.f32_dev(lp), gu.i32_dev(root), budget, 3000)
    acc = ddtree.ddt_tree_accept(gt, gu.i32_dev(tg))
    torch.cuda.synchronize()
    ref = oracle.tree_accept(ot, tg, D)
    got = acc.accept_len.cpu().numpy()
    np.testing.assert_array_equal(got, ref["accept_len"])
    np.testing.assert_array_equal(acc.commit_tok.cpu().numpy(), ref["commit_tok"])
    assert got.min() == 1 and got.max() == D + 1
    assert len(set(got.tolist())) >= 6
