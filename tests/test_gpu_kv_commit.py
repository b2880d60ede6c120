"""GPU parity of ddt_kv_commit (the append of the accepted path's keys after
accept) against the oracle: bit-exact on the whole cache, the prefix lengths
and the status words, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from mla_tree_verify_ddt_gb300 import ddtree, synth
from tests import gpu_util as gu
from tests.test_oracle_kv_commit import marked_cache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ddtree.lib()
    torch.cuda.init()


def u16_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def accept_dev(acc):
    return ddtree.Accept(gu.i32_dev(acc["accept_len"]), gu.i32_dev(acc["accept_idx"]),
                         gu.i32_dev(acc["commit_tok"]), gu.i32_dev(acc["next_root"]))


def run_gpu(acc_dev, kv, kr, pl, st):
    dkv, dkr, dpl, dst = u16_dev(kv), u16_dev(kr), gu.i32_dev(pl), gu.i32_dev(st)
    ddtree.ddt_kv_commit(acc_dev, dkv, dkr, dpl, dst)
    torch.cuda.synchronize()
    return (dkv.cpu().numpy().view(np.uint16), dkr.cpu().numpy().view(np.uint16), dpl.cpu().numpy(),
            dst.cpu().numpy())


def assert_same(got, ref):
    for g, r, name in zip(got, ref, ("c_kv", "k_rope", "prefix_len", "status")):
        np.testing.assert_array_equal(g, r, err_msg=name)


@pytest.mark.parametrize("idx", [0, 1, 2, 3])
def test_commit_parity_on_the_oracle_accept(idx):
    inp = synth.make_inputs(idx, attention=False)
    wl = inp.wl
    tree = oracle.tree_build(inp.draft_tok, inp.draft_lp, inp.root_tok, wl.budget, wl.vocab)
    tgt = synth.synth_target_argmax(tree.depth, tree.n_nodes, inp.draft_tok, inp.target_u, inp.target_alt,
                                    wl.p_match)
    acc = oracle.tree_accept(tree, tgt, wl.D)
    Tcap = int(inp.prefix_len.max()) + wl.budget + 1
    kv, kr = marked_cache(wl.B, Tcap, idx)
    st = np.zeros(wl.B, np.int32)
    ref = oracle.kv_commit(acc["accept_len"], acc["accept_idx"], kv, kr, inp.prefix_len, st, wl.D)
    assert_same(run_gpu(accept_dev(acc), kv, kr, inp.prefix_len, st), ref)


@pytest.mark.parametrize("idx", [0, 2, 3])
def test_gpu_chain_build_accept_commit(idx):
    """Tree build, accept and commit all on the GPU, against the oracle chain."""
    inp = synth.make_inputs(idx, attention=False)
    wl = inp.wl
    ot = oracle.tree_build(inp.draft_tok, inp.draft_lp, inp.root_tok, wl.budget, wl.vocab)
    tgt = synth.synth_target_argmax(ot.depth, ot.n_nodes, inp.draft_tok, inp.target_u, inp.target_alt,
                                    wl.p_match)
    oacc = oracle.tree_accept(ot, tgt, wl.D)
    gt = ddtree.ddt_tree_build(gu.i32_dev(inp.draft_tok), gu.f32_dev(inp.draft_lp), gu.i32_dev(inp.root_tok),
                               wl.budget, wl.vocab)
    gacc = ddtree.ddt_tree_accept(gt, gu.i32_dev(tgt))
    Tcap = int(inp.prefix_len.max()) + wl.budget + 1
    kv, kr = marked_cache(wl.B, Tcap, 100 + idx)
    st = np.zeros(wl.B, np.int32)
    ref = oracle.kv_commit(oacc["accept_len"], oacc["accept_idx"], kv, kr, inp.prefix_len, st, wl.D)
    assert_same(run_gpu(gacc, kv, kr, inp.prefix_len, st), ref)


def test_overlapping_path_and_bad_sequences():
    """Sequence 0 commits the overlapping path 0 -> 2 -> 3; sequences 1-3 are
    flagged (path not rising, past the key capacity, length 0) and untouched."""
    D, Tcap = 4, 16
    kv, kr = marked_cache(4, Tcap, 7)
    acc = dict(accept_len=np.array([3, 3, 2, 0], np.int32),
               accept_idx=np.array([[0, 2, 3, -1, -1], [0, 2, 2, -1, -1], [0, 1, -1, -1, -1],
                                    [0, -1, -1, -1, -1]], np.int32),
               commit_tok=np.zeros((4, D + 1), np.int32), next_root=np.zeros(4, np.int32))
    pl = np.array([5, 2, 15, 3], np.int32)
    st = np.zeros(4, np.int32)
    ref = oracle.kv_commit(acc["accept_len"], acc["accept_idx"], kv, kr, pl, st, D)
    assert list(ref[3]) == [0, oracle.BADINPUT, oracle.BADINPUT, oracle.BADINPUT]
    assert_same(run_gpu(accept_dev(acc), kv, kr, pl, st), ref)
