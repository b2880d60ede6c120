"""GPU parity of ddt_verify_mla_attn_paged (the block-table KV cache): on a
shuffled pool with junk rows it must give the contiguous kernel's output bit
for bit (same data, same arithmetic), and the oracle's within the attention
tolerance."""
import numpy as np
import pytest
import torch

import oracle
from mla_tree_verify_ddt_gb300 import ddtree, synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ddtree.lib()
    torch.cuda.init()


def paged_inputs(inp, n_nodes, seed, hide_past_end=True):
    """A pool holding every (b, p) row of the contiguous cache at a random
    row, plus junk rows; entries past each sequence's key end are -1."""
    rng = np.random.default_rng(seed)
    B, Tcap = inp.c_kv.shape[:2]
    P = B * Tcap + 37
    perm = rng.permutation(P)
    kvi = perm[: B * Tcap].reshape(B, Tcap).astype(np.int32)
    pool_kv = rng.integers(0, 1 << 16, size=(P, 512), dtype=np.uint16)
    pool_kr = rng.integers(0, 1 << 16, size=(P, 64), dtype=np.uint16)
    pool_kv[kvi.ravel()] = inp.c_kv.reshape(-1, 512)
    pool_kr[kvi.ravel()] = inp.k_rope.reshape(-1, 64)
    if hide_past_end:
        for b in range(B):
            kvi[b, int(inp.prefix_len[b]) + int(n_nodes[b]):] = -1
    return pool_kv, pool_kr, kvi


def bf16(a):
    return gu.bf16_dev(a)


@pytest.mark.parametrize("idx", [0, 1, 2])
def test_paged_matches_contiguous_bitwise(idx):
    inp = synth.make_inputs(idx)
    wl = inp.wl
    tree = ddtree.ddt_tree_build(gu.i32_dev(inp.draft_tok), gu.f32_dev(inp.draft_lp), gu.i32_dev(inp.root_tok),
                                 wl.budget, wl.vocab)
    n_nodes = tree.n_nodes.cpu().numpy()
    dev = gu.attn_dev(inp)
    ref_out, ref_lse = ddtree.ddt_verify_mla_attn(*dev, tree, inp.scale)
    pool_kv, pool_kr, kvi = paged_inputs(inp, n_nodes, 11 + idx)
    out, lse = ddtree.ddt_verify_mla_attn_paged(dev[0], dev[1], bf16(pool_kv), bf16(pool_kr), dev[4],
                                                gu.i32_dev(kvi), tree, inp.scale)
    torch.cuda.synchronize()
    assert (tree.status.cpu().numpy() == 0).all()
    np.testing.assert_array_equal(out.cpu().numpy().view(np.uint32), ref_out.cpu().numpy().view(np.uint32))
    np.testing.assert_array_equal(lse.cpu().numpy().view(np.uint32), ref_lse.cpu().numpy().view(np.uint32))


def test_paged_matches_the_oracle():
    inp = synth.make_inputs(0)
    wl = inp.wl
    ot = gu.oracle_tree(inp)
    tree = ddtree.ddt_tree_build(gu.i32_dev(inp.draft_tok), gu.f32_dev(inp.draft_lp), gu.i32_dev(inp.root_tok),
                                 wl.budget, wl.vocab)
    pool_kv, pool_kr, kvi = paged_inputs(inp, ot.n_nodes, 5)
    gkv, gkr = oracle.gather_paged(pool_kv, pool_kr, kvi)
    ref_out, ref_lse = oracle.attn_all(inp.q_lat, inp.q_rope, gkv, gkr, inp.prefix_len, ot.mask, ot.n_nodes,
                                       inp.scale)
    dev = gu.attn_dev(inp)
    out, lse = ddtree.ddt_verify_mla_attn_paged(dev[0], dev[1], bf16(pool_kv), bf16(pool_kr), dev[4],
                                                gu.i32_dev(kvi), tree, inp.scale)
    torch.cuda.synchronize()
    B, Qc, H = wl.B, wl.Qc, wl.H
    gu.check_rows(out.cpu().numpy().reshape(-1, 512), lse.cpu().numpy().ravel(),
                  ref_out.reshape(-1, 512), ref_lse.ravel(), "paged tiny")


def test_bad_entry_below_the_key_end_is_flagged():
    inp = synth.make_inputs(0)
    wl = inp.wl
    tree = ddtree.ddt_tree_build(gu.i32_dev(inp.draft_tok), gu.f32_dev(inp.draft_lp), gu.i32_dev(inp.root_tok),
                                 wl.budget, wl.vocab)
    n_nodes = tree.n_nodes.cpu().numpy()
    pool_kv, pool_kr, kvi = paged_inputs(inp, n_nodes, 9)
    kvi[0, 3] = pool_kv.shape[0]  # one past the pool, inside the prefix
    dev = gu.attn_dev(inp)
    ddtree.ddt_verify_mla_attn_paged(dev[0], dev[1], bf16(pool_kv), bf16(pool_kr), dev[4], gu.i32_dev(kvi), tree,
                                     inp.scale)
    torch.cuda.synchronize()
    assert tree.status.cpu().numpy()[0] == ddtree.DDT_E_BADINPUT


@pytest.mark.parametrize("idx", [1, 2])
def test_paged_matches_the_oracle_on_sampled_rows(idx):
    """Single stream (its keys split over many ranges, then merged) and small
    batch (ragged prefixes), in the launch configuration the benchmark times:
    sampled rows against the oracle on the gathered cache."""
    inp = synth.make_inputs(idx)
    wl = inp.wl
    ot = gu.oracle_tree(inp)
    tree = ddtree.ddt_tree_build(gu.i32_dev(inp.draft_tok), gu.f32_dev(inp.draft_lp), gu.i32_dev(inp.root_tok),
                                 wl.budget, wl.vocab)
    pool_kv, pool_kr, kvi = paged_inputs(inp, ot.n_nodes, 21 + idx)
    dev = gu.attn_dev(inp)
    out, lse = ddtree.ddt_verify_mla_attn_paged(dev[0], dev[1], bf16(pool_kv), bf16(pool_kr), dev[4],
                                                gu.i32_dev(kvi), tree, inp.scale)
    torch.cuda.synchronize()
    assert (tree.status.cpu().numpy() == 0).all()
    rows = gu.sample_rows(wl.B, wl.Qc, wl.H, ot.n_nodes, seed=40 + idx)
    gkv, gkr = oracle.gather_paged(pool_kv, pool_kr, kvi)
    ref_out, ref_lse, _ = oracle.attn_rows(inp.q_lat, inp.q_rope, gkv, gkr, inp.prefix_len, ot.mask, ot.n_nodes,
                                           inp.scale, rows)
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    b, i, h = rows[:, 0], rows[:, 1], rows[:, 2]
    gu.check_rows(o[b, i, h], l[b, i, h], ref_out, ref_lse, f"paged {wl.name}")
