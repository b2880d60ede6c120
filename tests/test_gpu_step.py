"""The whole verify step through ddt_verify_step, chained on one stream with
no host round-trip, against the oracle's chain; CUDA-graph capture and
replay; the bounded-wait self-test."""
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


def make_step(inp, tg):
    wl = inp.wl
    q_lat, q_rope, c_kv, k_rope, pl = gu.attn_dev(inp)
    return ddtree.VerifyStep(gu.i32_dev(inp.draft_tok), gu.f32_dev(inp.draft_lp),
                             gu.i32_dev(inp.root_tok), wl.vocab, wl.budget, q_lat, q_rope, c_kv,
                             k_rope, pl, gu.i32_dev(tg), inp.scale)


def check_step(step, inp, ot, tg, rows=None):
    wl = inp.wl
    gu.assert_tree_equal(step.tree, ot)
    ref = oracle.tree_accept(ot, tg, wl.D)
    for k in ("accept_len", "accept_idx", "commit_tok", "next_root"):
        np.testing.assert_array_equal(getattr(step.acc, k).cpu().numpy(), ref[k], err_msg=k)
    out, lse = step.out.cpu().numpy(), step.lse.cpu().numpy()
    if rows is None:
        ref_out, ref_lse = oracle.attn_all(inp.q_lat, inp.q_rope, inp.c_kv, inp.k_rope,
                                           inp.prefix_len, ot.mask, ot.n_nodes, inp.scale)
        gu.check_rows(out, lse, ref_out, ref_lse, wl.name)
    else:
        ref_out, ref_lse = gu.oracle_rows(inp, ot, rows)
        gu.check_rows(out[rows[:, 0], rows[:, 1], rows[:, 2]],
                      lse[rows[:, 0], rows[:, 1], rows[:, 2]], ref_out, ref_lse, wl.name)


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_step_matches_oracle_chain(idx):
    inp = synth.make_inputs(idx)
    wl = inp.wl
    ot = gu.oracle_tree(inp)
    tg = gu.target_for(inp, ot)
    step = make_step(inp, tg)
    step.run()
    torch.cuda.synchronize()
    rows = None if idx <= 1 else gu.sample_rows(wl.B, wl.Qc, wl.H, ot.n_nodes, seed=100 + idx,
                                                per_seq_heads=1, max_seqs=4)
    check_step(step, inp, ot, tg, rows)
    st = ddtree.ddt_read_device_status(step.tree.status)
    assert (st == ddtree.DDT_OK).all()


def test_split_keys_step_with_flagged_and_underfull_sequences():
    """With the key range split, the merge kernel also runs the accept walk:
    a chain (underfull) tree, a full tree, and a sequence whose prefix leaves
    no room for its nodes (flagged, zero output), against the oracle chain."""
    from tests.test_gpu_attn import custom_inputs, nan_tail
    inp = custom_inputs(21, 3, 4, 4, 8, 4, [2500, 1200, 3000], underfull=1)
    wl = inp.wl
    inp.prefix_len[2] = inp.Tcap - 2  # T + n_nodes > Tcap
    ws = ddtree.ddt_workspace_size(wl.B, wl.D, wl.K, wl.budget, wl.H, inp.Tcap)
    assert ws // (wl.B * wl.Qc * wl.H * 513 * 4) > 1, "the key range must be split"
    ot = gu.oracle_tree(inp)
    assert ot.n_nodes[0] < wl.Qc and ot.n_nodes[1] == wl.Qc
    nan_tail(inp, ot)
    tg = gu.target_for(inp, ot)
    step = make_step(inp, tg)
    step.run()
    torch.cuda.synchronize()
    # the tree build passes every sequence; the attention flags the third
    ot["status"] = ot["status"].copy()
    ot["status"][2] = ddtree.DDT_E_BADINPUT
    gu.assert_tree_equal(step.tree, ot)
    ref = oracle.tree_accept(ot, tg, wl.D)
    for k in ("accept_len", "accept_idx", "commit_tok", "next_root"):
        np.testing.assert_array_equal(getattr(step.acc, k).cpu().numpy(), ref[k], err_msg=k)
    out, lse = step.out.cpu().numpy(), step.lse.cpu().numpy()
    ref_out, ref_lse = oracle.attn_all(inp.q_lat[:2], inp.q_rope[:2], inp.c_kv[:2], inp.k_rope[:2],
                                       inp.prefix_len[:2], ot.mask[:2], ot.n_nodes[:2], inp.scale)
    gu.check_rows(out[:2], lse[:2], ref_out, ref_lse, "split keys, sequences 0-1")
    assert np.all(out[2] == 0) and np.all(lse[2] == -np.inf)


@pytest.mark.parametrize("idx", [1, 2])
def test_graph_capture_replays_bit_identically(idx):
    inp = synth.make_inputs(idx)
    ot = gu.oracle_tree(inp)
    tg = gu.target_for(inp, ot)
    step = make_step(inp, tg)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step.run(s)  # first call on the device happens before capture
    torch.cuda.synchronize()
    eager = [t.clone() for t in (step.out, step.lse, step.acc.accept_len, step.acc.commit_tok,
                                 step.tree.token, step.tree.mask)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step.run(s)
    for t in (step.out, step.lse):
        t.zero_()
    for _ in range(20):
        g.replay()
    torch.cuda.synchronize()
    now = (step.out, step.lse, step.acc.accept_len, step.acc.commit_tok, step.tree.token,
           step.tree.mask)
    for a, b in zip(eager, now):
        assert torch.equal(a, b)


def test_bounded_wait_selftest_reports_timeout():
    st = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    ddtree.ddt_selftest_bounded_wait(st, 20000)  # 20 ms limit on a barrier nobody signals
    torch.cuda.synchronize()
    assert int(st.item()) == ddtree.DDT_E_TIMEOUT
    # the context is still usable afterwards
    x = torch.arange(10, device="cuda").sum()
    assert int(x.item()) == 45
