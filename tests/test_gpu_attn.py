"""GPU tree-verify attention vs the float64 oracle.

Small cases are compared on every row; the large workloads, in the launch
configuration the benchmark times, on sampled rows the oracle computes one
by one. Tolerance: max-abs 2e-3 and rel 1e-2 per element (gpu_util)."""
import dataclasses
import math

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


def run_attn(inp, gt=None):
    wl = inp.wl
    if gt is None:
        gt = ddtree.ddt_tree_build(gu.i32_dev(inp.draft_tok), gu.f32_dev(inp.draft_lp),
                                   gu.i32_dev(inp.root_tok), wl.budget, wl.vocab)
    q_lat, q_rope, c_kv, k_rope, pl = gu.attn_dev(inp)
    out, lse = ddtree.ddt_verify_mla_attn(q_lat, q_rope, c_kv, k_rope, pl, gt, inp.scale)
    torch.cuda.synchronize()
    return gt, out.cpu().numpy(), lse.cpu().numpy()


def custom_inputs(seed, B, D, K, budget, H, T, tail="nan", underfull=0, vocab=4000):
    wl = synth.Workload(f"custom{seed}", B, D, K, budget, H, 0, vocab, 0.7, underfull)
    rng = np.random.default_rng(seed)
    tok, lp = random_rows(rng, B, D, K, vocab=vocab)
    for b in range(underfull):
        lp[b] = -np.inf
        lp[b, :, 0] = 0.0
    T = np.asarray(T, np.int32)
    Tcap = int(T.max()) + wl.Qc + 5
    inp = synth.StepInputs(
        wl, tok, lp, rng.integers(0, vocab, B).astype(np.int32), T, Tcap,
        synth.normal_bf16(rng, (B, wl.Qc, H, 512)), synth.normal_bf16(rng, (B, wl.Qc, H, 64)),
        synth.normal_bf16(rng, (B, Tcap, 512)), synth.normal_bf16(rng, (B, Tcap, 64)),
        rng.random((B, wl.Qc)), rng.integers(0, vocab, (B, wl.Qc)).astype(np.int32),
        synth.SOFTMAX_SCALE)
    return inp


def nan_tail(inp, ot):
    """Fill every KV row no node may see (past T_b + n_nodes) and every padded
    query row with NaN: none of it may reach an output."""
    for b in range(inp.wl.B):
        lo = int(inp.prefix_len[b]) + int(ot.n_nodes[b])
        inp.c_kv[b, lo:] = 0x7FC0
        inp.k_rope[b, lo:] = 0x7FC0
        inp.q_lat[b, int(ot.n_nodes[b]):] = 0x7FC0
        inp.q_rope[b, int(ot.n_nodes[b]):] = 0x7FC0


def full_check(inp, what):
    ot = gu.oracle_tree(inp)
    nan_tail(inp, ot)
    gt, out, lse = run_attn(inp)
    gu.assert_tree_equal(gt, ot)
    ref_out, ref_lse = oracle.attn_all(inp.q_lat, inp.q_rope, inp.c_kv, inp.k_rope,
                                       inp.prefix_len, ot.mask, ot.n_nodes, inp.scale)
    err = gu.check_rows(out, lse, ref_out, ref_lse, what)
    return err


@pytest.mark.parametrize("idx", [0, 1])
def test_full_parity_small_workloads(idx):
    err = full_check(synth.make_inputs(idx), synth.WORKLOADS[idx].name)
    print(f"max abs err {err:.3e}")


@pytest.mark.parametrize("seed,B,D,K,budget,H,T,underfull", [
    (1, 3, 5, 4, 20, 8, [0, 37, 300], 0),        # 2 row tiles, ragged prefixes, T=0
    (2, 2, 16, 8, 64, 2, [129, 64], 0),          # W=2 masks, node keys across tiles
    (3, 4, 15, 4, 32, 5, [1, 63, 64, 65], 1),    # odd H, tile-edge prefixes, a chain
    (4, 1, 1, 1, 1, 1, [0], 0),                  # budget 1, H 1, no prefix
    (5, 2, 8, 8, 16, 64, [500, 1337], 0),        # H 64: rows = 2 nodes per tile
    (6, 1, 4, 4, 8, 130, [70], 0),               # H > 128: a node spans tiles
])
def test_full_parity_custom(seed, B, D, K, budget, H, T, underfull):
    inp = custom_inputs(seed, B, D, K, budget, H, T, underfull=underfull)
    full_check(inp, f"custom seed {seed}")


@pytest.mark.parametrize("seed,T,lo,hi", [
    (7, 1500, 5, 8),     # the merge's 8-wide early loads
    (8, 6000, 17, 64),   # 16 early loads, then the rest in batches of 8
])
def test_full_parity_many_key_range_chunks(seed, T, lo, hi):
    """One row tile (9 nodes x 4 heads) over a long prefix: the keys split
    into many ranges, so the merge's wider variants and its batch loop run."""
    inp = custom_inputs(seed, 1, 4, 4, 8, 4, [T])
    wl = inp.wl
    ws = ddtree.ddt_workspace_size(1, wl.D, wl.K, wl.budget, wl.H, inp.Tcap)
    nsplit = ws // (wl.Qc * wl.H * 513 * 4)
    assert lo <= nsplit <= hi, f"{nsplit} key-range chunks"
    full_check(inp, f"{nsplit} key-range chunks")


@pytest.mark.parametrize("seed,B,H,T,lo,hi", [
    (13, 1, 4, [16000], 33, 64),      # one tile, more than 32 chunks (two lse values per merge lane)
    (14, 20, 1, [4000] * 20, 5, 8),   # many sequences, 8 early loads
    (15, 16, 1, [8000] * 16, 9, 16),  # many sequences, 16 early loads
])
def test_full_parity_merge_of_many_chunks(seed, B, H, T, lo, hi):
    """The merge of split key ranges with more than 32 chunks of one
    sequence's keys, and with many sequences at once, against the oracle on
    every row."""
    inp = custom_inputs(seed, B, 4, 4, 8, H, T)
    wl = inp.wl
    ws = ddtree.ddt_workspace_size(B, wl.D, wl.K, wl.budget, wl.H, inp.Tcap)
    nsplit = ws // (B * wl.Qc * wl.H * 513 * 4)
    assert lo <= nsplit <= hi, f"{nsplit} key-range chunks"
    full_check(inp, f"{B} sequences, {nsplit} key-range chunks")


@pytest.mark.parametrize("seed,B,T", [
    (11, 5, [100, 3000, 40, 2000, 700]),      # prefix lengths far apart
    (12, 7, [4000, 4000, 1, 4000, 63, 64, 65]),
])
def test_full_parity_ragged_prefixes_over_row_tiles(seed, B, T):
    """Ragged prefixes over several row tiles per sequence (9 nodes x 20
    heads = 2 row tiles): every sequence's key ranges are cut from its own
    prefix length on the device, so ranges of different lengths, ranges
    past a short sequence's keys and the merge of split ranges all occur."""
    inp = custom_inputs(seed, B, 4, 4, 8, 20, T)
    wl = inp.wl
    ws = ddtree.ddt_workspace_size(B, wl.D, wl.K, wl.budget, wl.H, inp.Tcap)
    assert ws > 0, "the key range must be split"
    full_check(inp, f"ragged prefixes, seed {seed}")


@pytest.mark.parametrize("case", ["custom1", "custom2", "single_stream"])
def test_full_parity_sharp_logits(case):
    """Logits eight times sharper than the N(0,1) inputs give (the softmax
    scale multiplied by 8): the partner's partial scores cross the cluster
    block-scaled to 16 bits, an error in proportion to the scores' magnitude,
    and the output must still meet the tolerance on every row."""
    if case == "single_stream":
        inp = synth.make_inputs(1)
    elif case == "custom1":
        inp = custom_inputs(1, 3, 5, 4, 20, 8, [0, 37, 300])
    else:
        inp = custom_inputs(2, 2, 16, 8, 64, 2, [129, 64])
    inp = dataclasses.replace(inp, scale=inp.scale * 8.0)
    err = full_check(inp, f"{case}, logits x8")
    print(f"max abs err {err:.3e}")


@pytest.mark.parametrize("idx", [2, 3, 4])
def test_sampled_parity_large_workloads(idx):
    inp = synth.make_inputs(idx)
    wl = inp.wl
    ot = gu.oracle_tree(inp)
    gt, out, lse = run_attn(inp)
    gu.assert_tree_equal(gt, ot)
    heads = 3 if idx != 4 else 1
    rows = gu.sample_rows(wl.B, wl.Qc, wl.H, ot.n_nodes, seed=idx, per_seq_heads=heads,
                          max_seqs=8 if idx != 4 else 4)
    ref_out, ref_lse = gu.oracle_rows(inp, ot, rows)
    got_out = out[rows[:, 0], rows[:, 1], rows[:, 2]]
    got_lse = lse[rows[:, 0], rows[:, 1], rows[:, 2]]
    err = gu.check_rows(got_out, got_lse, ref_out, ref_lse, wl.name)
    print(f"{wl.name}: {len(rows)} rows, max abs err {err:.3e}")
    # properties at full size: padded rows are exactly zero; all else finite
    for b in range(wl.B):
        n = int(ot.n_nodes[b])
        assert np.all(out[b, n:] == 0) and np.all(lse[b, n:] == -np.inf)
        assert np.all(np.isfinite(out[b, :n])) and np.all(np.isfinite(lse[b, :n]))


def test_prefix_out_of_range_is_flagged():
    inp = custom_inputs(9, 3, 4, 4, 8, 4, [10, 10, 10])
    inp.prefix_len[1] = inp.Tcap - 2  # T + n_nodes > Tcap
    gt, out, lse = run_attn(inp)
    st = ddtree.ddt_read_device_status(gt.status)
    assert list(st) == [ddtree.DDT_OK, ddtree.DDT_E_BADINPUT, ddtree.DDT_OK]
    assert np.all(out[1] == 0) and np.all(lse[1] == -np.inf)
    assert np.all(np.isfinite(out[0, :9])) and np.all(np.isfinite(out[2, :9]))


def test_root_only_tree_without_prefix_is_its_own_row():
    """T = 0 and a chain budget of 1 with a -inf drafter: node 0 sees only
    its own key, so out is that key's latent exactly."""
    inp = custom_inputs(10, 2, 3, 2, 4, 3, [0, 0])
    inp.draft_lp[:] = -np.inf
    ot = gu.oracle_tree(inp)
    assert (ot.n_nodes == 1).all()
    gt, out, lse = run_attn(inp)
    for b in range(2):
        row = synth.bf16_bits_to_f64(inp.c_kv[b, 0]).astype(np.float32)
        for h in range(3):
            np.testing.assert_array_equal(out[b, 0, h], row)
