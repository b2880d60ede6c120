"""Helpers for the GPU parity tests: move seeded inputs to the device, run the
oracle on the same inputs, and compare."""
import numpy as np
import torch

import oracle
from mla_tree_verify_ddt_gb300 import synth

# Attention tolerance, elementwise: |gpu - ref| <= ATOL + RTOL * |ref| on the
# [H,512] latent output (max-abs 2e-3, rel 1e-2 against the float64 oracle).
ATOL, RTOL = 2e-3, 1e-2
# lse: the row sum adds bf16-rounded probabilities (relative error <= 2^-9
# each), so |d lse| <= 2^-9 ~ 1.95e-3 in the worst case.
LSE_ATOL = 2e-3

TREE_FIELDS = ("token", "parent", "depth", "rank", "first_child", "next_sibling", "n_nodes",
               "status")


def bf16_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def i32_dev(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def f32_dev(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def attn_dev(inp: synth.StepInputs):
    return (bf16_dev(inp.q_lat), bf16_dev(inp.q_rope), bf16_dev(inp.c_kv), bf16_dev(inp.k_rope),
            i32_dev(inp.prefix_len))


def oracle_tree(inp: synth.StepInputs):
    wl = inp.wl
    return oracle.tree_build(inp.draft_tok, inp.draft_lp, inp.root_tok, wl.budget, wl.vocab)


def assert_tree_equal(gt, ot):
    """Bit-exact comparison of a device tree against the oracle's."""
    for f in TREE_FIELDS:
        np.testing.assert_array_equal(getattr(gt, f).cpu().numpy(), ot[f], err_msg=f)
    np.testing.assert_array_equal(gt.score.cpu().numpy().view(np.uint32),
                                  ot.score.view(np.uint32), err_msg="score bits")
    np.testing.assert_array_equal(gt.mask.cpu().numpy().view(np.uint64), ot.mask, err_msg="mask")


def target_for(inp, ot):
    return synth.synth_target_argmax(ot.depth, ot.n_nodes, inp.draft_tok, inp.target_u,
                                     inp.target_alt, inp.wl.p_match)


def check_rows(out, lse, ref_out, ref_lse, what=""):
    """out/lse: numpy float32 rows; ref: float64 rows from the oracle."""
    out = np.asarray(out, np.float64)
    lse = np.asarray(lse, np.float64)
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    err = np.abs(out - ref_out)
    bad = err > ATOL + RTOL * np.abs(ref_out)
    assert not bad.any(), (f"{what}: {bad.sum()} elements out of tolerance, max abs err "
                           f"{err.max():.3e}")
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: lse finiteness differs"
    if fin.any():
        lerr = np.abs(lse[fin] - ref_lse[fin])
        assert lerr.max() <= LSE_ATOL, f"{what}: lse max err {lerr.max():.3e}"
    return float(err.max())


def sample_rows(B, Qc, H, n_nodes, seed, per_seq_heads=3, max_seqs=8):
    """(b, i, h) triples: every node slot (valid and padded) of a few heads —
    always head 0 and head H-1 — for up to max_seqs sequences, plus one row in
    every 128-row tile boundary neighbourhood."""
    rng = np.random.default_rng(seed)
    seqs = sorted(set([0, B - 1] + list(rng.choice(B, min(B, max_seqs), replace=False))))[:max_seqs]
    rows = []
    for b in seqs:
        heads = sorted(set([0, H - 1] + list(rng.integers(0, H, per_seq_heads))))
        for h in heads:
            for i in range(Qc):
                rows.append((b, i, h))
        for g in range(127, Qc * H, 128):
            for gg in (g, g + 1):
                if gg < Qc * H:
                    rows.append((b, gg // H, gg % H))
    return np.array(sorted(set(rows)), np.int32)


def oracle_rows(inp, ot, rows):
    out, lse, _ = oracle.attn_rows(inp.q_lat, inp.q_rope, inp.c_kv, inp.k_rope, inp.prefix_len,
                                   ot.mask, ot.n_nodes, inp.scale, rows)
    return out, lse
