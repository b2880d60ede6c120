"""Pins for the oracle's float64 tree-verify attention (CPU only).

Checked against torch's scaled_dot_product_attention in float64 with a
boolean mask (a library routine), and against closed forms: a single visible
key, a zero query, a dominant logit, invisible keys that cannot matter, and
padded rows.
"""
import numpy as np
import pytest
import torch

import oracle
from mla_tree_verify_ddt_gb300 import synth

SCALE = synth.SOFTMAX_SCALE


def random_tree(rng, Qc, n):
    """Random rooted tree on nodes 0..n-1 (parent[i] < i), ancestor masks."""
    W = (Qc + 63) // 64
    parent = np.full(Qc, -1, np.int64)
    mask = np.zeros((Qc, W), np.uint64)
    bits = [0] * Qc
    for i in range(n):
        if i > 0:
            parent[i] = rng.integers(0, i)
            bits[i] = bits[parent[i]]
        bits[i] |= 1 << i
        for w in range(W):
            mask[i, w] = (bits[i] >> (64 * w)) & ((1 << 64) - 1)
    return parent, mask, bits


def make_case(seed, B, Qc, H, T, n_nodes, Tcap=None):
    rng = np.random.default_rng(seed)
    T = np.asarray(T, np.int32)
    Tcap = Tcap or int(T.max()) + Qc + 3
    W = (Qc + 63) // 64
    mask = np.zeros((B, Qc, W), np.uint64)
    bits = []
    for b in range(B):
        _, m, bt = random_tree(rng, Qc, int(n_nodes[b]))
        mask[b] = m
        bits.append(bt)
    q_lat = synth.normal_bf16(rng, (B, Qc, H, 512))
    q_rope = synth.normal_bf16(rng, (B, Qc, H, 64))
    c_kv = synth.normal_bf16(rng, (B, Tcap, 512))
    k_rope = synth.normal_bf16(rng, (B, Tcap, 64))
    return dict(q_lat=q_lat, q_rope=q_rope, c_kv=c_kv, k_rope=k_rope, prefix_len=T,
                mask=mask, n_nodes=np.asarray(n_nodes, np.int32)), bits


def run(case, **kw):
    return oracle.attn_all(case["q_lat"], case["q_rope"], case["c_kv"], case["k_rope"],
                           case["prefix_len"], case["mask"], case["n_nodes"], kw.get("scale", SCALE))


def sdpa_reference(case, bits):
    f = synth.bf16_bits_to_f64
    B, Qc, H, _ = case["q_lat"].shape
    out = np.zeros((B, Qc, H, 512))
    for b in range(B):
        T = int(case["prefix_len"][b])
        n = int(case["n_nodes"][b])
        keys = torch.from_numpy(np.concatenate([f(case["c_kv"][b, :T + n]),
                                                f(case["k_rope"][b, :T + n])], 1))
        vals = torch.from_numpy(f(case["c_kv"][b, :T + n]))
        q = torch.from_numpy(np.concatenate([f(case["q_lat"][b, :n]), f(case["q_rope"][b, :n])],
                                            2)).reshape(n * H, 576)
        allow = torch.zeros(n * H, T + n, dtype=torch.bool)
        allow[:, :T] = True
        for i in range(n):
            for m in range(n):
                if (bits[b][i] >> m) & 1:
                    allow[i * H:(i + 1) * H, T + m] = True
        o = torch.nn.functional.scaled_dot_product_attention(
            q[None], keys[None], vals[None], attn_mask=allow[None], scale=SCALE)[0]
        out[b, :n] = o.reshape(n, H, 512).numpy()
    return out


@pytest.mark.parametrize("seed,B,Qc,H,T,n", [
    (1, 1, 9, 4, [64], [9]),
    (2, 2, 17, 3, [0, 5], [17, 6]),
    (3, 3, 33, 2, [40, 1, 13], [33, 2, 20]),
    (4, 1, 65, 2, [7], [65]),
    (5, 2, 66, 1, [3, 30], [66, 64]),
])
def test_matches_sdpa_float64(seed, B, Qc, H, T, n):
    case, bits = make_case(seed, B, Qc, H, T, n)
    out, lse = run(case)
    ref = sdpa_reference(case, bits)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    for b in range(B):
        assert np.all(np.isfinite(lse[b, :n[b]]))
        assert np.all(lse[b, n[b]:] == -np.inf)
        assert np.all(out[b, n[b]:] == 0)


def test_single_visible_key_is_exact():
    """T=0 and a root-only tree: the root sees only its own key."""
    case, _ = make_case(11, 2, 5, 3, [0, 0], [1, 1])
    out, lse = run(case)
    f = synth.bf16_bits_to_f64
    for b in range(2):
        for h in range(3):
            np.testing.assert_array_equal(out[b, 0, h], f(case["c_kv"][b, 0]))
            s = SCALE * (f(case["q_lat"][b, 0, h]) @ f(case["c_kv"][b, 0]) +
                         f(case["q_rope"][b, 0, h]) @ f(case["k_rope"][b, 0]))
            assert abs(lse[b, 0, h] - s) <= 1e-12 * max(1.0, abs(s))


def test_zero_query_is_the_mean_of_visible_rows():
    case, bits = make_case(12, 1, 9, 2, [20], [9])
    case["q_lat"][:] = 0
    case["q_rope"][:] = 0
    out, lse = run(case)
    f = synth.bf16_bits_to_f64
    for i in range(9):
        vis = list(range(20)) + [20 + m for m in range(9) if (bits[0][i] >> m) & 1]
        mean = f(case["c_kv"][0, vis]).mean(0)
        for h in range(2):
            np.testing.assert_allclose(out[0, i, h], mean, rtol=1e-13, atol=1e-13)
            assert abs(lse[0, i, h] - np.log(len(vis))) < 1e-13


def test_dominant_logit_selects_its_row():
    case, _ = make_case(13, 1, 3, 1, [10], [3])
    # query = 8 x key 4: its logit exceeds every other one by far
    case["q_lat"][0, :, 0] = synth.f32_to_bf16_bits(
        8.0 * synth.bf16_bits_to_f64(case["c_kv"][0, 4]).astype(np.float32))
    case["q_rope"][0, :, 0] = synth.f32_to_bf16_bits(
        8.0 * synth.bf16_bits_to_f64(case["k_rope"][0, 4]).astype(np.float32))
    out, _ = run(case)
    row = synth.bf16_bits_to_f64(case["c_kv"][0, 4])
    for i in range(3):
        np.testing.assert_allclose(out[0, i, 0], row, atol=1e-6)


def test_invisible_keys_do_not_matter():
    case, bits = make_case(14, 1, 17, 2, [12], [11])
    out0, lse0 = run(case)
    T, n = 12, 11
    hidden_everywhere = [T + m for m in range(n, 17)] + list(range(T + 17, case["c_kv"].shape[1]))
    case["c_kv"][0, hidden_everywhere] = 0x7FC0  # NaN
    case["k_rope"][0, hidden_everywhere] = 0x7FC0
    out1, lse1 = run(case)
    np.testing.assert_array_equal(out0, out1)
    np.testing.assert_array_equal(lse0, lse1)
    # a leaf's key is invisible to its siblings' subtrees: perturb it
    leaf = max(range(n), key=lambda i: bin(bits[0][i]).count("1"))
    seers = [i for i in range(n) if (bits[0][i] >> leaf) & 1]
    case["c_kv"][0, T + leaf] ^= 0x0040
    out2, _ = run(case)
    for i in range(n):
        same = np.array_equal(out1[0, i], out2[0, i])
        assert same == (i not in seers)


def test_padded_rows_and_nan_queries():
    case, _ = make_case(15, 1, 9, 2, [4], [3])
    case["q_lat"][0, 3:] = 0x7FC0
    out, lse = run(case)
    assert np.all(out[0, 3:] == 0) and np.all(lse[0, 3:] == -np.inf)
    assert np.all(np.isfinite(out[0, :3]))


def test_tiny_workload_against_sdpa():
    inp = synth.make_inputs(0)
    wl = inp.wl
    t = oracle.tree_build(inp.draft_tok, inp.draft_lp, inp.root_tok, wl.budget, wl.vocab)
    case = dict(q_lat=inp.q_lat, q_rope=inp.q_rope, c_kv=inp.c_kv, k_rope=inp.k_rope,
                prefix_len=inp.prefix_len, mask=t.mask, n_nodes=t.n_nodes)
    bits = [[int(t.mask[b, i, 0]) for i in range(wl.Qc)] for b in range(wl.B)]
    out, _ = run(case)
    np.testing.assert_allclose(out, sdpa_reference(case, bits), rtol=1e-12, atol=1e-12)
