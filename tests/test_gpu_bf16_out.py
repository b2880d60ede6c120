"""ddt_verify_mla_attn_bf16: the latent output in bfloat16. Each element must
be the float32 entry point's value rounded to nearest even, bit for bit, and
within the attention tolerance of the oracle."""
import numpy as np
import pytest
import torch

from mla_tree_verify_ddt_gb300 import ddtree, synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ddtree.lib()
    torch.cuda.init()


def rne_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (finite values)."""
    u = x32.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


@pytest.mark.parametrize("idx", [0, 1, 2, 3])
def test_bf16_output_is_the_rounded_float32_output(idx):
    inp = synth.make_inputs(idx)
    wl = inp.wl
    tree = ddtree.ddt_tree_build(gu.i32_dev(inp.draft_tok), gu.f32_dev(inp.draft_lp), gu.i32_dev(inp.root_tok),
                                 wl.budget, wl.vocab)
    dev = gu.attn_dev(inp)
    ref, ref_lse = ddtree.ddt_verify_mla_attn(*dev, tree, inp.scale)
    out, lse = ddtree.ddt_verify_mla_attn_bf16(*dev, tree, inp.scale)
    torch.cuda.synchronize()
    ref = ref.cpu().numpy()
    got = out.cpu().view(torch.int16).numpy().view(np.uint16)
    want = rne_bf16_bits(ref)
    # (with a split key range the merge computes the same float32 sum either
    # way and rounds it, so the match is exact there too)
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(lse.cpu().numpy(), ref_lse.cpu().numpy())


def test_bf16_output_against_the_oracle():
    inp = synth.make_inputs(0)
    wl = inp.wl
    tree = ddtree.ddt_tree_build(gu.i32_dev(inp.draft_tok), gu.f32_dev(inp.draft_lp), gu.i32_dev(inp.root_tok),
                                 wl.budget, wl.vocab)
    dev = gu.attn_dev(inp)
    out, lse = ddtree.ddt_verify_mla_attn_bf16(*dev, tree, inp.scale)
    torch.cuda.synchronize()
    ot = gu.oracle_tree(inp)
    import oracle
    ref_out, ref_lse = oracle.attn_all(inp.q_lat, inp.q_rope, inp.c_kv, inp.k_rope, inp.prefix_len, ot.mask,
                                       ot.n_nodes, inp.scale)
    gu.check_rows(out.float().cpu().numpy().reshape(-1, 512), lse.cpu().numpy().ravel(),
                  ref_out.reshape(-1, 512), ref_lse.ravel(), "bf16 output")


@pytest.mark.parametrize("idx", [2, 3])
def test_bf16_output_against_the_oracle_on_sampled_rows(idx):
    """Small batch (ragged prefixes) and wide batch (underfull trees), sampled
    rows against the oracle."""
    import oracle
    inp = synth.make_inputs(idx)
    wl = inp.wl
    tree = ddtree.ddt_tree_build(gu.i32_dev(inp.draft_tok), gu.f32_dev(inp.draft_lp), gu.i32_dev(inp.root_tok),
                                 wl.budget, wl.vocab)
    dev = gu.attn_dev(inp)
    out, lse = ddtree.ddt_verify_mla_attn_bf16(*dev, tree, inp.scale)
    torch.cuda.synchronize()
    ot = gu.oracle_tree(inp)
    rows = gu.sample_rows(wl.B, wl.Qc, wl.H, ot.n_nodes, seed=60 + idx)
    ref_out, ref_lse = gu.oracle_rows(inp, ot, rows)
    o, l = out.float().cpu().numpy(), lse.cpu().numpy()
    b, i, h = rows[:, 0], rows[:, 1], rows[:, 2]
    gu.check_rows(o[b, i, h], l[b, i, h], ref_out, ref_lse, f"bf16 output {wl.name}")
