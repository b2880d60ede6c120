"""The whole verify step on seeded random shapes against the oracle: tree and
accept bit for bit, attention on every row within the tolerance; and on the
same shapes the paged-cache and bfloat16-output attention against the
contiguous float32 call, bit for bit. The shapes draw batch, depth, top-K,
budget (node masks of one or two words), heads (row tiles that end
mid-tile, nodes spanning tiles) and ragged prefix lengths (prefixes ending
anywhere in a key tile, split key ranges, ranges past a short sequence's
keys), some sequences with an underfull tree."""
import numpy as np
import pytest
import torch

from mla_tree_verify_ddt_gb300 import ddtree
from tests import gpu_util as gu
from tests.test_gpu_attn import custom_inputs, nan_tail
from tests.test_gpu_bf16_out import rne_bf16_bits
from tests.test_gpu_paged import paged_inputs
from tests.test_gpu_step import check_step, make_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ddtree.lib()
    torch.cuda.init()


def random_case(seed):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 7))
    D = int(rng.integers(1, 17))
    K = int(rng.integers(1, 9))
    budget = int(rng.integers(1, 65))
    H = int(rng.choice([1, 2, 3, 5, 8, 16, 20, 33, 64]))
    # keep the oracle's work (rows x keys) to a few million per case
    rows = B * (budget + 1) * H
    t_hi = max(2, min(6000, int(4e6 / rows)))
    T = [int(rng.integers(0, t_hi)) for _ in range(B)]
    underfull = int(rng.integers(0, B)) if B > 1 and rng.random() < 0.3 else 0
    return B, D, K, budget, H, T, underfull


@pytest.mark.parametrize("seed", range(40))
def test_random_shape_step_against_the_oracle(seed):
    B, D, K, budget, H, T, underfull = random_case(seed)
    inp = custom_inputs(seed, B, D, K, budget, H, T, underfull=underfull)
    ot = gu.oracle_tree(inp)
    nan_tail(inp, ot)
    tg = gu.target_for(inp, ot)
    step = make_step(inp, tg)
    step.run()
    torch.cuda.synchronize()
    check_step(step, inp, ot, tg)
    st = ddtree.ddt_read_device_status(step.tree.status)
    assert (st == ddtree.DDT_OK).all(), f"B={B} D={D} K={K} budget={budget} H={H} T={T}: status {st}"


@pytest.mark.parametrize("seed", range(40, 56))
def test_random_shape_paged_and_bf16_match_the_contiguous_call(seed):
    B, D, K, budget, H, T, underfull = random_case(seed)
    inp = custom_inputs(seed, B, D, K, budget, H, T, underfull=underfull)
    wl = inp.wl
    tree = ddtree.ddt_tree_build(gu.i32_dev(inp.draft_tok), gu.f32_dev(inp.draft_lp), gu.i32_dev(inp.root_tok),
                                 wl.budget, wl.vocab)
    dev = gu.attn_dev(inp)
    ref, ref_lse = ddtree.ddt_verify_mla_attn(*dev, tree, inp.scale)
    out16, lse16 = ddtree.ddt_verify_mla_attn_bf16(*dev, tree, inp.scale)
    pool_kv, pool_kr, kvi = paged_inputs(inp, tree.n_nodes.cpu().numpy(), seed)
    outp, lsep = ddtree.ddt_verify_mla_attn_paged(dev[0], dev[1], gu.bf16_dev(pool_kv), gu.bf16_dev(pool_kr), dev[4],
                                                  gu.i32_dev(kvi), tree, inp.scale)
    torch.cuda.synchronize()
    assert (ddtree.ddt_read_device_status(tree.status) == ddtree.DDT_OK).all()
    ref_np = ref.cpu().numpy()
    np.testing.assert_array_equal(outp.cpu().numpy().view(np.uint32), ref_np.view(np.uint32))
    np.testing.assert_array_equal(lsep.cpu().numpy().view(np.uint32), ref_lse.cpu().numpy().view(np.uint32))
    np.testing.assert_array_equal(out16.cpu().view(torch.int16).numpy().view(np.uint16), rne_bf16_bits(ref_np))
    np.testing.assert_array_equal(lse16.cpu().numpy(), ref_lse.cpu().numpy())
