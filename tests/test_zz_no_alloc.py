"""ddt_verify_mla_attn_noalloc, the attention entry point for callers that
cannot allocate device memory (an engine that has given all spare HBM to its
KV cache, a host that only passes input and output buffers, code that must
not call cudaMalloc because it synchronises the device).

It runs the same kernels as ddt_verify_mla_attn with the key-range partials
in the library's fixed scratch instead of a caller workspace, so its results
must equal that entry point's bit for bit, through the C ABI, on two calls in
a row (the second reuses the scratch as the first left it). Shapes whose
partials exceed the scratch are refused. This file is named to be collected
last, so a failure here comes after every other test has run; it also passes
on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from mla_tree_verify_ddt_gb300 import ddtree, synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

# A batch of short ragged prefixes with few rows per sequence: the planner
# splits every sequence's keys over several ranges, so the scratch partials
# and their merge run with B > 1.
SPLIT_B3 = synth.Workload("split_b3_d4_k4_q9_h16_t700to1500", B=3, D=4, K=4, budget=8, H=16,
                          T=(700, 1500), vocab=1000, p_match=0.7)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ddtree.lib()
    torch.cuda.init()


def _inputs(idx, wl=None):
    inp = synth.make_inputs(idx, wl)
    wl = inp.wl
    tree = ddtree.ddt_tree_build(gu.i32_dev(inp.draft_tok), gu.f32_dev(inp.draft_lp),
                                 gu.i32_dev(inp.root_tok), wl.budget, wl.vocab)
    return inp, tree, gu.attn_dev(inp)


@pytest.mark.parametrize("case", ["tiny", "single_stream", "small_batch", "split_b3"])
def test_noalloc_matches_the_workspace_entry_point_on_two_calls(case):
    idx, wl = {"tiny": (0, None), "single_stream": (1, None), "small_batch": (2, None),
               "split_b3": (0, SPLIT_B3)}[case]
    inp, tree, dev = _inputs(idx, wl)
    wl = inp.wl
    need = ddtree.ddt_workspace_size(wl.B, wl.D, wl.K, wl.budget, wl.H, inp.Tcap)
    assert need <= ddtree.NOALLOC_SCRATCH_BYTES
    if case in ("single_stream", "split_b3"):
        # these shapes split their keys, so the scratch is really used
        assert need > 0, f"{case}: the planner no longer splits this shape"
    ref_out, ref_lse = ddtree.ddt_verify_mla_attn(*dev, tree, inp.scale)
    torch.cuda.synchronize()
    ref_out, ref_lse = ref_out.cpu().numpy(), ref_lse.cpu().numpy()
    out = torch.empty_like(torch.from_numpy(ref_out)).cuda()
    lse = torch.empty_like(torch.from_numpy(ref_lse)).cuda()
    for call in range(2):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        ddtree.ddt_verify_mla_attn_noalloc(*dev, tree, inp.scale, out, lse)
        torch.cuda.synchronize()
        got_out, got_lse = out.cpu().numpy(), lse.cpu().numpy()
        # the same kernels on the same inputs: identical bits
        assert np.array_equal(got_out.view(np.uint32), ref_out.view(np.uint32)), f"{wl.name} call {call}: out"
        assert np.array_equal(got_lse.view(np.uint32), ref_lse.view(np.uint32)), f"{wl.name} call {call}: lse"
        # (and so within the attention tolerance of the workspace entry point)
        gu.check_rows(got_out, got_lse, ref_out.astype(np.float64), ref_lse.astype(np.float64),
                      f"{wl.name} call {call}")


def test_noalloc_refuses_shapes_beyond_its_scratch():
    # the max-budget long-context shape splits each sequence's keys over
    # several ranges on a 152-SM GB300, whose partials need more than the
    # fixed scratch holds
    wl = synth.WORKLOADS[4]
    Tcap = wl.T_max + wl.Qc
    Tcap = (Tcap + 7) // 8 * 8
    need = ddtree.ddt_workspace_size(wl.B, wl.D, wl.K, wl.budget, wl.H, Tcap)
    if need <= ddtree.NOALLOC_SCRATCH_BYTES:
        pytest.skip(f"this device splits the shape into {need} bytes of partials, within the scratch")
    fake = 0x1000  # 16-byte aligned, never dereferenced: the size check comes before any launch
    a = ddtree.DdtAttnIn(wl.H, Tcap, fake, fake, fake, fake, fake)
    t = ddtree.DdtTree(wl.B, wl.D, wl.Qc, wl.W, *([fake] * 10))
    o = ddtree.DdtAttnOut(fake, fake)
    rc = ddtree.lib().ddt_verify_mla_attn_noalloc(ctypes.byref(a), ctypes.byref(t),
                                                  ctypes.c_float(synth.SOFTMAX_SCALE), ctypes.byref(o), None)
    assert rc == ddtree.DDT_E_SCRATCH_LIMIT
    assert "scratch" in ddtree.status_str(rc)
    # an invalid argument is reported as such, even on an oversized shape
    bad = ddtree.DdtAttnIn(wl.H, Tcap, fake, fake, fake, fake, fake)
    rc = ddtree.lib().ddt_verify_mla_attn_noalloc(ctypes.byref(bad), ctypes.byref(t),
                                                  ctypes.c_float(-1.0), ctypes.byref(o), None)
    assert rc == ddtree.DDT_E_INVAL
