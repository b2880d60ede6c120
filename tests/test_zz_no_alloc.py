"""ddt_verify_mla_attn_noalloc, the attention entry point for callers that
cannot allocate device memory (an engine that has given all spare HBM to its
KV cache, a host that only passes input and output buffers, code that must
not call cudaMalloc because it synchronises the device).

It must produce what ddt_verify_mla_attn produces, through the C ABI, on two
calls in a row (the second reuses the library's scratch as the first left
it), and refuse shapes whose key-range partials exceed its fixed scratch.
This file is named to be collected last, so a failure here comes after every
other test has run; it also passes on its own in a fresh process."""
import ctypes

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


def _inputs(idx):
    inp = synth.make_inputs(idx)
    wl = inp.wl
    tree = ddtree.ddt_tree_build(gu.i32_dev(inp.draft_tok), gu.f32_dev(inp.draft_lp),
                                 gu.i32_dev(inp.root_tok), wl.budget, wl.vocab)
    return inp, tree, gu.attn_dev(inp)


@pytest.mark.parametrize("idx", [0, 1, 2])
def test_noalloc_matches_the_workspace_entry_point_on_two_calls(idx):
    inp, tree, dev = _inputs(idx)
    wl = inp.wl
    need = ddtree.ddt_workspace_size(wl.B, wl.D, wl.K, wl.budget, wl.H, inp.Tcap)
    assert need <= ddtree.NOALLOC_SCRATCH_BYTES
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
        gu.check_rows(got_out, got_lse, ref_out.astype(np.float64), ref_lse.astype(np.float64),
                      f"{wl.name} call {call}")


def test_noalloc_refuses_shapes_beyond_its_scratch():
    # the max-budget long-context shape splits its keys over two ranges on a
    # 152-SM GB300, which needs more partial storage than the fixed scratch
    wl = synth.WORKLOADS[4]
    Tcap = wl.T_max + wl.Qc
    need = ddtree.ddt_workspace_size(wl.B, wl.D, wl.K, wl.budget, wl.H, Tcap)
    if need <= ddtree.NOALLOC_SCRATCH_BYTES:
        pytest.skip(f"this device splits the shape into {need} bytes of partials, within the scratch")
    fake = 0x1000  # never dereferenced: the size check comes first
    a = ddtree.DdtAttnIn(wl.H, Tcap, fake, fake, fake, fake, fake)
    t = ddtree.DdtTree(wl.B, wl.D, wl.Qc, wl.W, *([fake] * 10))
    o = ddtree.DdtAttnOut(fake, fake)
    rc = ddtree.lib().ddt_verify_mla_attn_noalloc(ctypes.byref(a), ctypes.byref(t),
                                                  ctypes.c_float(synth.SOFTMAX_SCALE), ctypes.byref(o), None)
    assert rc == ddtree.DDT_E_SCRATCH_LIMIT
    assert "scratch" in ddtree.status_str(rc)
