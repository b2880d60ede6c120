"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/ddtree.h declares, and rejects bad host-side arguments with
DDT_E_INVAL before touching the device."""
import ctypes
import os
import re

import pytest

from mla_tree_verify_ddt_gb300 import build, ddtree

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    hdr = open(os.path.join(ROOT, "include", "ddtree.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(ddt_[a-z_0-9]+)\s*\(",
                                 hdr, flags=re.M)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return ddtree.lib()


def test_header_declares_the_four_steps():
    names = declared_functions()
    for f in ("ddt_tree_build", "ddt_verify_mla_attn", "ddt_tree_accept", "ddt_verify_step",
              "ddt_workspace_size"):
        assert f in names
    assert set(names) == set(ddtree.EXPORTED)


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_struct_layouts_match_header():
    # pointers are 8 bytes, ints 4: the ctypes mirrors must have the C sizes
    assert ctypes.sizeof(ddtree.DdtDraft) == 4 * 4 + 3 * 8
    assert ctypes.sizeof(ddtree.DdtTree) == 4 * 4 + 10 * 8
    assert ctypes.sizeof(ddtree.DdtAttnIn) == 2 * 4 + 5 * 8
    assert ctypes.sizeof(ddtree.DdtAttnOut) == 2 * 8
    assert ctypes.sizeof(ddtree.DdtAccept) == 4 * 8


def test_status_strings(L):
    for code in range(6):
        assert L.ddt_status_str(code)
    assert b"unknown" in L.ddt_status_str(99)


FAKE = 0x1000  # never dereferenced: every call below fails its host checks first


def _tree(B=2, D=3, Qc=9, W=1):
    return ddtree.DdtTree(B, D, Qc, W, *([FAKE] * 10))


@pytest.mark.parametrize("mutate", [
    lambda d, t: setattr(d, "tok", None),
    lambda d, t: setattr(d, "K", 17),
    lambda d, t: setattr(d, "D", 0),
    lambda d, t: setattr(d, "D", 17),
    lambda d, t: setattr(t, "Qc", 10),
    lambda d, t: setattr(t, "W", 2),
    lambda d, t: setattr(t, "B", 3),
    lambda d, t: setattr(t, "mask", None),
    lambda d, t: setattr(d, "vocab", 0),
])
def test_tree_build_rejects_bad_arguments(L, mutate):
    d = ddtree.DdtDraft(2, 3, 4, 100, FAKE, FAKE, FAKE)
    t = _tree()
    mutate(d, t)
    assert L.ddt_tree_build(ctypes.byref(d), 8, ctypes.byref(t), None) == ddtree.DDT_E_INVAL


@pytest.mark.parametrize("budget", [0, 65, -1])
def test_tree_build_rejects_budget(L, budget):
    d = ddtree.DdtDraft(2, 3, 4, 100, FAKE, FAKE, FAKE)
    t = _tree(Qc=budget + 1, W=max(1, (budget + 64) // 64))
    assert L.ddt_tree_build(ctypes.byref(d), budget, ctypes.byref(t), None) == ddtree.DDT_E_INVAL


def test_attention_rejects_misaligned_and_null(L):
    t = _tree()
    good = dict(H=4, Tcap=100, q_lat=FAKE, q_rope=FAKE, c_kv=FAKE, k_rope=FAKE, prefix_len=FAKE)
    o = ddtree.DdtAttnOut(FAKE, FAKE)
    for field, val in [("q_lat", FAKE + 2), ("c_kv", FAKE + 8), ("k_rope", None), ("H", 0),
                       ("Tcap", 0)]:
        a = ddtree.DdtAttnIn(**{**good, field: val})
        assert L.ddt_verify_mla_attn(ctypes.byref(a), ctypes.byref(t), ctypes.c_float(0.1),
                                     ctypes.byref(o), None, 0, None) == ddtree.DDT_E_INVAL


@pytest.mark.parametrize("scale", [0.0, -0.07, float("nan"), float("inf")])
def test_attention_rejects_scale_that_is_not_positive_and_finite(L, scale):
    t = _tree()
    a = ddtree.DdtAttnIn(4, 100, FAKE, FAKE, FAKE, FAKE, FAKE)
    o = ddtree.DdtAttnOut(FAKE, FAKE)
    sc = ctypes.c_float(scale)
    assert L.ddt_verify_mla_attn(ctypes.byref(a), ctypes.byref(t), sc, ctypes.byref(o), None, 0,
                                 None) == ddtree.DDT_E_INVAL
    assert L.ddt_verify_mla_attn_bf16(ctypes.byref(a), ctypes.byref(t), sc, FAKE, FAKE, None, 0,
                                      None) == ddtree.DDT_E_INVAL
    assert L.ddt_verify_mla_attn_paged(ctypes.byref(a), ctypes.byref(t), sc, ctypes.byref(o), None, 0,
                                       FAKE, 8, None) == ddtree.DDT_E_INVAL


def test_accept_rejects_null(L):
    t = _tree()
    acc = ddtree.DdtAccept(FAKE, None, FAKE, FAKE)
    assert L.ddt_tree_accept(ctypes.byref(t), FAKE, ctypes.byref(acc), None) == ddtree.DDT_E_INVAL
    acc = ddtree.DdtAccept(FAKE, FAKE, FAKE, FAKE)
    assert L.ddt_tree_accept(ctypes.byref(t), None, ctypes.byref(acc), None) == ddtree.DDT_E_INVAL


def test_workspace_size_rejects_bad_shapes(L):
    assert L.ddt_workspace_size(0, 4, 4, 8, 4, 64) == 0
    assert L.ddt_workspace_size(1, 4, 4, 65, 4, 64) == 0


def test_kv_commit_rejects_bad_arguments(L):
    acc = ddtree.DdtAccept(FAKE, FAKE, FAKE, FAKE)
    kv = 0x2000  # 16-byte aligned, never dereferenced
    args = dict(B=2, D=8, Tcap=64, kv=kv, kr=kv, pl=FAKE, st=FAKE)

    def call(acc_=acc, **kw):
        a = dict(args, **kw)
        return L.ddt_kv_commit(ctypes.byref(acc_) if acc_ is not None else None, a["B"], a["D"], a["Tcap"],
                               a["kv"], a["kr"], a["pl"], a["st"], None)
    assert call(acc_=None) == ddtree.DDT_E_INVAL
    assert call(acc_=ddtree.DdtAccept(None, FAKE, FAKE, FAKE)) == ddtree.DDT_E_INVAL
    assert call(B=0) == ddtree.DDT_E_INVAL
    assert call(D=0) == ddtree.DDT_E_INVAL
    assert call(D=17) == ddtree.DDT_E_INVAL
    assert call(Tcap=0) == ddtree.DDT_E_INVAL
    assert call(kv=kv + 2) == ddtree.DDT_E_INVAL
    assert call(kr=None) == ddtree.DDT_E_INVAL
    assert call(pl=None) == ddtree.DDT_E_INVAL


def test_paged_attention_rejects_missing_block_table(L):
    a = ddtree.DdtAttnIn(4, 64, FAKE, FAKE, FAKE, FAKE, FAKE)
    t = _tree()
    o = ddtree.DdtAttnOut(FAKE, FAKE)
    assert L.ddt_verify_mla_attn_paged(ctypes.byref(a), ctypes.byref(t), ctypes.c_float(0.1), ctypes.byref(o),
                                       None, 0, None, 8, None) == ddtree.DDT_E_INVAL
    assert L.ddt_verify_mla_attn_paged(ctypes.byref(a), ctypes.byref(t), ctypes.c_float(0.1), ctypes.byref(o),
                                       None, 0, FAKE, 0, None) == ddtree.DDT_E_INVAL


def test_tree_sample_rejects_bad_arguments(L):
    t = _tree()
    P = ctypes.c_void_p

    def call(tree=t, logits=FAKE, vocab=1000, tau=1.0, u=FAKE, tok=FAKE, p=FAKE):
        return L.ddt_tree_sample(ctypes.byref(tree) if tree is not None else None, P(logits), vocab,
                                 ctypes.c_float(tau), P(u), P(tok), P(p), None)
    assert call(tree=None) == ddtree.DDT_E_INVAL
    assert call(logits=None) == ddtree.DDT_E_INVAL
    assert call(logits=FAKE + 4) == ddtree.DDT_E_INVAL       # not 16-byte aligned
    assert call(vocab=1002) == ddtree.DDT_E_INVAL            # not a multiple of 4
    assert call(vocab=0) == ddtree.DDT_E_INVAL
    assert call(tau=float("nan")) == ddtree.DDT_E_INVAL
    assert call(tau=float("inf")) == ddtree.DDT_E_INVAL
    assert call(tau=1e-35) == ddtree.DDT_E_INVAL
    assert call(u=None) == ddtree.DDT_E_INVAL                # sampling needs the uniforms
    assert call(tok=None) == ddtree.DDT_E_INVAL
    assert call(p=None) == ddtree.DDT_E_INVAL
    bad = _tree(Qc=66, W=2)
    assert call(tree=bad) == ddtree.DDT_E_INVAL
