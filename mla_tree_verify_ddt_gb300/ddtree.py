"""ctypes binding for libddtree (include/ddtree.h).

Argument marshalling only: every step of the verify path runs in the CUDA
kernels of libddtree.so. PyTorch provides device memory and streams. If the
library is missing this module raises at import-time use; there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libddtree.so")

DDT_OK, DDT_E_INVAL, DDT_E_CUDA, DDT_E_UNSUPPORTED, DDT_E_BADINPUT, DDT_E_TIMEOUT = range(6)
DDT_E_SCRATCH_LIMIT = 6
NOALLOC_SCRATCH_BYTES = 64 << 20
MAX_DEPTH, MAX_TOPK, MAX_BUDGET, LATENT, ROPE = 16, 16, 64, 512, 64

EXPORTED = ["ddt_workspace_size", "ddt_tree_build", "ddt_verify_mla_attn", "ddt_tree_accept",
            "ddt_verify_step", "ddt_status_str", "ddt_read_device_status",
            "ddt_selftest_bounded_wait", "ddt_verify_mla_attn_noalloc", "ddt_kv_commit",
            "ddt_verify_mla_attn_paged", "ddt_verify_mla_attn_bf16", "ddt_tree_sample"]

P = ctypes.c_void_p
I = ctypes.c_int


class DdtDraft(ctypes.Structure):
    _fields_ = [("B", I), ("D", I), ("K", I), ("vocab", I), ("tok", P), ("lp", P), ("root_tok", P)]


class DdtTree(ctypes.Structure):
    _fields_ = [("B", I), ("D", I), ("Qc", I), ("W", I), ("token", P), ("parent", P), ("depth", P),
                ("rank", P), ("score", P), ("first_child", P), ("next_sibling", P), ("mask", P),
                ("n_nodes", P), ("status", P)]


class DdtAttnIn(ctypes.Structure):
    _fields_ = [("H", I), ("Tcap", I), ("q_lat", P), ("q_rope", P), ("c_kv", P), ("k_rope", P),
                ("prefix_len", P)]


class DdtAttnOut(ctypes.Structure):
    _fields_ = [("out", P), ("lse", P)]


class DdtAccept(ctypes.Structure):
    _fields_ = [("accept_len", P), ("accept_idx", P), ("commit_tok", P), ("next_root", P)]


class DdtError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_str(code)} ({code})")
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """Load libddtree.so (built by mla_tree_verify_ddt_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libddtree.so is not built ({LIB_PATH}); run "
                               "python -m mla_tree_verify_ddt_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        L.ddt_workspace_size.argtypes = [I, I, I, I, I, I]
        L.ddt_workspace_size.restype = ctypes.c_size_t
        L.ddt_tree_build.argtypes = [ctypes.POINTER(DdtDraft), I, ctypes.POINTER(DdtTree), P]
        L.ddt_verify_mla_attn.argtypes = [ctypes.POINTER(DdtAttnIn), ctypes.POINTER(DdtTree),
                                          ctypes.c_float, ctypes.POINTER(DdtAttnOut), P,
                                          ctypes.c_size_t, P]
        L.ddt_tree_accept.argtypes = [ctypes.POINTER(DdtTree), P, ctypes.POINTER(DdtAccept), P]
        L.ddt_verify_step.argtypes = [ctypes.POINTER(DdtDraft), I, ctypes.POINTER(DdtTree),
                                      ctypes.POINTER(DdtAttnIn), ctypes.c_float,
                                      ctypes.POINTER(DdtAttnOut), P, ctypes.POINTER(DdtAccept), P,
                                      ctypes.c_size_t, P]
        L.ddt_verify_mla_attn_noalloc.argtypes = [ctypes.POINTER(DdtAttnIn), ctypes.POINTER(DdtTree),
                                                  ctypes.c_float, ctypes.POINTER(DdtAttnOut), P]
        L.ddt_kv_commit.argtypes = [ctypes.POINTER(DdtAccept), I, I, I, P, P, P, P, P]
        L.ddt_verify_mla_attn_bf16.argtypes = [ctypes.POINTER(DdtAttnIn), ctypes.POINTER(DdtTree), ctypes.c_float,
                                               P, P, P, ctypes.c_size_t, P]
        L.ddt_verify_mla_attn_paged.argtypes = [ctypes.POINTER(DdtAttnIn), ctypes.POINTER(DdtTree), ctypes.c_float,
                                                ctypes.POINTER(DdtAttnOut), P, ctypes.c_size_t, P, I, P]
        L.ddt_tree_sample.argtypes = [ctypes.POINTER(DdtTree), P, I, ctypes.c_float, P, P, P, P]
        L.ddt_status_str.argtypes = [I]
        L.ddt_status_str.restype = ctypes.c_char_p
        L.ddt_read_device_status.argtypes = [P, I, P]
        L.ddt_selftest_bounded_wait.argtypes = [P, ctypes.c_uint, P]
        for f in ("ddt_tree_build", "ddt_verify_mla_attn", "ddt_tree_accept", "ddt_verify_step",
                  "ddt_read_device_status", "ddt_selftest_bounded_wait",
                  "ddt_verify_mla_attn_noalloc", "ddt_kv_commit", "ddt_verify_mla_attn_paged",
                  "ddt_verify_mla_attn_bf16", "ddt_tree_sample"):
            getattr(L, f).restype = I
        _lib = L
    return _lib


def status_str(code: int) -> str:
    return lib().ddt_status_str(int(code)).decode()


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream_ptr(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(rc: int, what: str):
    if rc != DDT_OK:
        raise DdtError(rc, what)


# ------------------------------------------------------------------ buffers

@dataclass
class Tree:
    """Device tensors of one built tree batch (shapes as in ddtree.h)."""
    B: int
    D: int
    Qc: int
    W: int
    token: torch.Tensor
    parent: torch.Tensor
    depth: torch.Tensor
    rank: torch.Tensor
    score: torch.Tensor
    first_child: torch.Tensor
    next_sibling: torch.Tensor
    mask: torch.Tensor          # int64 view of the uint64 words
    n_nodes: torch.Tensor
    status: torch.Tensor

    @staticmethod
    def empty(B: int, D: int, budget: int, device="cuda") -> "Tree":
        Qc = budget + 1
        W = (Qc + 63) // 64
        i32 = dict(dtype=torch.int32, device=device)
        return Tree(B, D, Qc, W, *[torch.empty(B, Qc, **i32) for _ in range(4)],
                    torch.empty(B, Qc, dtype=torch.float32, device=device),
                    torch.empty(B, Qc, **i32), torch.empty(B, Qc, **i32),
                    torch.empty(B, Qc, W, dtype=torch.int64, device=device),
                    torch.empty(B, **i32), torch.empty(B, **i32))

    def c(self) -> DdtTree:
        return DdtTree(self.B, self.D, self.Qc, self.W, *[_ptr(getattr(self, f)) for f in
                       ("token", "parent", "depth", "rank", "score", "first_child",
                        "next_sibling", "mask", "n_nodes", "status")])


@dataclass
class Accept:
    accept_len: torch.Tensor
    accept_idx: torch.Tensor
    commit_tok: torch.Tensor
    next_root: torch.Tensor

    @staticmethod
    def empty(B: int, D: int, device="cuda") -> "Accept":
        i32 = dict(dtype=torch.int32, device=device)
        return Accept(torch.empty(B, **i32), torch.empty(B, D + 1, **i32),
                      torch.empty(B, D + 1, **i32), torch.empty(B, **i32))

    def c(self) -> DdtAccept:
        return DdtAccept(_ptr(self.accept_len), _ptr(self.accept_idx), _ptr(self.commit_tok),
                         _ptr(self.next_root))


def draft_struct(tok, lp, root_tok, vocab: int) -> DdtDraft:
    B, D, K = tok.shape
    return DdtDraft(B, D, K, vocab, _ptr(tok), _ptr(lp), _ptr(root_tok))


def attn_in_struct(q_lat, q_rope, c_kv, k_rope, prefix_len) -> DdtAttnIn:
    return DdtAttnIn(q_lat.shape[2], c_kv.shape[1], _ptr(q_lat), _ptr(q_rope), _ptr(c_kv),
                     _ptr(k_rope), _ptr(prefix_len))


_I32, _F32, _BF16 = (torch.int32,), (torch.float32,), (torch.bfloat16,)
_HALFWORD = (torch.bfloat16, torch.float16, torch.int16)  # moved as raw 2-byte elements


def _need(t, name: str, dtypes, shape):
    """Checks the C ABI cannot make on a raw pointer: element type, shape
    (None matches any extent) and dense row-major layout. Device memory is
    checked by _on_device once every argument has passed these."""
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {' or '.join(str(d) for d in dtypes)}")
    if t.dim() != len(shape) or any(e is not None and e != g for e, g in zip(shape, t.shape)):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected "
                         f"[{', '.join('*' if e is None else str(e) for e in shape)}]")
    if not t.is_contiguous():
        raise ValueError(f"{name}: libddtree takes dense row-major tensors")


def _on_device(*ts, stream=None):
    """Every tensor in device memory of the current CUDA device, and the
    stream (if given) on that device too. The C ABI plans the launch for,
    encodes its tensor maps on, and launches on the current device, so a
    tensor of another GPU would reach its kernels as a foreign pointer."""
    cur = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("libddtree takes CUDA tensors (device memory)")
        if cur is None:
            cur = torch.cuda.current_device()
        if t.device.index != cur:
            raise ValueError(f"tensor on {t.device}, but the current CUDA device is cuda:{cur}: "
                             "libddtree launches on the current device (torch.cuda.set_device)")
    if stream is not None:
        if cur is None:
            cur = torch.cuda.current_device()
        if stream.device.index != cur:
            raise ValueError(f"stream of {stream.device}, but the current CUDA device is cuda:{cur}")


def _tree_attn(tree: "Tree"):
    """The tree tensors the attention reads."""
    return tree.mask, tree.n_nodes, tree.status


def _need_attn(q_lat, q_rope, c_kv, k_rope, prefix_len, tree: "Tree"):
    _need(q_lat, "q_lat", _BF16, (tree.B, tree.Qc, None, LATENT))
    H = q_lat.shape[2]
    _need(q_rope, "q_rope", _BF16, (tree.B, tree.Qc, H, ROPE))
    _need(c_kv, "c_kv", _BF16, (tree.B, None, LATENT))
    _need(k_rope, "k_rope", _BF16, (tree.B, c_kv.shape[1], ROPE))
    _need(prefix_len, "prefix_len", _I32, (tree.B,))
    return H


def _need_accept(acc: "Accept", B: int, D: int):
    _need(acc.accept_len, "accept_len", _I32, (B,))
    _need(acc.accept_idx, "accept_idx", _I32, (B, D + 1))
    _need(acc.commit_tok, "commit_tok", _I32, (B, D + 1))
    _need(acc.next_root, "next_root", _I32, (B,))


def _need_out(out, lse, tree: "Tree", H: int, out_dtypes):
    if out is not None:
        _need(out, "out", out_dtypes, (tree.B, tree.Qc, H, LATENT))
    if lse is not None:
        _need(lse, "lse", _F32, (tree.B, tree.Qc, H))


# ------------------------------------------------------------------ calls

def ddt_workspace_size(B: int, D: int, K: int, budget: int, H: int, Tcap: int) -> int:
    return int(lib().ddt_workspace_size(B, D, K, budget, H, Tcap))


def ddt_tree_build(tok, lp, root_tok, budget: int, vocab: int, out: Tree | None = None,
                   stream=None) -> Tree:
    _need(tok, "tok", _I32, (None, None, None))
    B, D, K = tok.shape
    _need(lp, "lp", _F32, (B, D, K))
    _need(root_tok, "root_tok", _I32, (B,))
    _on_device(tok, lp, root_tok, stream=stream)
    out = out or Tree.empty(B, D, budget, tok.device)
    d, t = draft_struct(tok, lp, root_tok, vocab), out.c()
    _check(lib().ddt_tree_build(ctypes.byref(d), budget, ctypes.byref(t), _stream_ptr(stream)),
           "ddt_tree_build")
    return out


def ddt_verify_mla_attn(q_lat, q_rope, c_kv, k_rope, prefix_len, tree: Tree, scale: float,
                        out=None, lse=None, workspace=None, stream=None):
    _need_out(out, lse, tree, _need_attn(q_lat, q_rope, c_kv, k_rope, prefix_len, tree), _F32)
    _on_device(q_lat, q_rope, c_kv, k_rope, prefix_len, out, lse, workspace, *_tree_attn(tree), stream=stream)
    B, Qc, H, _ = q_lat.shape
    if out is None:
        out = torch.empty(B, Qc, H, LATENT, dtype=torch.float32, device=q_lat.device)
    if lse is None:
        lse = torch.empty(B, Qc, H, dtype=torch.float32, device=q_lat.device)
    ws = ddt_workspace_size(B, tree.D, 1, Qc - 1, H, c_kv.shape[1])
    if workspace is None and ws:
        workspace = torch.empty(ws, dtype=torch.uint8, device=q_lat.device)
    a = attn_in_struct(q_lat, q_rope, c_kv, k_rope, prefix_len)
    o = DdtAttnOut(_ptr(out), _ptr(lse))
    t = tree.c()
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().ddt_verify_mla_attn(ctypes.byref(a), ctypes.byref(t), float(scale),
                                     ctypes.byref(o), _ptr(workspace), wsb, _stream_ptr(stream)),
           "ddt_verify_mla_attn")
    return out, lse


def ddt_verify_mla_attn_bf16(q_lat, q_rope, c_kv, k_rope, prefix_len, tree: Tree, scale: float,
                             out=None, lse=None, workspace=None, stream=None):
    """ddt_verify_mla_attn with the latent output in bfloat16."""
    _need_out(out, lse, tree, _need_attn(q_lat, q_rope, c_kv, k_rope, prefix_len, tree), _BF16)
    _on_device(q_lat, q_rope, c_kv, k_rope, prefix_len, out, lse, workspace, *_tree_attn(tree), stream=stream)
    B, Qc, H, _ = q_lat.shape
    if out is None:
        out = torch.empty(B, Qc, H, LATENT, dtype=torch.bfloat16, device=q_lat.device)
    if lse is None:
        lse = torch.empty(B, Qc, H, dtype=torch.float32, device=q_lat.device)
    ws = ddt_workspace_size(B, tree.D, 1, Qc - 1, H, c_kv.shape[1])
    if workspace is None and ws:
        workspace = torch.empty(ws, dtype=torch.uint8, device=q_lat.device)
    a = attn_in_struct(q_lat, q_rope, c_kv, k_rope, prefix_len)
    t = tree.c()
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().ddt_verify_mla_attn_bf16(ctypes.byref(a), ctypes.byref(t), float(scale), _ptr(out), _ptr(lse),
                                          _ptr(workspace), wsb, _stream_ptr(stream)), "ddt_verify_mla_attn_bf16")
    return out, lse


def ddt_verify_mla_attn_paged(q_lat, q_rope, pool_kv, pool_kr, prefix_len, kv_index, tree: Tree, scale: float,
                              out=None, lse=None, workspace=None, stream=None):
    """Attention on a block-table cache: key position p of sequence b is row
    kv_index[b, p] of pool_kv [P,512] / pool_kr [P,64] (bf16); kv_index is
    int32 [B, Tcap]."""
    _need(q_lat, "q_lat", _BF16, (tree.B, tree.Qc, None, LATENT))
    _need(q_rope, "q_rope", _BF16, (tree.B, tree.Qc, q_lat.shape[2], ROPE))
    _need(pool_kv, "pool_kv", _BF16, (None, LATENT))
    _need(pool_kr, "pool_kr", _BF16, (pool_kv.shape[0], ROPE))
    _need(prefix_len, "prefix_len", _I32, (tree.B,))
    _need(kv_index, "kv_index", _I32, (tree.B, None))
    _need_out(out, lse, tree, q_lat.shape[2], _F32)
    _on_device(q_lat, q_rope, pool_kv, pool_kr, prefix_len, kv_index, out, lse, workspace, *_tree_attn(tree),
               stream=stream)
    B, Qc, H, _ = q_lat.shape
    Tcap = kv_index.shape[1]
    if out is None:
        out = torch.empty(B, Qc, H, LATENT, dtype=torch.float32, device=q_lat.device)
    if lse is None:
        lse = torch.empty(B, Qc, H, dtype=torch.float32, device=q_lat.device)
    ws = ddt_workspace_size(B, tree.D, 1, Qc - 1, H, Tcap)
    if workspace is None and ws:
        workspace = torch.empty(ws, dtype=torch.uint8, device=q_lat.device)
    a = DdtAttnIn(H, Tcap, _ptr(q_lat), _ptr(q_rope), _ptr(pool_kv), _ptr(pool_kr), _ptr(prefix_len))
    o = DdtAttnOut(_ptr(out), _ptr(lse))
    t = tree.c()
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().ddt_verify_mla_attn_paged(ctypes.byref(a), ctypes.byref(t), float(scale), ctypes.byref(o),
                                           _ptr(workspace), wsb, _ptr(kv_index), pool_kv.shape[0],
                                           _stream_ptr(stream)), "ddt_verify_mla_attn_paged")
    return out, lse


def ddt_verify_mla_attn_noalloc(q_lat, q_rope, c_kv, k_rope, prefix_len, tree: Tree, scale: float,
                                out=None, lse=None, stream=None):
    """Same as ddt_verify_mla_attn, for callers that cannot allocate: the
    key-range partials go to the library's own fixed device scratch
    (NOALLOC_SCRATCH_BYTES per GPU). Output tensors, if not given, are
    created here by torch; pass them in to allocate nothing at all."""
    _need_out(out, lse, tree, _need_attn(q_lat, q_rope, c_kv, k_rope, prefix_len, tree), _F32)
    _on_device(q_lat, q_rope, c_kv, k_rope, prefix_len, out, lse, *_tree_attn(tree), stream=stream)
    B, Qc, H, _ = q_lat.shape
    if out is None:
        out = torch.empty(B, Qc, H, LATENT, dtype=torch.float32, device=q_lat.device)
    if lse is None:
        lse = torch.empty(B, Qc, H, dtype=torch.float32, device=q_lat.device)
    a = attn_in_struct(q_lat, q_rope, c_kv, k_rope, prefix_len)
    o = DdtAttnOut(_ptr(out), _ptr(lse))
    t = tree.c()
    _check(lib().ddt_verify_mla_attn_noalloc(ctypes.byref(a), ctypes.byref(t), float(scale),
                                             ctypes.byref(o), _stream_ptr(stream)),
           "ddt_verify_mla_attn_noalloc")
    return out, lse


def ddt_tree_accept(tree: Tree, target_argmax, out: Accept | None = None, stream=None) -> Accept:
    _need(target_argmax, "target_argmax", _I32, (tree.B, tree.Qc))
    if out is not None:
        _need_accept(out, tree.B, tree.D)
        _on_device(out.accept_len, out.accept_idx, out.commit_tok, out.next_root)
    _on_device(target_argmax, tree.token, tree.parent, tree.n_nodes, stream=stream)
    out = out or Accept.empty(tree.B, tree.D, target_argmax.device)
    t, a = tree.c(), out.c()
    _check(lib().ddt_tree_accept(ctypes.byref(t), _ptr(target_argmax), ctypes.byref(a),
                                 _stream_ptr(stream)), "ddt_tree_accept")
    return out


def ddt_kv_commit(acc: Accept, c_kv, k_rope, prefix_len, status, stream=None):
    """Moves the accepted path's keys into the committed prefix, in place on
    c_kv [B,Tcap,512] and k_rope [B,Tcap,64] (bf16), and advances prefix_len
    (int32 [B]); status (int32 [B]) gets DDT_E_BADINPUT for a sequence whose
    values do not fit."""
    _need(c_kv, "c_kv", _HALFWORD, (acc.accept_len.shape[0], None, LATENT))
    B, Tcap, _ = c_kv.shape
    _need_accept(acc, B, acc.accept_idx.shape[1] - 1)
    _need(k_rope, "k_rope", _HALFWORD, (B, Tcap, ROPE))
    _need(prefix_len, "prefix_len", _I32, (B,))
    _need(status, "status", _I32, (B,))
    _on_device(c_kv, k_rope, prefix_len, status, acc.accept_len, acc.accept_idx, stream=stream)
    D = acc.accept_idx.shape[1] - 1
    a = acc.c()
    _check(lib().ddt_kv_commit(ctypes.byref(a), B, D, Tcap, _ptr(c_kv), _ptr(k_rope), _ptr(prefix_len),
                               _ptr(status), _stream_ptr(stream)), "ddt_kv_commit")


def ddt_tree_sample(tree: Tree, logits, temperature: float, u01=None, sample_tok=None, node_p=None,
                    stream=None):
    """Temperature sampling at every tree node. ``logits`` float32
    [B,Qc,V] (V a multiple of 4), ``u01`` float32 [B,Qc] (not read when
    temperature <= 0, the greedy limit). Returns (sample_tok int32 [B,Qc],
    node_p float32 [B,Qc]); pass sample_tok to ddt_tree_accept as its target."""
    _need(logits, "logits", _F32, (tree.B, tree.Qc, None))
    if u01 is not None:
        _need(u01, "u01", _F32, (tree.B, tree.Qc))
    if sample_tok is not None:
        _need(sample_tok, "sample_tok", _I32, (tree.B, tree.Qc))
    if node_p is not None:
        _need(node_p, "node_p", _F32, (tree.B, tree.Qc))
    _on_device(logits, u01, sample_tok, node_p, tree.token, tree.parent, tree.n_nodes, tree.status,
               stream=stream)
    B, Qc, V = logits.shape
    if sample_tok is None:
        sample_tok = torch.empty(B, Qc, dtype=torch.int32, device=logits.device)
    if node_p is None:
        node_p = torch.empty(B, Qc, dtype=torch.float32, device=logits.device)
    t = tree.c()
    _check(lib().ddt_tree_sample(ctypes.byref(t), _ptr(logits), V, float(temperature), _ptr(u01),
                                 _ptr(sample_tok), _ptr(node_p), _stream_ptr(stream)), "ddt_tree_sample")
    return sample_tok, node_p


class VerifyStep:
    """All buffers of one ddt_verify_step call, allocated once.

    ``run()`` enqueues the whole step (build -> attention -> merge -> accept)
    through the single C-ABI call, with the marshalled structs prebuilt so a
    call costs one ctypes transition.
    """

    def __init__(self, tok, lp, root_tok, vocab: int, budget: int, q_lat, q_rope, c_kv, k_rope,
                 prefix_len, target_argmax, scale: float, acc: "Accept | None" = None):
        _need(tok, "tok", _I32, (None, None, None))
        dev = tok.device
        B, D, K = tok.shape
        _need(lp, "lp", _F32, (B, D, K))
        _need(root_tok, "root_tok", _I32, (B,))
        shape = Tree(B, D, budget + 1, 0, *([None] * 10))  # (only B and Qc are read)
        H = _need_attn(q_lat, q_rope, c_kv, k_rope, prefix_len, shape)
        _need(target_argmax, "target_argmax", _I32, (B, budget + 1))
        if acc is not None:
            _need_accept(acc, B, D)
            _on_device(acc.accept_len, acc.accept_idx, acc.commit_tok, acc.next_root)
        _on_device(tok, lp, root_tok, q_lat, q_rope, c_kv, k_rope, prefix_len, target_argmax)
        self.inputs = (tok, lp, root_tok, q_lat, q_rope, c_kv, k_rope, prefix_len, target_argmax)
        self.tree = Tree.empty(B, D, budget, dev)
        self.acc = acc if acc is not None else Accept.empty(B, D, dev)
        self.out = torch.empty(B, budget + 1, H, LATENT, dtype=torch.float32, device=dev)
        self.lse = torch.empty(B, budget + 1, H, dtype=torch.float32, device=dev)
        self.ws_bytes = ddt_workspace_size(B, D, K, budget, H, c_kv.shape[1])
        self.workspace = torch.empty(max(self.ws_bytes, 1), dtype=torch.uint8, device=dev)
        self.budget = budget
        self.scale = float(scale)
        self._d = draft_struct(tok, lp, root_tok, vocab)
        self._t = self.tree.c()
        self._a = attn_in_struct(q_lat, q_rope, c_kv, k_rope, prefix_len)
        self._o = DdtAttnOut(_ptr(self.out), _ptr(self.lse))
        self._c = self.acc.c()
        self._tg = _ptr(target_argmax)
        self._dev = dev.index

    def run(self, stream=None):
        if stream is not None and stream.device.index != self._dev:
            raise ValueError(f"stream of {stream.device}, but the step's tensors are on cuda:{self._dev}")
        rc = lib().ddt_verify_step(ctypes.byref(self._d), self.budget, ctypes.byref(self._t),
                                   ctypes.byref(self._a), self.scale, ctypes.byref(self._o),
                                   self._tg, ctypes.byref(self._c), _ptr(self.workspace),
                                   self.ws_bytes, _stream_ptr(stream))
        _check(rc, "ddt_verify_step")


def ddt_read_device_status(status: torch.Tensor):
    import numpy as np
    host = np.empty(status.numel(), np.int32)
    _check(lib().ddt_read_device_status(_ptr(status), status.numel(),
                                        host.ctypes.data_as(ctypes.c_void_p)),
           "ddt_read_device_status")
    return host


def ddt_selftest_bounded_wait(status: torch.Tensor, timeout_us: int, stream=None):
    _check(lib().ddt_selftest_bounded_wait(_ptr(status), int(timeout_us), _stream_ptr(stream)),
           "ddt_selftest_bounded_wait")
