"""CPU oracle for the DDTree verify step (TEST INFRASTRUCTURE).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. The CUDA library never links or calls it; the
two share no code. The arithmetic lives in ``ddt_oracle.c`` (plain C, float64
attention, float32 tree scores); this module only builds it with gcc and
marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ddt_oracle.c")
_LIB = os.path.join(_HERE, "libddt_oracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
BADINPUT = 4


def build(force: bool = False) -> str:
    """Compile ddt_oracle.c into libddt_oracle.so (gcc, OpenMP, strict fp)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i = ctypes.c_int
            lib.ddto_tree_build.argtypes = [i, i, i, i, P, P, P, i, i, i] + [P] * 10
            lib.ddto_tree_build.restype = i
            lib.ddto_attn_rows.argtypes = [i, i, i, i, P, P, P, P, P, P, P, ctypes.c_double,
                                           P, ctypes.c_long, P, P, i]
            lib.ddto_attn_rows.restype = i
            lib.ddto_tree_accept.argtypes = [i, i, i, P, P, P, P, P, P, P, P]
            lib.ddto_tree_accept.restype = i
            lib.ddto_kv_commit.argtypes = [i, i, i, P, P, P, P, P, P]
            lib.ddto_kv_commit.restype = i
            lib.ddto_tree_sample.argtypes = [i, i, i, P, ctypes.c_double, P, P, P, P, P, P, P]
            lib.ddto_tree_sample.restype = i
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


class Tree(dict):
    """Named tree arrays: token, parent, depth, rank, score, first_child,
    next_sibling ([B,Qc]), mask ([B,Qc,W] uint64), n_nodes, status ([B])."""
    __getattr__ = dict.__getitem__


def tree_build(draft_tok, draft_lp, root_tok, budget: int, vocab: int) -> Tree:
    lib = _load()
    draft_tok = np.ascontiguousarray(draft_tok, np.int32)
    draft_lp = np.ascontiguousarray(draft_lp, np.float32)
    root_tok = np.ascontiguousarray(root_tok, np.int32)
    B, D, K = draft_tok.shape
    Qc = budget + 1
    W = (Qc + 63) // 64
    t = Tree(
        token=np.empty((B, Qc), np.int32), parent=np.empty((B, Qc), np.int32),
        depth=np.empty((B, Qc), np.int32), rank=np.empty((B, Qc), np.int32),
        score=np.empty((B, Qc), np.float32), first_child=np.empty((B, Qc), np.int32),
        next_sibling=np.empty((B, Qc), np.int32), mask=np.empty((B, Qc, W), np.uint64),
        n_nodes=np.empty(B, np.int32), status=np.empty(B, np.int32))
    rc = lib.ddto_tree_build(B, D, K, vocab, _p(draft_tok), _p(draft_lp), _p(root_tok), budget,
                             Qc, W, _p(t.token), _p(t.parent), _p(t.depth), _p(t.rank),
                             _p(t.score), _p(t.first_child), _p(t.next_sibling), _p(t.mask),
                             _p(t.n_nodes), _p(t.status))
    if rc != 0:
        raise ValueError("oracle tree_build rejected its arguments")
    return t


def attn_rows(q_lat, q_rope, c_kv, k_rope, prefix_len, mask, n_nodes, scale: float,
              rows, n_threads: int = 0):
    """float64 attention for the (b, node, head) triples in ``rows`` [n,3].

    Inputs are bfloat16 bit patterns (uint16). Returns (out [n,512] float64,
    lse [n] float64, threads used)."""
    lib = _load()
    B, Qc, H, _ = q_lat.shape
    Tcap = c_kv.shape[1]
    W = mask.shape[2]
    rows = np.ascontiguousarray(rows, np.int32).reshape(-1, 3)
    n = rows.shape[0]
    out = np.empty((n, 512), np.float64)
    lse = np.empty(n, np.float64)
    arrs = [np.ascontiguousarray(a) for a in (q_lat, q_rope, c_kv, k_rope)]
    for a in arrs:
        assert a.dtype == np.uint16
    pl = np.ascontiguousarray(prefix_len, np.int32)
    mk = np.ascontiguousarray(mask, np.uint64)
    nn = np.ascontiguousarray(n_nodes, np.int32)
    used = lib.ddto_attn_rows(Qc, W, H, Tcap, *[_p(a) for a in arrs], _p(pl), _p(mk), _p(nn),
                              float(scale), _p(rows), n, _p(out), _p(lse), int(n_threads))
    return out, lse, used


def attn_all(q_lat, q_rope, c_kv, k_rope, prefix_len, mask, n_nodes, scale: float,
             n_threads: int = 0):
    """Every row: out [B,Qc,H,512] float64, lse [B,Qc,H] float64."""
    B, Qc, H, _ = q_lat.shape
    b, i, h = np.meshgrid(np.arange(B), np.arange(Qc), np.arange(H), indexing="ij")
    rows = np.stack([b.ravel(), i.ravel(), h.ravel()], 1)
    out, lse, _ = attn_rows(q_lat, q_rope, c_kv, k_rope, prefix_len, mask, n_nodes, scale,
                            rows, n_threads)
    return out.reshape(B, Qc, H, 512), lse.reshape(B, Qc, H)


def tree_accept(tree: Tree, target_argmax, D: int):
    """Greedy walk. Returns dict accept_len [B], accept_idx [B,D+1],
    commit_tok [B,D+1], next_root [B]."""
    lib = _load()
    B, Qc = tree.token.shape
    tg = np.ascontiguousarray(target_argmax, np.int32)
    r = dict(accept_len=np.empty(B, np.int32), accept_idx=np.empty((B, D + 1), np.int32),
             commit_tok=np.empty((B, D + 1), np.int32), next_root=np.empty(B, np.int32))
    lib.ddto_tree_accept(B, D, Qc, _p(tree.token), _p(tree.parent), _p(tree.n_nodes), _p(tg),
                         _p(r["accept_len"]), _p(r["accept_idx"]), _p(r["commit_tok"]),
                         _p(r["next_root"]))
    return r


def kv_commit(accept_len, accept_idx, c_kv_bits, k_rope_bits, prefix_len, status, D: int):
    """Moves the accepted path's keys into the committed prefix. Works on
    copies: c_kv_bits [B,Tcap,512] and k_rope_bits [B,Tcap,64] as uint16 bf16
    bit patterns, prefix_len and status int32 [B]. Returns the four new arrays
    (c_kv, k_rope, prefix_len, status)."""
    lib = _load()
    kv = np.array(c_kv_bits, dtype=np.uint16, order="C", copy=True)
    kr = np.array(k_rope_bits, dtype=np.uint16, order="C", copy=True)
    B, Tcap, _ = kv.shape
    pl = np.array(prefix_len, dtype=np.int32, copy=True)
    st = np.array(status, dtype=np.int32, copy=True)
    al = np.ascontiguousarray(accept_len, np.int32)
    ai = np.ascontiguousarray(accept_idx, np.int32)
    rc = lib.ddto_kv_commit(B, D, Tcap, _p(al), _p(ai), _p(kv), _p(kr), _p(pl), _p(st))
    if rc != 0:
        raise MemoryError("ddto_kv_commit: out of host memory")
    return kv, kr, pl, st


def gather_paged(pool_kv, pool_kr, kv_index):
    """The contiguous cache a block-table cache stands for: row p of sequence
    b is pool row kv_index[b, p]. Entries outside [0, P) give zero rows (such
    positions must not be visible to any node)."""
    kvi = np.asarray(kv_index)
    P = pool_kv.shape[0]
    ok = (kvi >= 0) & (kvi < P)
    idx = np.where(ok, kvi, 0)
    kv = np.asarray(pool_kv)[idx]
    kr = np.asarray(pool_kr)[idx]
    kv[~ok] = 0
    kr[~ok] = 0
    return kv, kr


def tree_sample(tree: Tree, logits, temperature: float, u01, status=None):
    """Temperature sampling at every node of the tree (float64).

    ``logits`` float32 [B,Qc,V], ``u01`` float32 [B,Qc]; ``tree`` needs
    token, parent and n_nodes. Returns (sample_tok int32 [B,Qc], node_p
    float64 [B,Qc], status int32 [B]); ``status`` (default: all OK) is copied
    and BADINPUT is set where a row has no distribution or a child token is out
    of range."""
    lib = _load()
    lg = np.ascontiguousarray(logits, np.float32)
    B, Qc, V = lg.shape
    uu = np.ascontiguousarray(u01, np.float32).reshape(B, Qc)
    st = np.zeros(B, np.int32) if status is None else np.array(status, dtype=np.int32, copy=True)
    tok = np.empty((B, Qc), np.int32)
    npb = np.empty((B, Qc), np.float64)
    rc = lib.ddto_tree_sample(B, Qc, V, _p(lg), float(temperature), _p(uu),
                              _p(np.ascontiguousarray(tree.token, np.int32)),
                              _p(np.ascontiguousarray(tree.parent, np.int32)),
                              _p(np.ascontiguousarray(tree.n_nodes, np.int32)), _p(tok), _p(npb), _p(st))
    if rc != 0:
        raise MemoryError("ddto_tree_sample: out of host memory")
    return tok, npb, st
