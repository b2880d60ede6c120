"""Seeded synthetic inputs for the DDTree verify step.

This module only draws random inputs. It holds none of the verify step's
arithmetic (no tree selection, no attention, no acceptance), so the CUDA path
and the CPU oracle can both be fed from it without sharing any of the method.

Workloads follow the drafter/target description of "The Architecture of a
Thousand-Parameter Decision: Designing a Native DDTree Inference Engine for
Kimi K2.6" (section "What to Build New", items 2-4: per-depth top-k drafter
output, latent KV of 576 elements per token, tree-verify over up to 64 nodes)
and the five seeded configurations below. No public dataset is involved.

Recipe (one ``numpy.random.default_rng(20260 + config_index)`` per config):

* drafter rows: for every (b, d) draw K distinct token ids uniformly from
  [0, vocab), K+1 logits ~ N(0, 2); log-probs are the log-softmax of the K+1
  logits in float64 with the last (the "rest mass") dropped, sorted
  descending together with their tokens, then cast to float32;
* "underfull" sequences get log-probs [0, -inf, -inf, ...] on every row, which
  makes their draft tree a single chain;
* root tokens uniform in [0, vocab);
* q_lat, q_rope, c_kv, k_rope ~ N(0, 1) rounded to bfloat16 (round to nearest
  even); the prefix length T_b is fixed per config or uniform in an inclusive
  range; node m of sequence b owns KV row T_b + m;
* target argmax per tree node: with probability p the rank-0 token of the next
  depth row, else a uniform id (nodes at the last depth always draw uniform);
* target logits per tree node (sampling path): float32 background
  N(0, sigma^2) over the whole vocabulary; a node at depth d < D then gets the
  drafter's row-d tokens raised to log(V) + sigma^2 / 2 + lead - step * rank
  (log(V) + sigma^2 / 2 is about the log of the background's total mass, so
  the drafter's rank-0 token carries roughly half the probability at
  temperature 1 and the target agrees with the draft tree often, as a
  well-matched drafter would); the uniforms for sampling are float32 draws in
  [0, 1). The sampling draws of config k come from their own
  ``default_rng(20360 + k)``, after the tree is known.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

NEG_INF = np.float32(-np.inf)
LATENT = 512
ROPE = 64
# 1/sqrt(192): a head's q.k width before absorption (128 no-position + 64 rotary)
SOFTMAX_SCALE = 1.0 / math.sqrt(192.0)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    D: int
    K: int
    budget: int
    H: int
    T: object            # int, or (lo, hi) inclusive for a ragged prefix
    vocab: int
    p_match: float
    underfull: int = 0   # number of leading sequences whose drafter rows are a chain

    @property
    def Qc(self) -> int:
        return self.budget + 1

    @property
    def W(self) -> int:
        return (self.Qc + 63) // 64

    @property
    def T_max(self) -> int:
        return self.T[1] if isinstance(self.T, tuple) else self.T


# The five seeded workloads: tiny, single stream at budget 8, small batch at
# budget 16 with ragged prefixes, wide batch with a deep tree and underfull
# sequences, maximum budget with a long context.
WORKLOADS = [
    Workload("tiny_b1_d4_k4_q9_h4_t64", 1, 4, 4, 8, 4, 64, 1000, 0.7),
    Workload("single_stream_b1_d8_k8_q9_h64_t4096", 1, 8, 8, 8, 64, 4096, 163840, 0.7),
    Workload("small_batch_b8_d8_k8_q17_h64_t4096to8192", 8, 8, 8, 16, 64, (4096, 8192), 163840, 0.75),
    Workload("wide_batch_b64_d15_k4_q33_h64_t2048", 64, 15, 4, 32, 64, 2048, 163840, 0.7, underfull=4),
    Workload("max_budget_b4_d16_k8_q65_h64_t32768", 4, 16, 8, 64, 64, 32768, 163840, 0.8),
]

SEED_BASE = 20260


def rng_for(index: int) -> np.random.Generator:
    return np.random.default_rng(SEED_BASE + index)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); return the uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = 0x7FC0
    return r


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def draft_rows(rng: np.random.Generator, B: int, D: int, K: int, vocab: int,
               underfull: int = 0):
    """Drafter per-depth top-K: tokens int32 [B,D,K], log-probs float32 [B,D,K]."""
    tok = np.empty((B, D, K), np.int32)
    lp = np.empty((B, D, K), np.float32)
    for b in range(B):
        for d in range(D):
            ids = rng.choice(vocab, K, replace=False)
            logits = rng.normal(0.0, 2.0, K + 1)
            mx = logits.max()
            ls = logits - (mx + math.log(np.exp(logits - mx).sum()))
            ls = ls[:K]
            order = np.argsort(-ls, kind="stable")
            tok[b, d] = ids[order]
            lp[b, d] = ls[order].astype(np.float32)
            if b < underfull:
                lp[b, d] = NEG_INF
                lp[b, d, 0] = 0.0
    return tok, lp


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) values rounded to bfloat16, returned as uint16 bit patterns."""
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    step = 1 << 24
    for s in range(0, n, step):
        e = min(n, s + step)
        out[s:e] = f32_to_bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


@dataclasses.dataclass
class StepInputs:
    wl: Workload
    draft_tok: np.ndarray     # int32 [B,D,K]
    draft_lp: np.ndarray      # float32 [B,D,K]
    root_tok: np.ndarray      # int32 [B]
    prefix_len: np.ndarray    # int32 [B]
    Tcap: int
    q_lat: np.ndarray         # uint16 (bf16 bits) [B,Qc,H,512]
    q_rope: np.ndarray        # uint16 [B,Qc,H,64]
    c_kv: np.ndarray          # uint16 [B,Tcap,512]
    k_rope: np.ndarray        # uint16 [B,Tcap,64]
    target_u: np.ndarray      # float64 [B,Qc] uniform draws for the synthetic target
    target_alt: np.ndarray    # int32 [B,Qc] uniform token draws for the synthetic target
    scale: float


def make_inputs(index: int, wl: Workload | None = None, *, attention: bool = True,
                tail_fill: str = "normal") -> StepInputs:
    """Draw every input of one verify step for workload ``index``.

    ``tail_fill`` chooses what sits in KV rows past T_b + Qc (never visible):
    "normal" (more N(0,1) rows) or "nan" (NaN rows, to prove they are never read
    into a result).
    """
    wl = wl or WORKLOADS[index]
    rng = rng_for(index)
    tok, lp = draft_rows(rng, wl.B, wl.D, wl.K, wl.vocab, wl.underfull)
    root = rng.integers(0, wl.vocab, wl.B).astype(np.int32)
    if isinstance(wl.T, tuple):
        T = rng.integers(wl.T[0], wl.T[1] + 1, wl.B).astype(np.int32)
    else:
        T = np.full(wl.B, wl.T, np.int32)
    Tcap = int(T.max()) + wl.Qc
    Tcap = (Tcap + 7) // 8 * 8
    target_u = rng.random((wl.B, wl.Qc))
    target_alt = rng.integers(0, wl.vocab, (wl.B, wl.Qc)).astype(np.int32)
    if attention:
        q_lat = normal_bf16(rng, (wl.B, wl.Qc, wl.H, LATENT))
        q_rope = normal_bf16(rng, (wl.B, wl.Qc, wl.H, ROPE))
        c_kv = normal_bf16(rng, (wl.B, Tcap, LATENT))
        k_rope = normal_bf16(rng, (wl.B, Tcap, ROPE))
        if tail_fill == "nan":
            for b in range(wl.B):
                c_kv[b, T[b] + wl.Qc:] = 0x7FC0
                k_rope[b, T[b] + wl.Qc:] = 0x7FC0
    else:
        q_lat = q_rope = c_kv = k_rope = None
    return StepInputs(wl, tok, lp, root, T, Tcap, q_lat, q_rope, c_kv, k_rope,
                      target_u, target_alt, SOFTMAX_SCALE)


def synth_target_argmax(depth: np.ndarray, n_nodes: np.ndarray, draft_tok: np.ndarray,
                        u: np.ndarray, alt: np.ndarray, p: float) -> np.ndarray:
    """Synthetic target model: the argmax the target 'predicts' after each node.

    ``depth`` [B,Qc] and ``n_nodes`` [B] describe an already-built tree (the
    caller passes the tree it trusts); ``u``/``alt`` are the seeded draws.
    A node at depth d < D predicts the drafter's rank-0 token of depth row d
    with probability p, otherwise the uniform draw.
    """
    B, Qc = depth.shape
    D = draft_tok.shape[1]
    out = alt.copy()
    for b in range(B):
        for i in range(int(n_nodes[b])):
            d = int(depth[b, i])
            if d < D and u[b, i] < p:
                out[b, i] = draft_tok[b, d, 0]
    return out


def target_logits(rng: np.random.Generator, depth: np.ndarray, n_nodes: np.ndarray,
                  draft_tok: np.ndarray, vocab: int, sigma: float = 1.5, lead: float = 1.0,
                  step: float = 1.5) -> np.ndarray:
    """Synthetic target logits after each tree node: float32 [B,Qc,vocab].

    ``depth`` [B,Qc] and ``n_nodes`` [B] describe a built tree (the caller
    passes the tree it trusts). Padding slots keep the plain background."""
    B, Qc = depth.shape
    D, K = draft_tok.shape[1], draft_tok.shape[2]
    out = np.empty((B, Qc, vocab), np.float32)
    for b in range(B):
        for i in range(Qc):
            out[b, i] = rng.standard_normal(vocab, dtype=np.float32) * np.float32(sigma)
    base = math.log(vocab) + sigma * sigma / 2.0
    boost = (base + lead - step * np.arange(K)).astype(np.float32)
    for b in range(B):
        for i in range(int(n_nodes[b])):
            d = int(depth[b, i])
            if 0 <= d < D:
                ids = draft_tok[b, d]
                keep = ids < vocab  # a smaller vocabulary drops the drafter's larger ids
                out[b, i, ids[keep]] = boost[keep]
    return out


def sample_uniforms(rng: np.random.Generator, B: int, Qc: int) -> np.ndarray:
    """float32 uniforms in [0, 1), one per tree node slot: [B,Qc]."""
    return rng.random((B, Qc), dtype=np.float32)


def sampling_inputs(index: int, depth: np.ndarray, n_nodes: np.ndarray, draft_tok: np.ndarray,
                    vocab: int | None = None):
    """(logits float32 [B,Qc,V], u01 float32 [B,Qc]) for workload ``index``
    and the tree given by ``depth`` / ``n_nodes``."""
    wl = WORKLOADS[index]
    rng = np.random.default_rng(SEED_BASE + 100 + index)
    V = wl.vocab if vocab is None else vocab
    lg = target_logits(rng, depth, n_nodes, draft_tok, V)
    return lg, sample_uniforms(rng, depth.shape[0], depth.shape[1])
