/*
 * libddtree — the DDTree speculative-decoding verify step on one GB300 GPU.
 *
 * The verify step has three parts, chained on one CUDA stream with no host
 * round-trip:
 *
 *   1. draft-tree build   best-first top-k expansion of the drafter's per-depth
 *                         top-K log-probs into a token tree ("The Architecture
 *                         of a Thousand-Parameter Decision: Designing a Native
 *                         DDTree Inference Engine for Kimi K2.6", section "What
 *                         to Build New", item 3 — a GPU builder replacing the
 *                         per-request CPU heapq and its host syncs);
 *   2. verify attention   MLA-absorb attention of every tree node against the
 *                         latent KV prefix plus its own ancestors (same page,
 *                         "What to Build New", item 2; "The Milestone Message:
 *                         When an AI Summarizes Its Own Engineering Triumph",
 *                         section "Architectural Abstraction": nodes processed
 *                         at positions L+depth with the mask [ones | visibility]);
 *   3. greedy accept      follow the verified tree from the root while the
 *                         target's argmax matches a child ("The Architecture of
 *                         Closure: How a Summary Message Encodes an Entire
 *                         Engineering Session", section "The Table as a
 *                         Decision Artifact", the tree_accept.cu row).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every pointer inside the structs is a DEVICE pointer on the current CUDA
 *    device, owned by the caller. Arrays are dense, row-major, in the shapes
 *    given below; there are no stride arguments. The library allocates no
 *    memory and keeps no state between calls; it is safe to call from several
 *    host threads on different streams.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). All work
 *    is enqueued on it; no call synchronises the device or the stream (except
 *    ddt_read_device_status, a debugging helper). The enqueuing calls are safe
 *    to record into a CUDA graph, provided one call of the same kind has been
 *    made on the device before capture starts (the first call resolves the
 *    driver's tensor-map encoder and sets kernel attributes).
 *  - Node index 0 of every tree is the root (the last verified token). A tree
 *    holds up to Qc = budget + 1 nodes; W = ceil(Qc / 64) is the number of
 *    uint64 words in each node's ancestor mask.
 *  - Return value: DDT_OK, or an error detected on the host before anything
 *    is enqueued (DDT_E_INVAL: null pointer, shape out of range, struct fields
 *    inconsistent, misaligned buffer, workspace too small; DDT_E_UNSUPPORTED:
 *    the current device is not sm_103; DDT_E_CUDA: a launch failed). Problems
 *    found in the DATA are reported per sequence in tree->status on the device
 *    without any sync: DDT_E_BADINPUT (bad drafter row, token out of range,
 *    prefix length out of range) or DDT_E_TIMEOUT (a bounded on-chip wait
 *    expired); the attention kernel writes DDT_E_CUDA to every sequence
 *    if it finds its shared memory misaligned for its operand
 *    layouts (not expected; its outputs are then undefined). A flagged
 *    sequence otherwise still gets defined outputs: a root-only tree
 *    (n_nodes = 1), zero attention rows, accept_len = 1.
 */
#ifndef DDTREE_H
#define DDTREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    DDT_OK = 0,
    DDT_E_INVAL = 1,
    DDT_E_CUDA = 2,
    DDT_E_UNSUPPORTED = 3,
    DDT_E_BADINPUT = 4,
    DDT_E_TIMEOUT = 5,
    DDT_E_SCRATCH_LIMIT = 6  /* ddt_verify_mla_attn_noalloc: shape needs more scratch than it holds */
};

#define DDT_MAX_DEPTH 16   /* D */
#define DDT_MAX_TOPK 16    /* K */
#define DDT_MAX_BUDGET 64  /* budget; Qc <= 65, W <= 2 */
#define DDT_LATENT 512     /* MLA latent width (the value / c_kv width) */
#define DDT_ROPE 64        /* MLA decoupled rotary width */

/* Drafter output for B sequences: per depth row d (0-based, the drafter's
 * guess for depth d+1) the top-K tokens and their log-probs. */
typedef struct ddt_draft {
    int B;                   /* sequences, >= 1 */
    int D;                   /* depth rows, 1..16 */
    int K;                   /* top-K per row, 1..16 */
    int vocab;               /* valid token ids are [0, vocab) */
    const int32_t *tok;      /* [B,D,K] token ids */
    const float *lp;         /* [B,D,K] log-probs: each row finite or -inf, <= 0,
                                non-increasing in k */
    const int32_t *root_tok; /* [B] the last verified token (node 0) */
} ddt_draft;

/* A built tree, Qc node slots per sequence. Slots i >= n_nodes[b] are padding:
 * token/parent/depth/rank/first_child/next_sibling = -1, score = -inf, mask = 0. */
typedef struct ddt_tree {
    int B, D, Qc, W;         /* host-side shape; Qc = budget+1, W = ceil(Qc/64) */
    int32_t *token;          /* [B,Qc] node token (root: root_tok) */
    int32_t *parent;         /* [B,Qc] parent index (< own index), root -1 */
    int32_t *depth;          /* [B,Qc] root 0 */
    int32_t *rank;           /* [B,Qc] rank within its depth row, root -1 */
    float *score;            /* [B,Qc] float32 sum of log-probs root..node */
    int32_t *first_child;    /* [B,Qc] smallest child index or -1 */
    int32_t *next_sibling;   /* [B,Qc] next larger index with the same parent or -1 */
    uint64_t *mask;          /* [B,Qc,W] bit m of node i: m is i or an ancestor of i */
    int32_t *n_nodes;        /* [B] 1 + selected draft nodes */
    int32_t *status;         /* [B] DDT_OK / DDT_E_BADINPUT / DDT_E_TIMEOUT (/ DDT_E_CUDA, see above) */
} ddt_tree;

/* Attention inputs in bfloat16 (raw 16-bit patterns). Node m of sequence b
 * must already have its latent and rotary key at KV row prefix_len[b] + m. */
typedef struct ddt_attn_in {
    int H;                   /* heads, >= 1 */
    int Tcap;                /* KV rows per sequence; prefix_len[b] + n_nodes[b] <= Tcap */
    const void *q_lat;       /* [B,Qc,H,512] absorbed query (w_kc folded in); 16 B aligned */
    const void *q_rope;      /* [B,Qc,H,64] rotary query; 16 B aligned */
    const void *c_kv;        /* [B,Tcap,512] latent KV; 16 B aligned */
    const void *k_rope;      /* [B,Tcap,64] rotary key; 16 B aligned */
    const int32_t *prefix_len; /* [B] T_b, committed prefix length (>= 0) */
} ddt_attn_in;

/* Attention outputs, float32. Row (b, i, h) for i >= n_nodes[b] is zero with
 * lse = -inf. */
typedef struct ddt_attn_out {
    float *out;              /* [B,Qc,H,512] softmax-weighted latent, before w_vc */
    float *lse;              /* [B,Qc,H] natural-log sum of exp(logits) */
} ddt_attn_out;

/* Greedy accept result; rows have D+1 entries, unused entries are -1. */
typedef struct ddt_accept {
    int32_t *accept_len;     /* [B] accepted nodes including the root, 1..D+1 */
    int32_t *accept_idx;     /* [B,D+1] node indices root first */
    int32_t *commit_tok;     /* [B,D+1] accepted draft tokens, then the bonus token */
    int32_t *next_root;      /* [B] bonus token: target argmax after the last node */
} ddt_accept;

/* Bytes of device workspace ddt_verify_mla_attn / ddt_verify_step need for
 * this shape on the CURRENT device (the split of the key range over CTAs
 * depends on its SM count). May be 0. D and K are accepted for symmetry with
 * the other calls and do not change the result. Returns 0 for shapes the
 * library rejects. */
size_t ddt_workspace_size(int B, int D, int K, int budget, int H, int Tcap);

/* Step 1: build B draft trees of up to `budget` (1..64) nodes plus the root.
 * Selection order is score descending, then depth ascending, then rank path
 * lexicographic ascending; a candidate with score -inf is never selected.
 * Node indices follow selection order, so parent[i] < i and scores are
 * non-increasing in i. Requires out->B == in->B, out->D == in->D,
 * out->Qc == budget + 1, out->W == ceil(out->Qc / 64). */
int ddt_tree_build(const ddt_draft *in, int budget, ddt_tree *out, void *stream);

/* Step 2: for each (b, node i < n_nodes[b], head h)
 *   s_j = scale * (q_lat . c_kv[b,j] + q_rope . k_rope[b,j])
 * over the visible rows j: 0..T_b-1 and T_b+m for every bit m set in
 * mask[b,i]; out = sum_j softmax(s)_j * c_kv[b,j]; lse = log sum_j exp(s_j).
 * Computed with bfloat16 tensor-core products, float32 accumulation and a
 * float32 online softmax. `scale` must be positive and finite (else
 * DDT_E_INVAL; 1/sqrt(192) for the absorbed 128+64 head dimension).
 * `workspace` must hold ddt_workspace_size(...) bytes (it may be NULL when
 * that is 0). Reads tree->mask, tree->n_nodes and writes DDT_E_BADINPUT /
 * DDT_E_TIMEOUT into tree->status. */
int ddt_verify_mla_attn(const ddt_attn_in *in, const ddt_tree *tree, float scale,
                        ddt_attn_out *out, void *workspace, size_t ws_bytes, void *stream);

/* Step 3: greedy walk. From the root, while some child of the current node has
 * token == target_argmax[b, current] (the lowest such index), move to it.
 * target_argmax is [B,Qc] int32: the target model's argmax after each node. */
int ddt_tree_accept(const ddt_tree *tree, const int32_t *target_argmax, ddt_accept *out,
                    void *stream);

/* Steps 1-3 enqueued back to back on one stream with no host
 * synchronisation: three launches. The tree build; the attention; then,
 * when the key range is split, the key-range merge, whose grid also runs the
 * accept walk (one warp per sequence, in blocks of its own), else the accept
 * alone. Results are identical to ddt_tree_build + ddt_verify_mla_attn +
 * ddt_tree_accept on the same stream. */
int ddt_verify_step(const ddt_draft *draft, int budget, ddt_tree *tree,
                    const ddt_attn_in *attn, float scale, ddt_attn_out *attn_out,
                    const int32_t *target_argmax, ddt_accept *acc, void *workspace,
                    size_t ws_bytes, void *stream);

/* Step 2 with the latent output in bfloat16, the type the absorbed-MLA
 * value up-projection that follows it takes ("The Milestone Message",
 * section "MLA": the absorb form with w_kc / w_vc). Same as
 * ddt_verify_mla_attn, except that out_bf16 [B,Qc,H,512] (16-byte aligned)
 * receives each output element rounded to nearest even from its float32
 * value; lse stays float32 [B,Qc,H]. Same workspace and errors. */
int ddt_verify_mla_attn_bf16(const ddt_attn_in *in, const ddt_tree *tree, float scale, uint16_t *out_bf16,
                             float *lse, void *workspace, size_t ws_bytes, void *stream);

/* Step 2 on a block-table (paged, page size 1) latent KV cache, the cache
 * layout the pages use ("The Architecture of a Thousand-Parameter Decision:
 * Designing a Native DDTree Inference Engine for Kimi K2.6", "What to Build
 * New", item 5: a paged MLA-latent KV cache manager; "The Milestone Message",
 * "Architectural Abstraction" for the positions). Same as ddt_verify_mla_attn
 * except that in->c_kv and in->k_rope are pools of `pool_rows` rows
 * ([pool_rows,512] and [pool_rows,64] bfloat16), and key position p of
 * sequence b (prefix keys 0..T_b-1, node m at T_b + m) is pool row
 * kv_index[b * in->Tcap + p]. kv_index is int32 [B, Tcap]; entries at and
 * past a sequence's key end (T_b + n_nodes[b]) are not read for anything but
 * may hold any value. An entry below the key end outside [0, pool_rows)
 * flags the sequence DDT_E_BADINPUT (its rows are then undefined); host
 * errors as for ddt_verify_mla_attn, plus DDT_E_INVAL for a null kv_index or
 * pool_rows < 1. Workspace: ddt_workspace_size as for the contiguous cache. */
int ddt_verify_mla_attn_paged(const ddt_attn_in *in, const ddt_tree *tree, float scale,
                              ddt_attn_out *out, void *workspace, size_t ws_bytes,
                              const int32_t *kv_index, int pool_rows, void *stream);

/* After accept: the KV append of the committed tokens ("The Architecture of a
 * Thousand-Parameter Decision: Designing a Native DDTree Inference Engine for
 * Kimi K2.6", "What to Build New", items 4 and 5: the step ends
 * draft -> build -> verify -> accept -> append; key layout of "The Milestone
 * Message", "Architectural Abstraction": node m's key at position L + m).
 * For each sequence b with T = prefix_len[b] and L = acc->accept_len[b], the
 * keys of the accepted path acc->accept_idx[b][0..L-1] (node 0, the root, is
 * already at row T) become rows T .. T+L-1 of c_kv [B,Tcap,512] and k_rope
 * [B,Tcap,64] (bfloat16 bit patterns, modified in place), and prefix_len[b]
 * becomes T + L. Rows below T are not touched; rows from T + L on keep
 * whatever they held. D is the accept rows' length minus one. Host errors:
 * DDT_E_INVAL for a null pointer, B < 1, D outside [1, DDT_MAX_DEPTH], Tcap
 * < 1 or a c_kv / k_rope pointer not 16-byte aligned. A sequence whose
 * accept_len, path indices (must rise from 0) or prefix length do not fit
 * Tcap is left unchanged and gets DDT_E_BADINPUT in status[b]; no sync. */
int ddt_kv_commit(const ddt_accept *acc, int B, int D, int Tcap, void *c_kv, void *k_rope,
                  int32_t *prefix_len, int32_t *status, void *stream);

/* Temperature sampling at every tree node, the sampling commit path ("The
 * Architecture of a Thousand-Parameter Decision: Designing a Native DDTree
 * Inference Engine for Kimi K2.6", section "What to Reuse", item 3:
 * temperature-based sampling from the verified token distribution; section
 * "What to Build New", item 2: the sampling-probability path that normalises
 * the target's probabilities over the tree nodes, and item 5: greedy and
 * temperature commit paths).
 *
 * logits is float32 [B, tree->Qc, vocab] (16-byte aligned): row (b, i) holds
 * the target's logits after node i. Its distribution is
 * p_j = exp((x_j - M) / temperature) / S, M the row's largest logit. With
 * u = u01[b, i] (float32 [B, Qc]) the node's sample is the first token id j
 * with p_j > 0 whose cumulative probability p_0 + ... + p_j exceeds u; when
 * none does (u >= 1, NaN, or rounding at the top) the last token with
 * p_j > 0. temperature <= 0 selects the greedy limit: the first index of the
 * largest logit (u01 is then not read and may be NULL).
 *
 *   sample_tok int32 [B, Qc]: the sample after each node; -1 for node slots
 *              at or past n_nodes[b] and for rows with no distribution.
 *   node_p     float32 [B, Qc]: node c's token's probability under its
 *              parent's row (1 or 0 in the greedy limit); node 0 gets 1,
 *              slots at or past n_nodes[b] get 0.
 *
 * Passing sample_tok to ddt_tree_accept as its target commits, at every
 * accepted node, a token distributed as p (lossless tree sampling with a
 * deterministic draft tree). Arithmetic: weights 2^((x - M) log2(e) / T)
 * in float32 (hardware exp2, weights below 2^-126 of the largest flush to
 * zero), sums in float32 up to 20480 tokens and float64 above; node_p is
 * the child token's weight over the row total in float32. Cumulative
 * probabilities are off by at most ~1e-5 of the total (worst case), so a
 * sample can differ from exact arithmetic's only for u that close to a
 * token boundary. A row holding a NaN, or (temperature > 0)
 * whose largest logit is +-inf, gets sample -1, children's node_p 0 and
 * DDT_E_BADINPUT in tree->status[b]; so does a child token outside
 * [0, vocab). Host errors: DDT_E_INVAL for a null pointer, vocab < 4 or not
 * a multiple of 4 or above 2883584 (1441792 on a device without 16-CTA
 * clusters), misaligned logits, a NaN or infinite temperature, a positive
 * temperature below 1e-30, or tree shape out of range. Reads tree->token,
 * tree->parent, tree->n_nodes; allocates nothing. */
int ddt_tree_sample(const ddt_tree *tree, const float *logits, int vocab, float temperature,
                    const float *u01, int32_t *sample_tok, float *node_p, void *stream);

/* Bytes of device scratch held by ddt_verify_mla_attn_noalloc (64 MiB). */
#define DDT_NOALLOC_SCRATCH_BYTES (64u << 20)

/* Step 2 for callers that cannot allocate device memory. The pages have no
 * counterpart; this is a convenience of this library.
 *
 * ddt_verify_mla_attn needs a workspace from the caller whenever it splits
 * each sequence's keys over several CTAs. Some callers cannot provide one:
 * a serving engine that reserves nearly all HBM for its KV cache at start-up
 * and has no allocator left to hand out more, a plugin or C host that is
 * given only its input and output buffers, or code that must not call
 * cudaMalloc because cudaMalloc synchronises the device. This call computes
 * exactly what ddt_verify_mla_attn computes (same kernels, same arguments
 * without the workspace) using a scratch array that the library defines at
 * file scope: DDT_NOALLOC_SCRATCH_BYTES on every GPU that loads the library,
 * held until the process exits. It allocates nothing.
 *
 *  - Arguments are checked first, as ddt_verify_mla_attn checks them
 *    (DDT_E_INVAL, DDT_E_UNSUPPORTED); then shapes whose key-range partials
 *    would not fit return DDT_E_SCRATCH_LIMIT before anything is enqueued
 *    (ddt_workspace_size tells how much a shape needs on the current device).
 *  - The first call on a device whose shape splits its keys looks up the
 *    scratch array's device address (cudaGetSymbolAddress, with that device
 *    current); make that first call before any stream capture. Made while
 *    `stream` is capturing, it returns DDT_E_INVAL and enqueues nothing. A
 *    failed lookup returns DDT_E_CUDA and is retried by the next call.
 *  - All calls share the one array and it keeps the last call's contents.
 *    Nothing in it needs to start at zero: a call writes every partial it
 *    later reads. Calls whose kernels overlap on the GPU (several streams,
 *    or several host threads) race on the array: serialise them. */
int ddt_verify_mla_attn_noalloc(const ddt_attn_in *in, const ddt_tree *tree, float scale,
                                ddt_attn_out *out, void *stream);

/* Static text for a status code. */
const char *ddt_status_str(int code);

/* Debugging helper, NOT for the hot path: copies B status words to the host
 * with a synchronous cudaMemcpy. */
int ddt_read_device_status(const int32_t *dev_status, int B, int32_t *host_out);

/* Self-test of the bounded on-chip wait: launches one CTA that waits on an
 * mbarrier nothing will ever arrive on, with a limit of `timeout_us`
 * microseconds, after which it writes DDT_E_TIMEOUT into *dev_status and
 * returns normally. Used to check the timeout path without faulting or
 * hanging the GPU. */
int ddt_selftest_bounded_wait(int32_t *dev_status, unsigned timeout_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DDTREE_H */
