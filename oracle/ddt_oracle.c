/*
 * CPU oracle for the DDTree verify step.  TEST INFRASTRUCTURE ONLY: nothing on
 * the product path links or calls this file; only the tests, the smoke check
 * and the benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * Plain, slow functions, each written from its definition:
 *
 *  ddto_tree_build  best-first draft-tree expansion with a binary heap, as the
 *                   per-request CPU builder the GPU builder replaces ("The
 *                   Architecture of a Thousand-Parameter Decision", section
 *                   "What to Build New", item 3; "The Meta-Cognitive Pivot",
 *                   the paragraph on moving tree construction off the CPU heapq).
 *  ddto_attn_rows   tree-verify MLA-absorb attention in float64 for a list of
 *                   (sequence, node, head) rows ("The Architecture of a
 *                   Thousand-Parameter Decision", "What to Build New", item 2;
 *                   "The Milestone Message", section "Architectural Abstraction":
 *                   the [ones | visibility] mask over positions L + depth).
 *  ddto_kv_commit   moves the accepted nodes' latent and rotary keys into the
 *                   committed prefix ("The Architecture of a Thousand-Parameter
 *                   Decision", "What to Build New", items 4 and 5: the step
 *                   ends with an append of the committed tokens' KV; node m's
 *                   key at row T_b + m as in "The Milestone Message",
 *                   "Architectural Abstraction").
 *  ddto_tree_accept greedy follow-the-verified-tree walk ("The Architecture of
 *                   Closure", the kernel table row for tree_accept.cu).
 *  ddto_tree_sample temperature sampling at every tree node by inverse
 *                   transform, plus each node's probability under its
 *                   parent's distribution ("The Architecture of a
 *                   Thousand-Parameter Decision", "What to Reuse" item 3 and
 *                   "What to Build New" item 2: the sampling-probability path).
 *
 * Readings taken where the pages are silent (each is a choice, documented in
 * the design notes): a node is a rank path (r_1..r_d); its score is the float32
 * sum of the drafter log-probs along the path, added root to leaf with
 * round-to-nearest and no fused multiply-add; candidates are ordered by score
 * descending, then depth ascending, then rank path lexicographically
 * ascending; a -inf candidate is never selected; the root is node 0; node m's
 * key is KV row T_b + m; a node sees itself; padded rows give zeros and -inf;
 * among children with equal tokens the lowest index wins; accept_len counts
 * the root.
 *
 * Build: gcc -O2 -std=c11 -fopenmp -ffp-contract=off -shared -fPIC -lm
 * (no -ffast-math: the tree scores must be IEEE float32 sums).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BADINPUT 4
#define MAXD 16

/* ------------------------------------------------------------------ */
/* tree build                                                          */
/* ------------------------------------------------------------------ */

typedef struct {
    float score;
    int depth;               /* 1..D */
    int ranks[MAXD];         /* ranks[0..depth-1] */
    int parent_node;         /* index of the parent in the output tree */
} cand_t;

/* negative when a is selected before b */
static int cand_cmp(const cand_t *a, const cand_t *b) {
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    if (a->depth != b->depth) return a->depth < b->depth ? -1 : 1;
    for (int i = 0; i < a->depth; ++i)
        if (a->ranks[i] != b->ranks[i]) return a->ranks[i] < b->ranks[i] ? -1 : 1;
    return 0;
}

static void heap_push(cand_t *h, int *n, const cand_t *c) {
    int i = (*n)++;
    h[i] = *c;
    while (i > 0) {
        int p = (i - 1) / 2;
        if (cand_cmp(&h[i], &h[p]) >= 0) break;
        cand_t t = h[i]; h[i] = h[p]; h[p] = t;
        i = p;
    }
}

static cand_t heap_pop(cand_t *h, int *n) {
    cand_t top = h[0];
    h[0] = h[--(*n)];
    int i = 0;
    for (;;) {
        int l = 2 * i + 1, r = l + 1, m = i;
        if (l < *n && cand_cmp(&h[l], &h[m]) < 0) m = l;
        if (r < *n && cand_cmp(&h[r], &h[m]) < 0) m = r;
        if (m == i) break;
        cand_t t = h[i]; h[i] = h[m]; h[m] = t;
        i = m;
    }
    return top;
}

/* A drafter row is usable when every log-prob is finite or -inf, <= 0, and
 * the row is non-increasing; every token must lie in [0, vocab). */
static int rows_valid(int D, int K, int vocab, const int32_t *tok, const float *lp,
                      int32_t root) {
    if (root < 0 || root >= vocab) return 0;
    for (int d = 0; d < D; ++d) {
        for (int k = 0; k < K; ++k) {
            float v = lp[d * K + k];
            int32_t t = tok[d * K + k];
            if (isnan(v) || v > 0.0f || v == INFINITY) return 0;
            if (k > 0 && v > lp[d * K + k - 1]) return 0;
            if (t < 0 || t >= vocab) return 0;
        }
    }
    return 1;
}

int ddto_tree_build(int B, int D, int K, int vocab, const int32_t *draft_tok,
                    const float *draft_lp, const int32_t *root_tok, int budget, int Qc,
                    int W, int32_t *token, int32_t *parent, int32_t *depth, int32_t *rank,
                    float *score, int32_t *first_child, int32_t *next_sibling,
                    uint64_t *mask, int32_t *n_nodes, int32_t *status) {
    if (D < 1 || D > MAXD || K < 1 || budget < 1 || Qc < budget + 1 || W * 64 < Qc)
        return -1;
    cand_t *heap = (cand_t *)malloc(sizeof(cand_t) * (size_t)(2 * budget + 4));
    int (*path)[MAXD] = malloc(sizeof(int[MAXD]) * (size_t)Qc);
    for (int b = 0; b < B; ++b) {
        const int32_t *tk = draft_tok + (size_t)b * D * K;
        const float *lp = draft_lp + (size_t)b * D * K;
        int32_t *o_tok = token + (size_t)b * Qc, *o_par = parent + (size_t)b * Qc;
        int32_t *o_dep = depth + (size_t)b * Qc, *o_rank = rank + (size_t)b * Qc;
        float *o_sc = score + (size_t)b * Qc;
        int32_t *o_fc = first_child + (size_t)b * Qc, *o_ns = next_sibling + (size_t)b * Qc;
        uint64_t *o_mask = mask + (size_t)b * Qc * W;
        for (int i = 0; i < Qc; ++i) {
            o_tok[i] = o_par[i] = o_dep[i] = o_rank[i] = o_fc[i] = o_ns[i] = -1;
            o_sc[i] = -INFINITY;
            for (int w = 0; w < W; ++w) o_mask[(size_t)i * W + w] = 0;
        }
        int ok = rows_valid(D, K, vocab, tk, lp, root_tok[b]);
        status[b] = ok ? ORACLE_OK : ORACLE_BADINPUT;
        /* root */
        o_tok[0] = root_tok[b];
        o_dep[0] = 0;
        o_sc[0] = 0.0f;
        o_mask[0] = 1ull;
        int n = 1;
        if (ok) {
            int hn = 0;
            cand_t c;
            memset(&c, 0, sizeof c);
            c.depth = 1;
            c.ranks[0] = 0;
            c.parent_node = 0;
            c.score = 0.0f + lp[0];
            heap_push(heap, &hn, &c);
            while (n < budget + 1 && hn > 0) {
                cand_t top = heap_pop(heap, &hn);
                if (top.score == -INFINITY) break;
                int i = n++;
                int d = top.depth, r = top.ranks[d - 1];
                o_tok[i] = tk[(d - 1) * K + r];
                o_par[i] = top.parent_node;
                o_dep[i] = d;
                o_rank[i] = r;
                o_sc[i] = top.score;
                memcpy(path[i], top.ranks, sizeof(int) * MAXD);
                for (int w = 0; w < W; ++w)
                    o_mask[(size_t)i * W + w] = o_mask[(size_t)top.parent_node * W + w];
                o_mask[(size_t)i * W + i / 64] |= 1ull << (i % 64);
                /* next sibling: same parent, rank r+1 */
                if (r + 1 < K) {
                    cand_t s = top;
                    s.ranks[d - 1] = r + 1;
                    s.score = o_sc[top.parent_node] + lp[(d - 1) * K + r + 1];
                    heap_push(heap, &hn, &s);
                }
                /* first child: depth d+1, rank 0 */
                if (d < D) {
                    cand_t ch = top;
                    ch.depth = d + 1;
                    ch.ranks[d] = 0;
                    ch.parent_node = i;
                    ch.score = top.score + lp[d * K + 0];
                    heap_push(heap, &hn, &ch);
                }
            }
        }
        n_nodes[b] = n;
        /* first child = smallest index whose parent is i; next sibling = next
         * larger index sharing the parent */
        for (int i = 0; i < n; ++i) {
            for (int j = i + 1; j < n; ++j)
                if (o_par[j] == i) { o_fc[i] = j; break; }
            if (i > 0)
                for (int j = i + 1; j < n; ++j)
                    if (o_par[j] == o_par[i]) { o_ns[i] = j; break; }
        }
    }
    free(heap);
    free(path);
    return 0;
}

/* ------------------------------------------------------------------ */
/* attention                                                           */
/* ------------------------------------------------------------------ */

static double bf16(uint16_t v) {
    uint32_t u = (uint32_t)v << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* One output row (b, node i, head h):
 *   s_j  = scale * (q_lat . c_kv[j] + q_rope . k_rope[j])   for visible j
 *   out  = sum_j softmax(s)_j c_kv[j]       (the 512-wide latent, before w_vc)
 *   lse  = log sum_j exp(s_j)
 * visible j: every prefix row 0..T_b-1, and row T_b+m for each m whose bit is
 * set in the node's ancestor-or-self mask. */
static void attn_row(int Qc, int W, int H, int Tcap, const uint16_t *q_lat,
                     const uint16_t *q_rope, const uint16_t *c_kv, const uint16_t *k_rope,
                     const int32_t *prefix_len, const uint64_t *mask, const int32_t *n_nodes,
                     double scale, int b, int i, int h, double *out, double *lse,
                     double *sbuf) {
    if (i >= n_nodes[b]) {
        for (int c = 0; c < 512; ++c) out[c] = 0.0;
        *lse = -INFINITY;
        return;
    }
    const int T = prefix_len[b];
    const uint16_t *ql = q_lat + (((size_t)b * Qc + i) * H + h) * 512;
    const uint16_t *qr = q_rope + (((size_t)b * Qc + i) * H + h) * 64;
    const uint64_t *mk = mask + ((size_t)b * Qc + i) * W;
    double ql64[512], qr64[64];
    for (int c = 0; c < 512; ++c) ql64[c] = bf16(ql[c]);
    for (int c = 0; c < 64; ++c) qr64[c] = bf16(qr[c]);
    int nvis = 0;
    int *keys = (int *)(sbuf + (T + Qc));
    for (int j = 0; j < T; ++j) keys[nvis++] = j;
    for (int m = 0; m < n_nodes[b]; ++m)
        if ((mk[m / 64] >> (m % 64)) & 1ull) keys[nvis++] = T + m;
    double mx = -INFINITY;
    for (int v = 0; v < nvis; ++v) {
        const uint16_t *kc = c_kv + ((size_t)b * Tcap + keys[v]) * 512;
        const uint16_t *kr = k_rope + ((size_t)b * Tcap + keys[v]) * 64;
        double acc = 0.0;
        for (int c = 0; c < 512; ++c) acc += ql64[c] * bf16(kc[c]);
        for (int c = 0; c < 64; ++c) acc += qr64[c] * bf16(kr[c]);
        sbuf[v] = acc * scale;
        if (sbuf[v] > mx) mx = sbuf[v];
    }
    double l = 0.0;
    for (int v = 0; v < nvis; ++v) {
        sbuf[v] = exp(sbuf[v] - mx);
        l += sbuf[v];
    }
    for (int c = 0; c < 512; ++c) out[c] = 0.0;
    for (int v = 0; v < nvis; ++v) {
        const uint16_t *kc = c_kv + ((size_t)b * Tcap + keys[v]) * 512;
        double p = sbuf[v] / l;
        for (int c = 0; c < 512; ++c) out[c] += p * bf16(kc[c]);
    }
    *lse = mx + log(l);
}

/* rows: n_rows triples (b, i, h); out [n_rows, 512]; lse [n_rows].
 * Returns the number of OpenMP threads used. */
int ddto_attn_rows(int Qc, int W, int H, int Tcap, const uint16_t *q_lat,
                   const uint16_t *q_rope, const uint16_t *c_kv, const uint16_t *k_rope,
                   const int32_t *prefix_len, const uint64_t *mask, const int32_t *n_nodes,
                   double scale, const int32_t *rows, long n_rows, double *out, double *lse,
                   int n_threads) {
    int used = 1;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel
    {
#pragma omp single
        used = omp_get_num_threads();
    }
#endif
    int maxT = 0;
    long nb = 0;
    for (long r = 0; r < n_rows; ++r) if (rows[3 * r] + 1 > nb) nb = rows[3 * r] + 1;
    for (long b = 0; b < nb; ++b) if (prefix_len[b] > maxT) maxT = prefix_len[b];
    size_t sb_doubles = (size_t)(maxT + Qc) * 2 + 16;
#pragma omp parallel
    {
        double *sbuf = (double *)malloc(sizeof(double) * sb_doubles);
#pragma omp for schedule(dynamic, 1)
        for (long r = 0; r < n_rows; ++r)
            attn_row(Qc, W, H, Tcap, q_lat, q_rope, c_kv, k_rope, prefix_len, mask, n_nodes,
                     scale, rows[3 * r], rows[3 * r + 1], rows[3 * r + 2], out + r * 512,
                     lse + r, sbuf);
        free(sbuf);
    }
    return used;
}

/* ------------------------------------------------------------------ */
/* greedy accept                                                       */
/* ------------------------------------------------------------------ */

/* Start at the root; while the target's argmax after the current node equals
 * the token of one of its children, move to that child (lowest index first).
 * accept_idx lists the visited nodes (root first), accept_len their count;
 * commit_tok holds the accepted draft tokens followed by the bonus token (the
 * target's argmax after the last accepted node), which is also next_root. */
int ddto_tree_accept(int B, int D, int Qc, const int32_t *token, const int32_t *parent,
                     const int32_t *n_nodes, const int32_t *target_argmax,
                     int32_t *accept_len, int32_t *accept_idx, int32_t *commit_tok,
                     int32_t *next_root) {
    for (int b = 0; b < B; ++b) {
        const int32_t *tk = token + (size_t)b * Qc, *pa = parent + (size_t)b * Qc;
        const int32_t *tg = target_argmax + (size_t)b * Qc;
        int32_t *ai = accept_idx + (size_t)b * (D + 1), *ct = commit_tok + (size_t)b * (D + 1);
        for (int k = 0; k <= D; ++k) ai[k] = ct[k] = -1;
        int cur = 0, len = 1;
        ai[0] = 0;
        for (;;) {
            int t = tg[cur], nxt = -1;
            for (int j = 1; j < n_nodes[b]; ++j)
                if (pa[j] == cur && tk[j] == t) { nxt = j; break; }
            if (nxt < 0 || len > D) break;
            ct[len - 1] = tk[nxt];
            ai[len++] = nxt;
            cur = nxt;
        }
        ct[len - 1] = tg[cur];
        accept_len[b] = len;
        next_root[b] = tg[cur];
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* KV commit                                                           */
/* ------------------------------------------------------------------ */

/* For each sequence b with T = prefix_len[b] and L = accept_len[b], the
 * accepted path is nodes accept_idx[b][0..L-1] (node 0, the root, first).
 * Node m's keys are rows T + m of c_kv (512 bf16 per row) and k_rope (64 bf16
 * per row). After the commit the path's keys are rows T .. T + L - 1 in path
 * order, rows below T are unchanged, and prefix_len[b] = T + L. A sequence
 * whose values are out of range (L outside [1, D+1], T < 0, T + L > Tcap, a
 * path index not increasing, or a node row at or past Tcap) is left
 * unchanged and flagged BADINPUT in status[b]; others keep their status.
 * Rows are 16-bit words copied as bytes. */
int ddto_kv_commit(int B, int D, int Tcap, const int32_t *accept_len, const int32_t *accept_idx,
                   uint16_t *c_kv, uint16_t *k_rope, int32_t *prefix_len, int32_t *status) {
    uint16_t *tmp_kv = (uint16_t *)malloc(sizeof(uint16_t) * 512 * (size_t)(D + 1));
    uint16_t *tmp_kr = (uint16_t *)malloc(sizeof(uint16_t) * 64 * (size_t)(D + 1));
    if (!tmp_kv || !tmp_kr) {
        free(tmp_kv);
        free(tmp_kr);
        return -1;
    }
    for (int b = 0; b < B; ++b) {
        const int T = prefix_len[b], L = accept_len[b];
        const int32_t *ai = accept_idx + (size_t)b * (D + 1);
        int ok = L >= 1 && L <= D + 1 && T >= 0 && (long long)T + L <= Tcap && ai[0] == 0;
        for (int k = 1; ok && k < L; ++k)
            if (ai[k] <= ai[k - 1] || (long long)T + ai[k] >= Tcap) ok = 0;
        if (!ok) {
            status[b] = ORACLE_BADINPUT;
            continue;
        }
        uint16_t *kv = c_kv + (size_t)b * Tcap * 512, *kr = k_rope + (size_t)b * Tcap * 64;
        /* read every source row before writing any (a later source row can be
         * an earlier destination) */
        for (int k = 0; k < L; ++k) {
            memcpy(tmp_kv + (size_t)k * 512, kv + (size_t)(T + ai[k]) * 512, sizeof(uint16_t) * 512);
            memcpy(tmp_kr + (size_t)k * 64, kr + (size_t)(T + ai[k]) * 64, sizeof(uint16_t) * 64);
        }
        for (int k = 0; k < L; ++k) {
            memcpy(kv + (size_t)(T + k) * 512, tmp_kv + (size_t)k * 512, sizeof(uint16_t) * 512);
            memcpy(kr + (size_t)(T + k) * 64, tmp_kr + (size_t)k * 64, sizeof(uint16_t) * 64);
        }
        prefix_len[b] = T + L;
    }
    free(tmp_kv);
    free(tmp_kr);
    return 0;
}

/* ------------------------------------------------------------------ */
/* temperature sampling over the tree                                  */
/* ------------------------------------------------------------------ */

/* The sampling commit path ("The Architecture of a Thousand-Parameter
 * Decision", "What to Reuse" item 3: temperature sampling from the verified
 * token distribution; "What to Build New" item 2: the sampling-probability
 * path that normalises the target's probabilities over the tree nodes).
 *
 * Row (b, i) of `logits` [B,Qc,V] is the target's logit vector after node i.
 * Its distribution is p_j = exp((x_j - M) / tau) / S with M = max_j x_j and
 * S = sum_j exp((x_j - M) / tau).  With one uniform u = u01[b,i] the node's
 * sample is drawn by inverse transform over token ids in increasing order:
 * the first token j with p_j > 0 whose cumulative probability C_j exceeds u
 * (u < 0 therefore gives the first token of nonzero probability); when no
 * token qualifies (u >= 1, NaN, or rounding at the top) the last token with
 * p_j > 0.  tau <= 0 is the greedy limit: the first index of the largest
 * logit.
 *
 * node_p[b,c] is the probability the parent's row gives node c's own token
 * (the normalised probability tree verification needs); node_p[b,0] = 1, and
 * node slots at or past n_nodes[b] get sample -1 and node_p 0.  In the
 * greedy limit node_p is 1 for the child whose token is the argmax and 0
 * otherwise.
 *
 * A row holding a NaN, or (tau > 0) whose largest logit is not finite, has
 * no distribution: its sample is -1, its children's node_p are 0 and the
 * sequence gets BADINPUT.  A child token outside [0, V) gets node_p 0 and
 * BADINPUT too.  Everything in float64; sums in token order. */
static void sample_row(int V, const float *x, double tau, double u, int *tok_out, double *S_out,
                       double *M_out, int *bad) {
    int has_nan = 0;
    double M = -INFINITY;
    int arg = 0;
    for (int j = 0; j < V; ++j) {
        if (x[j] != x[j]) { has_nan = 1; continue; }
        if ((double)x[j] > M) { M = x[j]; arg = j; }
    }
    *M_out = M;
    *S_out = 0.0;
    if (has_nan || (tau > 0.0 && !isfinite(M))) {
        *bad = 1;
        *tok_out = -1;
        return;
    }
    if (tau <= 0.0) {
        *tok_out = arg;
        return;
    }
    double S = 0.0;
    for (int j = 0; j < V; ++j) S += exp(((double)x[j] - M) / tau);
    *S_out = S;
    const double thr = u * S;
    double C = 0.0;
    int last_pos = -1, pick = -1;
    for (int j = 0; j < V; ++j) {
        const double w = exp(((double)x[j] - M) / tau);
        C += w;
        if (w > 0.0) {
            last_pos = j;
            if (C > thr) { pick = j; break; }
        }
    }
    if (pick < 0) {
        for (int j = V - 1; j >= 0; --j)
            if (exp(((double)x[j] - M) / tau) > 0.0) { last_pos = j; break; }
        pick = last_pos;
    }
    *tok_out = pick;
}

int ddto_tree_sample(int B, int Qc, int V, const float *logits, double tau, const float *u01,
                     const int32_t *token, const int32_t *parent, const int32_t *n_nodes,
                     int32_t *sample_tok, double *node_p, int32_t *status) {
    const long long rows = (long long)B * Qc;
    double *Ss = (double *)malloc(sizeof(double) * (size_t)rows);
    double *Ms = (double *)malloc(sizeof(double) * (size_t)rows);
    int *bad = (int *)calloc((size_t)rows, sizeof(int));
    if (!Ss || !Ms || !bad) {
        free(Ss);
        free(Ms);
        free(bad);
        return -1;
    }
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (long long r = 0; r < rows; ++r) {
        const int b = (int)(r / Qc), i = (int)(r % Qc);
        int n = n_nodes[b];
        n = n < 1 ? 1 : (n > Qc ? Qc : n);
        if (i >= n) {
            sample_tok[r] = -1;
            continue;
        }
        int t;
        sample_row(V, logits + (size_t)r * V, tau, (double)u01[r], &t, &Ss[r], &Ms[r], &bad[r]);
        sample_tok[r] = t;
    }
    for (int b = 0; b < B; ++b) {
        int n = n_nodes[b];
        n = n < 1 ? 1 : (n > Qc ? Qc : n);
        const size_t tb = (size_t)b * Qc;
        int flag = 0;
        for (int i = 0; i < n; ++i) flag |= bad[tb + i];
        node_p[tb] = 1.0;
        for (int c = 1; c < Qc; ++c) {
            if (c >= n) { node_p[tb + c] = 0.0; continue; }
            const int pi = parent[tb + c], tk = token[tb + c];
            const size_t row = tb + (size_t)pi;
            if (tk < 0 || tk >= V) { node_p[tb + c] = 0.0; flag = 1; continue; }
            if (bad[row]) { node_p[tb + c] = 0.0; continue; }
            if (tau <= 0.0)
                node_p[tb + c] = (sample_tok[row] == tk) ? 1.0 : 0.0;
            else
                node_p[tb + c] = exp(((double)logits[row * V + tk] - Ms[row]) / tau) / Ss[row];
        }
        if (flag) status[b] = ORACLE_BADINPUT;
    }
    free(Ss);
    free(Ms);
    free(bad);
    return 0;
}
