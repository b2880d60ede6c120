// GPU draft-tree builder: best-first top-budget expansion of the drafter's
// per-depth top-K, one warp per sequence, no host round-trip.
//
// Follows "The Architecture of a Thousand-Parameter Decision: Designing a
// Native DDTree Inference Engine for Kimi K2.6", section "What to Build New",
// item 3 (a warp-block-per-request best-first top-k expansion emitting parent
// indices, a visibility mask and first-child/next-sibling pointers, replacing
// the per-request CPU heapq and its host syncs).
//
// A candidate is a rank path (r_1..r_d). Its score is the float32 sum, root to
// leaf, of lp[b, l-1, r_l]. Candidates are taken in the total order
//   score descending, depth ascending, rank path lexicographic ascending,
// which the frontier realises exactly: a node's first child and next sibling
// both come after it in that order, so popping the frontier minimum each step
// yields the global order. The frontier never holds more than budget+1
// entries. It lives in registers, three slots per lane; a pop is one warp
// min-reduction of the 32-bit score key (redux.sync), with depth and rank
// path consulted only when scores tie. The rank path is packed into 64 bits,
// four per level, level 1 in the top nibble, so two paths of equal depth
// compare as integers.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "ddt_internal.h"

namespace ddt {
namespace {

constexpr int kFrontierSlots = 3;  // per lane: 96 >= budget + 1
constexpr int kWarpsPerBlock = 4;
constexpr int kMaxQc = DDT_MAX_BUDGET + 1;
constexpr int kMaxDK = DDT_MAX_DEPTH * DDT_MAX_TOPK;
constexpr uint32_t kNoKey = 0xffffffffu;  // above every score key, -inf included
constexpr unsigned kAll = 0xffffffffu;

// Order-preserving map of a score to a key where the larger score gets the
// smaller key (-0 and +0 share one key).
__device__ __forceinline__ uint32_t score_key(float s) {
    s = s + 0.0f;
    const uint32_t u = __float_as_uint(s);
    const uint32_t asc = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ~asc;
}

// One frontier slot. Unused slots have key == kNoKey.
struct Slot {
    uint32_t key;     // score_key(score)
    float score;
    float pscore;     // the parent's score (for the next sibling's score)
    int depth;
    int parent;       // node index of the parent
    uint64_t path;
};

__device__ __forceinline__ bool slot_less(const Slot &a, const Slot &b) {
    if (a.key != b.key) return a.key < b.key;
    if (a.depth != b.depth) return a.depth < b.depth;
    return a.path < b.path;
}

struct WarpSmem {
    // the sequence's drafter rows, staged once so that the pops, which form
    // one dependent chain, never wait on global memory
    float d_lp[kMaxDK];
    int d_tok[kMaxDK];
    // nodes in pop order
    float n_score[kMaxQc];
    int n_parent[kMaxQc];
    int n_depth[kMaxQc];
    int n_rank[kMaxQc];
    int n_token[kMaxQc];
    uint64_t n_mask[kMaxQc][2];
};

__global__ void __launch_bounds__(32 * kWarpsPerBlock)
    tree_build_kernel(int B, int D, int K, int vocab, const int32_t *__restrict__ draft_tok,
                      const float *__restrict__ draft_lp, const int32_t *__restrict__ root_tok,
                      int budget, int Qc, int W, int32_t *__restrict__ o_token,
                      int32_t *__restrict__ o_parent, int32_t *__restrict__ o_depth,
                      int32_t *__restrict__ o_rank, float *__restrict__ o_score,
                      int32_t *__restrict__ o_first_child, int32_t *__restrict__ o_next_sibling,
                      uint64_t *__restrict__ o_mask, int32_t *__restrict__ o_n_nodes,
                      int32_t *__restrict__ o_status) {
    __shared__ WarpSmem sm_all[kWarpsPerBlock];
    // the attention kernel of a verify step may start at once: it streams
    // the prefix before it needs the tree
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * kWarpsPerBlock + warp;
    if (b >= B) return;
    WarpSmem &sm = sm_all[warp];
    const int32_t *tok = draft_tok + static_cast<size_t>(b) * D * K;
    const float *lp = draft_lp + static_cast<size_t>(b) * D * K;

    // ---- validate the drafter rows (finite or -inf, <= 0, non-increasing,
    // tokens in range) and the root token
    bool bad = false;
    for (int e = lane; e < D * K; e += 32) {
        const float v = lp[e];
        const int t = tok[e];
        sm.d_lp[e] = v;
        sm.d_tok[e] = t;
        if (isnan(v) || v > 0.0f) bad = true;
        if (t < 0 || t >= vocab) bad = true;
    }
    const int32_t root = root_tok[b];
    if (root < 0 || root >= vocab) bad = true;
    __syncwarp();
    for (int e = lane; e < D * K; e += 32)
        if ((e % K) > 0 && sm.d_lp[e] > sm.d_lp[e - 1]) bad = true;
    bad = __any_sync(kAll, bad);

    if (lane == 0) {
        sm.n_score[0] = 0.0f;
        sm.n_parent[0] = -1;
        sm.n_depth[0] = 0;
        sm.n_rank[0] = -1;
        sm.n_token[0] = root;
        sm.n_mask[0][0] = 1ull;
        sm.n_mask[0][1] = 0ull;
    }
    Slot f[kFrontierSlots];
#pragma unroll
    for (int k = 0; k < kFrontierSlots; ++k) f[k] = Slot{kNoKey, 0.0f, 0.0f, 0, 0, 0ull};
    if (lane == 0) {
        // the only initial candidate: depth 1, rank 0
        const float s0 = __fadd_rn(0.0f, sm.d_lp[0]);
        f[0] = Slot{score_key(s0), s0, 0.0f, 1, 0, 0ull};
    }
    __syncwarp();

    int n = 1;
    if (!bad) {
        while (n < budget + 1) {
            // ---- this lane's best slot
            int ls = 0;
            Slot mine = f[0];
#pragma unroll
            for (int k = 1; k < kFrontierSlots; ++k)
                if (slot_less(f[k], mine)) {
                    mine = f[k];
                    ls = k;
                }
            // ---- the warp's best: score key first, depth and path on ties
            const uint32_t mkey = __reduce_min_sync(kAll, mine.key);
            if (mkey == kNoKey) break;  // frontier empty
            if (mkey == score_key(-INFINITY)) break;  // everything left is -inf
            unsigned tied = __ballot_sync(kAll, mine.key == mkey);
            if (__popc(tied) > 1) {
                const bool in1 = mine.key == mkey;
                const uint32_t md = __reduce_min_sync(kAll, in1 ? static_cast<uint32_t>(mine.depth) : kNoKey);
                const bool in2 = in1 && static_cast<uint32_t>(mine.depth) == md;
                tied = __ballot_sync(kAll, in2);
                if (__popc(tied) > 1) {
                    const uint32_t ph = static_cast<uint32_t>(mine.path >> 32);
                    const uint32_t mh = __reduce_min_sync(kAll, in2 ? ph : kNoKey);
                    const bool in3 = in2 && ph == mh;
                    tied = __ballot_sync(kAll, in3);
                    if (__popc(tied) > 1) {
                        const uint32_t pl = static_cast<uint32_t>(mine.path);
                        const uint32_t ml = __reduce_min_sync(kAll, in3 ? pl : kNoKey);
                        tied = __ballot_sync(kAll, in3 && pl == ml);  // paths are unique
                    }
                }
            }
            const int win = __ffs(tied) - 1;
            // ---- the popped candidate, to every lane
            const float s = __shfl_sync(kAll, mine.score, win);
            const int d = __shfl_sync(kAll, mine.depth, win);
            const uint64_t path = (static_cast<uint64_t>(__shfl_sync(kAll, static_cast<uint32_t>(mine.path >> 32), win))
                                   << 32) |
                                  __shfl_sync(kAll, static_cast<uint32_t>(mine.path), win);
            const int shift = 4 * (16 - d);
            const int r = static_cast<int>((path >> shift) & 15ull);
            const bool has_sibling = r + 1 < K;
            const bool has_child = d < D;
            const int i = n;  // the new node's index
            // the first child goes to the popped slot when there is no
            // sibling, else to the lowest free slot of the lowest lane with one
            int free_k = -1;
#pragma unroll
            for (int k = kFrontierSlots - 1; k >= 0; --k)
                if (f[k].key == kNoKey) free_k = k;
            const unsigned has_free = __ballot_sync(kAll, free_k >= 0);
            const int child_lane = has_sibling ? __ffs(has_free) - 1 : win;
            if (lane == win) {
                const int pnode = mine.parent;
                sm.n_score[i] = s;
                sm.n_parent[i] = pnode;
                sm.n_depth[i] = d;
                sm.n_rank[i] = r;
                sm.n_token[i] = sm.d_tok[(d - 1) * K + r];
                uint64_t m0 = sm.n_mask[pnode][0], m1 = sm.n_mask[pnode][1];
                if (i < 64) m0 |= 1ull << i;
                else m1 |= 1ull << (i - 64);
                sm.n_mask[i][0] = m0;
                sm.n_mask[i][1] = m1;
                // the popped slot becomes the next sibling (same parent, rank r+1)
#pragma unroll
                for (int k = 0; k < kFrontierSlots; ++k) {
                    if (k != ls) continue;
                    if (has_sibling) {
                        f[k].score = __fadd_rn(mine.pscore, sm.d_lp[(d - 1) * K + r + 1]);
                        f[k].key = score_key(f[k].score);
                        f[k].path = path + (1ull << shift);
                    } else {
                        f[k].key = kNoKey;
                    }
                }
            }
            if (has_child && lane == child_lane) {
                const int k_child = has_sibling ? free_k : ls;
                const float cs = __fadd_rn(s, sm.d_lp[d * K + 0]);
#pragma unroll
                for (int k = 0; k < kFrontierSlots; ++k)
                    if (k == k_child) f[k] = Slot{score_key(cs), cs, s, d + 1, i, path};
            }
            ++n;
            __syncwarp();
        }
    }
    __syncwarp();

    // ---- outputs
    const size_t base = static_cast<size_t>(b) * Qc;
    for (int i = lane; i < Qc; i += 32) {
        if (i < n) {
            int fc = -1, ns = -1;
            for (int j = i + 1; j < n; ++j)
                if (sm.n_parent[j] == i) {
                    fc = j;
                    break;
                }
            if (i > 0)
                for (int j = i + 1; j < n; ++j)
                    if (sm.n_parent[j] == sm.n_parent[i]) {
                        ns = j;
                        break;
                    }
            o_token[base + i] = sm.n_token[i];
            o_parent[base + i] = sm.n_parent[i];
            o_depth[base + i] = sm.n_depth[i];
            o_rank[base + i] = sm.n_rank[i];
            o_score[base + i] = sm.n_score[i];
            o_first_child[base + i] = fc;
            o_next_sibling[base + i] = ns;
            for (int w = 0; w < W; ++w) o_mask[(base + i) * W + w] = sm.n_mask[i][w];
        } else {
            o_token[base + i] = -1;
            o_parent[base + i] = -1;
            o_depth[base + i] = -1;
            o_rank[base + i] = -1;
            o_score[base + i] = -INFINITY;
            o_first_child[base + i] = -1;
            o_next_sibling[base + i] = -1;
            for (int w = 0; w < W; ++w) o_mask[(base + i) * W + w] = 0ull;
        }
    }
    if (lane == 0) {
        o_n_nodes[b] = n;
        o_status[b] = bad ? DDT_E_BADINPUT : DDT_OK;
    }
}

}  // namespace

cudaError_t launch_tree_build(const ddt_draft &in, int budget, const ddt_tree &out,
                              cudaStream_t s) {
    const int blocks = (in.B + kWarpsPerBlock - 1) / kWarpsPerBlock;
    tree_build_kernel<<<blocks, 32 * kWarpsPerBlock, 0, s>>>(
        in.B, in.D, in.K, in.vocab, in.tok, in.lp, in.root_tok, budget, out.Qc, out.W, out.token,
        out.parent, out.depth, out.rank, out.score, out.first_child, out.next_sibling, out.mask,
        out.n_nodes, out.status);
    return cudaGetLastError();
}

}  // namespace ddt
