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
// entries; each lane owns three slots and the warp finds the minimum with
// shuffles. The rank path is packed into 64 bits, four per level, level 1 in
// the top nibble, so two paths of equal depth compare as integers.
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

// Sort key: smaller is selected first.
struct Key {
    uint64_t hi;  // inverted ordered score (32) | depth (32)
    uint64_t lo;  // rank path
};

__device__ __forceinline__ uint32_t ordered_desc(float s) {
    s = s + 0.0f;  // -0 -> +0 so equal scores share one key
    uint32_t u = __float_as_uint(s);
    uint32_t asc = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ~asc;  // larger score -> smaller key
}

__device__ __forceinline__ bool key_less(const Key &a, const Key &b) {
    return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo);
}

struct WarpSmem {
    // the sequence's drafter rows, staged once so that the pops, which form
    // one dependent chain, never wait on global memory
    float d_lp[kMaxDK];
    int d_tok[kMaxDK];
    // frontier, slot = lane * kFrontierSlots + k
    float f_score[32 * kFrontierSlots];
    uint64_t f_path[32 * kFrontierSlots];
    int f_depth[32 * kFrontierSlots];
    int f_parent[32 * kFrontierSlots];
    int f_valid[32 * kFrontierSlots];
    // nodes
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
    bad = __any_sync(0xffffffffu, bad);

    for (int k = 0; k < kFrontierSlots; ++k) sm.f_valid[lane * kFrontierSlots + k] = 0;
    if (lane == 0) {
        sm.n_score[0] = 0.0f;
        sm.n_parent[0] = -1;
        sm.n_depth[0] = 0;
        sm.n_rank[0] = -1;
        sm.n_token[0] = root;
        sm.n_mask[0][0] = 1ull;
        sm.n_mask[0][1] = 0ull;
        // the only initial candidate: depth 1, rank 0
        sm.f_valid[0] = 1;
        sm.f_score[0] = __fadd_rn(0.0f, sm.d_lp[0]);
        sm.f_path[0] = 0ull;
        sm.f_depth[0] = 1;
        sm.f_parent[0] = 0;
    }
    __syncwarp();

    int n = 1;
    if (!bad) {
        while (n < budget + 1) {
            // warp arg-min over the frontier
            Key best{~0ull, ~0ull};
            int best_slot = -1;
            for (int k = 0; k < kFrontierSlots; ++k) {
                const int slot = lane * kFrontierSlots + k;
                if (!sm.f_valid[slot]) continue;
                Key c{(static_cast<uint64_t>(ordered_desc(sm.f_score[slot])) << 32) |
                          static_cast<uint32_t>(sm.f_depth[slot]),
                      sm.f_path[slot]};
                if (best_slot < 0 || key_less(c, best)) {
                    best = c;
                    best_slot = slot;
                }
            }
            for (int off = 16; off > 0; off >>= 1) {
                Key o{__shfl_xor_sync(0xffffffffu, best.hi, off),
                      __shfl_xor_sync(0xffffffffu, best.lo, off)};
                int os = __shfl_xor_sync(0xffffffffu, best_slot, off);
                if (os >= 0 && (best_slot < 0 || key_less(o, best) ||
                                (o.hi == best.hi && o.lo == best.lo && os < best_slot))) {
                    best = o;
                    best_slot = os;
                }
            }
            if (best_slot < 0) break;  // frontier empty
            const float s = sm.f_score[best_slot];
            if (s == -INFINITY) break;  // everything left is -inf
            const int d = sm.f_depth[best_slot];
            const uint64_t path = sm.f_path[best_slot];
            const int pnode = sm.f_parent[best_slot];
            const int shift = 4 * (16 - d);
            const int r = static_cast<int>((path >> shift) & 15ull);
            const bool has_sibling = r + 1 < K;
            const bool has_child = d < D;
            // the popped slot becomes the next sibling (same parent, rank r+1);
            // the first child (depth d+1, rank 0) takes the popped slot when
            // there is no sibling, else the lowest free slot, found by the warp
            int child_slot = best_slot;
            if (has_child && has_sibling) {
                int mine = 0x7fffffff;
                for (int k = 0; k < kFrontierSlots; ++k)
                    if (!sm.f_valid[lane * kFrontierSlots + k]) {
                        mine = lane * kFrontierSlots + k;
                        break;
                    }
                for (int off = 16; off > 0; off >>= 1) mine = min(mine, __shfl_xor_sync(0xffffffffu, mine, off));
                child_slot = mine;  // exists: at most budget+1 <= 65 live entries
            }
            __syncwarp();
            if (lane == 0) {
                const int i = n;
                sm.n_score[i] = s;
                sm.n_parent[i] = pnode;
                sm.n_depth[i] = d;
                sm.n_rank[i] = r;
                sm.n_token[i] = sm.d_tok[(d - 1) * K + r];
                sm.n_mask[i][0] = sm.n_mask[pnode][0];
                sm.n_mask[i][1] = sm.n_mask[pnode][1];
                sm.n_mask[i][i >> 6] |= 1ull << (i & 63);
                if (has_sibling) {
                    sm.f_score[best_slot] = __fadd_rn(sm.n_score[pnode], sm.d_lp[(d - 1) * K + r + 1]);
                    sm.f_path[best_slot] = path + (1ull << shift);
                } else if (!has_child) {
                    sm.f_valid[best_slot] = 0;
                }
                if (has_child) {
                    sm.f_valid[child_slot] = 1;
                    sm.f_score[child_slot] = __fadd_rn(s, sm.d_lp[d * K + 0]);
                    sm.f_path[child_slot] = path;
                    sm.f_depth[child_slot] = d + 1;
                    sm.f_parent[child_slot] = i;
                }
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
