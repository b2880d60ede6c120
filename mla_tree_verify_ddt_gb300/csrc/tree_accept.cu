// Greedy follow-the-verified-tree acceptance, one warp per sequence.
//
// Follows "The Architecture of Closure: How a Summary Message Encodes an
// Entire Engineering Session", section "The Table as a Decision Artifact"
// (tree_accept.cu: greedy follow_verified_tree on the GPU, accept lengths
// counted from the root). Starting at the root, the target's argmax after the
// current node is looked up among that node's children; the walk moves to the
// matching child (lowest index when tokens repeat) and stops when none
// matches. The accepted draft tokens plus the target's argmax after the last
// accepted node (the bonus token) are committed; the bonus token is also the
// next step's root.
#include <cuda_runtime.h>

#include <cstdint>

#include "ddt_internal.h"

namespace ddt {
namespace {

constexpr int kWarpsPerBlock = 4;

__global__ void __launch_bounds__(32 * kWarpsPerBlock)
    tree_accept_kernel(int B, int D, int Qc, const int32_t *__restrict__ token,
                       const int32_t *__restrict__ parent, const int32_t *__restrict__ n_nodes,
                       const int32_t *__restrict__ target, int32_t *__restrict__ accept_len,
                       int32_t *__restrict__ accept_idx, int32_t *__restrict__ commit_tok,
                       int32_t *__restrict__ next_root) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * kWarpsPerBlock + warp;
    if (b >= B) return;
    const size_t tb = static_cast<size_t>(b) * Qc;
    int n = n_nodes[b];
    n = n < 1 ? 1 : (n > Qc ? Qc : n);
    // each lane caches the (parent, token) of nodes lane+1, lane+33, lane+65
    // and the target's argmax after nodes lane, lane+32, lane+64, so the walk
    // below never waits on global memory
    int par[3], tok[3], tgt[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const int j = lane + 1 + 32 * k;
        par[k] = (j < n) ? parent[tb + j] : -2;
        tok[k] = (j < n) ? token[tb + j] : 0;
        const int c = lane + 32 * k;
        tgt[k] = (c < n) ? target[tb + c] : 0;
    }
    // the target's argmax after node c (c < n)
    auto target_after = [&](int c) {
        const int v = (c >> 5) == 0 ? tgt[0] : ((c >> 5) == 1 ? tgt[1] : tgt[2]);
        return __shfl_sync(0xffffffffu, v, c & 31);
    };
    int32_t *ai = accept_idx + static_cast<size_t>(b) * (D + 1);
    int32_t *ct = commit_tok + static_cast<size_t>(b) * (D + 1);
    int cur = 0, len = 1;
    int t = target_after(0);
    for (;;) {
        int found = 0x7fffffff;
#pragma unroll
        for (int k = 0; k < 3; ++k)
            if (par[k] == cur && tok[k] == t) found = min(found, lane + 1 + 32 * k);
        found = static_cast<int>(__reduce_min_sync(0xffffffffu, static_cast<unsigned>(found)));
        if (found == 0x7fffffff || len > D) break;
        if (lane == 0) {
            ct[len - 1] = t;  // the accepted child's token equals t
            ai[len] = found;
        }
        ++len;
        cur = found;
        t = target_after(cur);
    }
    for (int k = lane; k <= D; k += 32) {
        if (k == 0) ai[0] = 0;
        else if (k >= len) ai[k] = -1;
        if (k == len - 1) ct[k] = t;
        else if (k >= len) ct[k] = -1;
    }
    if (lane == 0) {
        accept_len[b] = len;
        next_root[b] = t;
    }
    // In a verify step this kernel may run beside the attention's merge
    // (it needs only the tree); it ends after the kernel before it, so that
    // work later on the stream also follows that one.
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

cudaError_t launch_tree_accept(const ddt_tree &tree, const int32_t *target,
                               const ddt_accept &out, cudaStream_t s, bool after_prev) {
    const int blocks = (tree.B + kWarpsPerBlock - 1) / kWarpsPerBlock;
    return launch_kernel(tree_accept_kernel, dim3(blocks), dim3(32 * kWarpsPerBlock), 0, s, after_prev, tree.B,
                         tree.D, tree.Qc, static_cast<const int32_t *>(tree.token),
                         static_cast<const int32_t *>(tree.parent), static_cast<const int32_t *>(tree.n_nodes),
                         target, out.accept_len, out.accept_idx, out.commit_tok, out.next_root);
}

}  // namespace ddt
