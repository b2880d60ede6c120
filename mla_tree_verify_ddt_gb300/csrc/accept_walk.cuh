// Greedy follow-the-verified-tree walk of one sequence by one warp: shared by
// the standalone accept kernel and the key-range merge kernel, which runs it
// in extra blocks of its own grid inside a verify step.
//
// Follows "The Architecture of Closure: How a Summary Message Encodes an
// Entire Engineering Session", section "The Table as a Decision Artifact"
// (greedy follow_verified_tree on the GPU, accept lengths counted from the
// root). Starting at the root, the target's argmax after the current node is
// looked up among that node's children; the walk moves to the matching child
// (lowest index when tokens repeat) and stops when none matches. The accepted
// draft tokens plus the target's argmax after the last accepted node (the
// bonus token) are committed; the bonus token is also the next step's root.
#pragma once
#include <cstdint>

#include "ddt_internal.h"

namespace ddt {

__device__ __forceinline__ void accept_walk(const AcceptArgs &a, int b, int lane) {
    const size_t tb = static_cast<size_t>(b) * a.Qc;
    int n = a.n_nodes[b];
    n = n < 1 ? 1 : (n > a.Qc ? a.Qc : n);
    // each lane caches the (parent, token) of nodes lane+1, lane+33, lane+65
    // and the target's argmax after nodes lane, lane+32, lane+64, so the walk
    // below never waits on global memory
    int par[3], tok[3], tgt[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const int j = lane + 1 + 32 * k;
        par[k] = (j < n) ? a.parent[tb + j] : -2;
        tok[k] = (j < n) ? a.token[tb + j] : 0;
        const int c = lane + 32 * k;
        tgt[k] = (c < n) ? a.target[tb + c] : 0;
    }
    // the target's argmax after node c (c < n)
    auto target_after = [&](int c) {
        const int v = (c >> 5) == 0 ? tgt[0] : ((c >> 5) == 1 ? tgt[1] : tgt[2]);
        return __shfl_sync(0xffffffffu, v, c & 31);
    };
    const int D = a.D;
    int32_t *ai = a.accept_idx + static_cast<size_t>(b) * (D + 1);
    int32_t *ct = a.commit_tok + static_cast<size_t>(b) * (D + 1);
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
        a.accept_len[b] = len;
        a.next_root[b] = t;
    }
}

}  // namespace ddt
