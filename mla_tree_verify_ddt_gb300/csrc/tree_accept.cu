// Greedy follow-the-verified-tree acceptance, one warp per sequence (the walk
// itself is accept_walk.cuh; inside a verify step whose keys are split, the
// merge kernel runs the same walk instead of this kernel).
#include <cuda_runtime.h>

#include <cstdint>

#include "accept_walk.cuh"
#include "ddt_internal.h"

namespace ddt {
namespace {

constexpr int kWarpsPerBlock = 4;

__global__ void __launch_bounds__(32 * kWarpsPerBlock) tree_accept_kernel(const AcceptArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * kWarpsPerBlock + warp;
    if (b < a.B) accept_walk(a, b, lane);
    // In a verify step this kernel may run beside the attention's merge
    // (it needs only the tree); it ends after the kernel before it, so that
    // work later on the stream also follows that one.
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

AcceptArgs accept_args(const ddt_tree &tree, const int32_t *target, const ddt_accept &out) {
    AcceptArgs a{};
    a.B = tree.B;
    a.D = tree.D;
    a.Qc = tree.Qc;
    a.token = tree.token;
    a.parent = tree.parent;
    a.n_nodes = tree.n_nodes;
    a.target = target;
    a.accept_len = out.accept_len;
    a.accept_idx = out.accept_idx;
    a.commit_tok = out.commit_tok;
    a.next_root = out.next_root;
    return a;
}

cudaError_t launch_tree_accept(const ddt_tree &tree, const int32_t *target,
                               const ddt_accept &out, cudaStream_t s, bool after_prev) {
    const int blocks = (tree.B + kWarpsPerBlock - 1) / kWarpsPerBlock;
    return launch_kernel(tree_accept_kernel, dim3(blocks), dim3(32 * kWarpsPerBlock), 0, s, after_prev,
                         accept_args(tree, target, out));
}

}  // namespace ddt
