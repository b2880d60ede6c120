// Internal launch interfaces between the C-ABI layer (ddt_api.cu) and the
// kernels. Not installed; the public contract is include/ddtree.h.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "ddtree.h"

namespace ddt {

// Bounded-wait limit for every on-chip wait of the attention kernel.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

cudaError_t launch_tree_build(const ddt_draft &in, int budget, const ddt_tree &out,
                              cudaStream_t s);
// With `after_prev` the kernel is launched with programmatic stream
// serialization: it may start before the previous kernel on the stream ends.
// Only the verify step chains its kernels this way (each kernel waits, in
// its code, for the data it needs); standalone calls launch normally.
cudaError_t launch_tree_accept(const ddt_tree &tree, const int32_t *target,
                               const ddt_accept &out, cudaStream_t s, bool after_prev = false);

// The greedy accept walk's inputs and outputs (accept_walk.cuh).
struct AcceptArgs {
    int B, D, Qc;
    const int32_t *token, *parent, *n_nodes, *target;
    int32_t *accept_len, *accept_idx, *commit_tok, *next_root;
};
AcceptArgs accept_args(const ddt_tree &tree, const int32_t *target, const ddt_accept &out);

struct AttnPlan {
    int mtiles;       // 128-row tiles of Qc*H rows per sequence
    int nsplit;       // key-range chunks per (sequence, row tile)
    size_t ws_bytes;  // partial outputs when nsplit > 1
};

// Geometry for one attention call on a device with `sms` multiprocessors.
AttnPlan plan_attention(int B, int Qc, int H, int Tcap, int sms);

// Every host-side check of an attention call (arguments, score scale, an
// sm_103 current device) and, when they pass, the geometry the launch on
// the current device will use (ddt_api.cu).
int check_attn_call(const ddt_attn_in *in, const ddt_tree *tree, float scale, const ddt_attn_out *out,
                    AttnPlan *plan);

// Encodes the tensor maps and enqueues the attention kernel (and the merge
// kernel when nsplit > 1). With `fused_accept`, a merge kernel also runs the
// accept walk in extra blocks of its grid and sets *accepted; without a
// merge nothing is fused and *accepted stays false.
int launch_verify_attn(const ddt_attn_in &in, const ddt_tree &tree, float scale,
                       const ddt_attn_out &out, void *workspace, size_t ws_bytes,
                       const AttnPlan &plan, cudaStream_t s, bool after_prev = false,
                       const int32_t *kv_index = nullptr, int pool_rows = 0, bool out_bf16 = false,
                       const AcceptArgs *fused_accept = nullptr, bool *accepted = nullptr);

// cudaLaunchKernelEx with the programmatic-stream-serialization attribute
// when `after_prev`, a plain launch otherwise.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          bool after_prev, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (after_prev) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

cudaError_t launch_kv_commit(int B, int D, int Tcap, const int32_t *accept_len, const int32_t *accept_idx,
                             void *c_kv, void *k_rope, int32_t *prefix_len, int32_t *status, cudaStream_t s);

// Temperature sampling at every tree node: a persistent grid of clusters of
// C CTAs per row; each CTA owns nreg regions of 128 R tokens (R odd).
constexpr int kSampleMaxRows = 11;      // R: float4 per lane in a region
constexpr int kSampleMaxRegions = 128;  // regions per CTA
constexpr int kSampleListCap = 128;     // rows per cluster and launch
struct SamplePlan {
    int C;        // CTAs per row (cluster size); 0 = shape not supported
    int R;        // float4 per lane in a region (odd)
    int nreg;     // regions per CTA (a multiple of 8)
    size_t smem;  // dynamic shared memory per CTA
};
SamplePlan plan_sample(int V, long long rows, int sms, int max_cluster);
// Largest cluster the sampling kernel may use on the current device (16 or
// 8; 0 if its attributes could not be set). Sets the kernel's attributes on
// the first call.
int sample_max_cluster();
// kd = log2(e) / temperature, or 0 for the greedy limit.
cudaError_t launch_tree_sample(const ddt_tree &tree, const float *logits, int V, double kd, const float *u01,
                               int32_t *sample_tok, float *node_p, const SamplePlan &plan, cudaStream_t s);

cudaError_t launch_selftest_wait(int32_t *status, unsigned timeout_us, cudaStream_t s);

}  // namespace ddt
