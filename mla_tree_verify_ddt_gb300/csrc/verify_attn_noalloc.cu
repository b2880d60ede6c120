// ddt_verify_mla_attn_noalloc: the tree-verify attention for callers that
// cannot allocate device memory.
//
// ddt_verify_mla_attn needs a caller-provided workspace whenever it splits a
// sequence's key range over several CTAs (it then writes per-range partial
// outputs and merges them). Some callers have no way to provide one: a
// serving engine that reserves nearly all HBM for its KV cache at start-up
// and runs its decode loop with no allocator to hand out more; a plugin or
// C host that receives only the input and output buffers; code that must
// not call cudaMalloc because it synchronises the device. This entry point
// gives them the same computation with the partials kept in a fixed scratch
// array that the library itself defines.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "ddt_internal.h"
#include "ddtree.h"

namespace {

// The scratch: one file-scope device array. Every GPU that loads the library
// holds DDT_NOALLOC_SCRATCH_BYTES of it until the process exits.
__device__ __align__(256) unsigned char g_noalloc_scratch[DDT_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu[kMaxDevices];
void *g_scratch_ptr[kMaxDevices];  // the array's device address on device d, once looked up

// In host code the array's name only stands in for the device object; its
// device address comes from cudaGetSymbolAddress with that device current.
// Only a successful lookup is kept, so a failed one (a transient error) is
// retried by the next call. The lookup may load the module, which a stream
// capture in progress would not allow: a first call on a device made while
// `s` is capturing is refused with DDT_E_INVAL instead.
int scratch_address(int dev, cudaStream_t s, void **out) {
    std::lock_guard<std::mutex> lock(g_scratch_mu[dev]);
    if (!g_scratch_ptr[dev]) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return DDT_E_CUDA;
        if (cs != cudaStreamCaptureStatusNone) return DDT_E_INVAL;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            (void)cudaGetLastError();  // not sticky: leave no error behind for the caller
            return DDT_E_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return DDT_OK;
}

}  // namespace

extern "C" int ddt_verify_mla_attn_noalloc(const ddt_attn_in *in, const ddt_tree *tree, float scale,
                                           ddt_attn_out *out, void *stream) {
    // every argument and device check first, then the exact geometry the
    // launch below uses: its partials must fit the scratch
    ddt::AttnPlan plan{};
    if (int rc = ddt::check_attn_call(in, tree, scale, out, &plan)) return rc;
    if (plan.ws_bytes > DDT_NOALLOC_SCRATCH_BYTES) return DDT_E_SCRATCH_LIMIT;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DDT_E_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *scratch = nullptr;
    if (plan.ws_bytes > 0) {
        if (int rc = scratch_address(dev, s, &scratch)) return rc;
    }
    return ddt::launch_verify_attn(*in, *tree, scale, *out, scratch, DDT_NOALLOC_SCRATCH_BYTES, plan, s);
}
