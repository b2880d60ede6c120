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

#include "ddtree.h"

namespace {

// The scratch: one file-scope device array. Every GPU that loads the library
// holds DDT_NOALLOC_SCRATCH_BYTES of it until the process exits.
__device__ __align__(256) unsigned char g_noalloc_scratch[DDT_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];
cudaError_t g_scratch_err[kMaxDevices];
std::once_flag g_scratch_once[kMaxDevices];

}  // namespace

extern "C" int ddt_verify_mla_attn_noalloc(const ddt_attn_in *in, const ddt_tree *tree, float scale,
                                           ddt_attn_out *out, void *stream) {
    if (!in || !tree || !out) return DDT_E_INVAL;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DDT_E_CUDA;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return DDT_E_CUDA;
    if (major * 10 + minor != 103) return DDT_E_UNSUPPORTED;
    // the scratch this shape needs on this device (0 when the key range is
    // not split, or when the shape is invalid: the call below rejects those)
    const size_t need = ddt_workspace_size(tree->B, tree->D, 1, tree->Qc - 1, in->H, in->Tcap);
    if (need > DDT_NOALLOC_SCRATCH_BYTES) return DDT_E_SCRATCH_LIMIT;
    // In host code the array's name only stands in for the device object; its
    // device address comes from cudaGetSymbolAddress, taken once per device
    // with that device current (the first call on a device does this).
    std::call_once(g_scratch_once[dev], [dev] {
        g_scratch_err[dev] = cudaGetSymbolAddress(&g_scratch_ptr[dev], g_noalloc_scratch);
    });
    if (g_scratch_err[dev] != cudaSuccess || !g_scratch_ptr[dev]) return DDT_E_CUDA;
    return ddt_verify_mla_attn(in, tree, scale, out, g_scratch_ptr[dev], DDT_NOALLOC_SCRATCH_BYTES,
                               stream);
}
