// C-ABI entry points of libddtree: host-side argument checks, launch
// geometry, and enqueueing of the device kernels. Nothing here synchronises
// the device except ddt_read_device_status.
#include <cuda_runtime.h>

#include <cfloat>
#include <cmath>
#include <cstdint>

#include "ddt_internal.h"
#include "ddtree.h"

namespace {

constexpr int kMaxDevices = 64;

struct DevInfo {
    int sms = 0;
    int cc = 0;  // major*10 + minor
};

// Per-device facts, read once (attribute queries are not stream work, so
// they are harmless inside a capture, but the first call should still come
// before capture).
const DevInfo *device_info() {
    static DevInfo info[kMaxDevices];
    static int ready[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    if (!__atomic_load_n(&ready[dev], __ATOMIC_ACQUIRE)) {
        DevInfo d;
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return nullptr;
        d.cc = major * 10 + minor;
        info[dev] = d;
        __atomic_store_n(&ready[dev], 1, __ATOMIC_RELEASE);
    }
    return &info[dev];
}

int check_device() {
    const DevInfo *d = device_info();
    if (!d) return DDT_E_CUDA;
    return d->cc == 103 ? DDT_OK : DDT_E_UNSUPPORTED;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_tree_shape(const ddt_tree *t, int budget) {
    if (!t) return DDT_E_INVAL;
    if (t->B < 1 || t->D < 1 || t->D > DDT_MAX_DEPTH) return DDT_E_INVAL;
    if (budget < 1 || budget > DDT_MAX_BUDGET || t->Qc != budget + 1) return DDT_E_INVAL;
    if (t->W != (t->Qc + 63) / 64) return DDT_E_INVAL;
    return DDT_OK;
}

int check_tree_ptrs(const ddt_tree *t) {
    if (!t->token || !t->parent || !t->depth || !t->rank || !t->score || !t->first_child ||
        !t->next_sibling || !t->mask || !t->n_nodes || !t->status)
        return DDT_E_INVAL;
    return DDT_OK;
}

int check_draft(const ddt_draft *in, const ddt_tree *out, int budget) {
    if (!in || !in->tok || !in->lp || !in->root_tok) return DDT_E_INVAL;
    if (in->B < 1 || in->D < 1 || in->D > DDT_MAX_DEPTH || in->K < 1 || in->K > DDT_MAX_TOPK ||
        in->vocab < 1)
        return DDT_E_INVAL;
    if (int rc = check_tree_shape(out, budget)) return rc;
    if (out->B != in->B || out->D != in->D) return DDT_E_INVAL;
    return check_tree_ptrs(out);
}

int check_attn(const ddt_attn_in *in, const ddt_tree *tree, const ddt_attn_out *out) {
    if (!in || !tree || !out || !out->out || !out->lse) return DDT_E_INVAL;
    if (!in->q_lat || !in->q_rope || !in->c_kv || !in->k_rope || !in->prefix_len) return DDT_E_INVAL;
    if (!tree->mask || !tree->n_nodes || !tree->status) return DDT_E_INVAL;
    if (tree->B < 1 || tree->Qc < 1 || tree->Qc > DDT_MAX_BUDGET + 1 || tree->W != (tree->Qc + 63) / 64)
        return DDT_E_INVAL;
    if (in->H < 1 || in->Tcap < 1) return DDT_E_INVAL;
    const long long rows = static_cast<long long>(tree->B) * tree->Qc * in->H;
    const long long kv_rows = static_cast<long long>(tree->B) * in->Tcap;
    if (rows >= (1LL << 31) || kv_rows >= (1LL << 31) || tree->B > 65535) return DDT_E_INVAL;
    if (!aligned16(in->q_lat) || !aligned16(in->q_rope) || !aligned16(in->c_kv) || !aligned16(in->k_rope) ||
        !aligned16(out->out))
        return DDT_E_INVAL;
    return DDT_OK;
}

int check_accept(const ddt_tree *tree, const int32_t *target, const ddt_accept *out) {
    if (!tree || !target || !out) return DDT_E_INVAL;
    if (!out->accept_len || !out->accept_idx || !out->commit_tok || !out->next_root) return DDT_E_INVAL;
    if (!tree->token || !tree->parent || !tree->n_nodes) return DDT_E_INVAL;
    if (tree->B < 1 || tree->D < 1 || tree->D > DDT_MAX_DEPTH || tree->Qc < 1 ||
        tree->Qc > DDT_MAX_BUDGET + 1)
        return DDT_E_INVAL;
    return DDT_OK;
}

// The attention's score scale: positive and finite (the kernel applies it
// after taking the maximum of the raw scores, which needs scale > 0).
int check_scale(float scale) { return (scale > 0.f && scale <= FLT_MAX) ? DDT_OK : DDT_E_INVAL; }

}  // namespace

namespace ddt {
int check_attn_call(const ddt_attn_in *in, const ddt_tree *tree, float scale, const ddt_attn_out *out,
                    AttnPlan *plan) {
    if (int rc = check_attn(in, tree, out)) return rc;
    if (int rc = check_scale(scale)) return rc;
    if (int rc = check_device()) return rc;
    *plan = plan_attention(tree->B, tree->Qc, in->H, in->Tcap, device_info()->sms);
    return DDT_OK;
}
}  // namespace ddt

extern "C" {

size_t ddt_workspace_size(int B, int D, int K, int budget, int H, int Tcap) {
    (void)D;
    (void)K;
    if (B < 1 || budget < 1 || budget > DDT_MAX_BUDGET || H < 1 || Tcap < 1) return 0;
    const DevInfo *d = device_info();
    if (!d) return 0;
    return ddt::plan_attention(B, budget + 1, H, Tcap, d->sms).ws_bytes;
}

int ddt_tree_build(const ddt_draft *in, int budget, ddt_tree *out, void *stream) {
    if (int rc = check_draft(in, out, budget)) return rc;
    if (int rc = check_device()) return rc;
    return ddt::launch_tree_build(*in, budget, *out, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? DDT_OK
               : DDT_E_CUDA;
}

int ddt_verify_mla_attn(const ddt_attn_in *in, const ddt_tree *tree, float scale, ddt_attn_out *out,
                        void *workspace, size_t ws_bytes, void *stream) {
    if (int rc = check_attn(in, tree, out)) return rc;
    if (int rc = check_scale(scale)) return rc;
    if (int rc = check_device()) return rc;
    const ddt::AttnPlan plan = ddt::plan_attention(tree->B, tree->Qc, in->H, in->Tcap, device_info()->sms);
    if (plan.ws_bytes > ws_bytes || (plan.ws_bytes && !workspace)) return DDT_E_INVAL;
    return ddt::launch_verify_attn(*in, *tree, scale, *out, workspace, ws_bytes, plan,
                                   static_cast<cudaStream_t>(stream));
}

int ddt_verify_mla_attn_bf16(const ddt_attn_in *in, const ddt_tree *tree, float scale, uint16_t *out_bf16,
                             float *lse, void *workspace, size_t ws_bytes, void *stream) {
    // (the float32 output slot carries the bfloat16 buffer; check_attn tests
    // its pointer and alignment)
    ddt_attn_out out{reinterpret_cast<float *>(out_bf16), lse};
    if (int rc = check_attn(in, tree, &out)) return rc;
    if (int rc = check_scale(scale)) return rc;
    if (int rc = check_device()) return rc;
    const ddt::AttnPlan plan = ddt::plan_attention(tree->B, tree->Qc, in->H, in->Tcap, device_info()->sms);
    if (plan.ws_bytes > ws_bytes || (plan.ws_bytes && !workspace)) return DDT_E_INVAL;
    return ddt::launch_verify_attn(*in, *tree, scale, out, workspace, ws_bytes, plan,
                                   static_cast<cudaStream_t>(stream), false, nullptr, 0, true);
}

int ddt_verify_mla_attn_paged(const ddt_attn_in *in, const ddt_tree *tree, float scale, ddt_attn_out *out,
                              void *workspace, size_t ws_bytes, const int32_t *kv_index, int pool_rows,
                              void *stream) {
    if (!kv_index || pool_rows < 1) return DDT_E_INVAL;
    if (int rc = check_attn(in, tree, out)) return rc;
    if (int rc = check_scale(scale)) return rc;
    if (int rc = check_device()) return rc;
    const ddt::AttnPlan plan = ddt::plan_attention(tree->B, tree->Qc, in->H, in->Tcap, device_info()->sms);
    if (plan.ws_bytes > ws_bytes || (plan.ws_bytes && !workspace)) return DDT_E_INVAL;
    return ddt::launch_verify_attn(*in, *tree, scale, *out, workspace, ws_bytes, plan,
                                   static_cast<cudaStream_t>(stream), false, kv_index, pool_rows);
}

int ddt_tree_accept(const ddt_tree *tree, const int32_t *target_argmax, ddt_accept *out, void *stream) {
    if (int rc = check_accept(tree, target_argmax, out)) return rc;
    if (int rc = check_device()) return rc;
    return ddt::launch_tree_accept(*tree, target_argmax, *out, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? DDT_OK
               : DDT_E_CUDA;
}

int ddt_verify_step(const ddt_draft *draft, int budget, ddt_tree *tree, const ddt_attn_in *attn,
                    float scale, ddt_attn_out *attn_out, const int32_t *target_argmax, ddt_accept *acc,
                    void *workspace, size_t ws_bytes, void *stream) {
    // every check first, so an error enqueues nothing
    if (int rc = check_draft(draft, tree, budget)) return rc;
    if (int rc = check_attn(attn, tree, attn_out)) return rc;
    if (int rc = check_scale(scale)) return rc;
    if (int rc = check_accept(tree, target_argmax, acc)) return rc;
    if (int rc = check_device()) return rc;
    const ddt::AttnPlan plan = ddt::plan_attention(tree->B, tree->Qc, attn->H, attn->Tcap, device_info()->sms);
    if (plan.ws_bytes > ws_bytes || (plan.ws_bytes && !workspace)) return DDT_E_INVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (ddt::launch_tree_build(*draft, budget, *tree, s) != cudaSuccess) return DDT_E_CUDA;
    // the attention starts while the tree is being built (it waits, in the
    // kernel, before it reads the tree); with split keys the merge kernel
    // also runs the accept walk, else the accept follows the attention
    const ddt::AcceptArgs acc_args = ddt::accept_args(*tree, target_argmax, *acc);
    bool accepted = false;
    if (int rc = ddt::launch_verify_attn(*attn, *tree, scale, *attn_out, workspace, ws_bytes, plan, s, true,
                                         nullptr, 0, false, &acc_args, &accepted))
        return rc;
    if (!accepted && ddt::launch_tree_accept(*tree, target_argmax, *acc, s, true) != cudaSuccess)
        return DDT_E_CUDA;
    return DDT_OK;
}

int ddt_kv_commit(const ddt_accept *acc, int B, int D, int Tcap, void *c_kv, void *k_rope,
                  int32_t *prefix_len, int32_t *status, void *stream) {
    if (!acc || !acc->accept_len || !acc->accept_idx || !c_kv || !k_rope || !prefix_len || !status)
        return DDT_E_INVAL;
    if (B < 1 || B > 65535 || D < 1 || D > DDT_MAX_DEPTH || Tcap < 1) return DDT_E_INVAL;
    if (!aligned16(c_kv) || !aligned16(k_rope)) return DDT_E_INVAL;
    if (int rc = check_device()) return rc;
    return ddt::launch_kv_commit(B, D, Tcap, acc->accept_len, acc->accept_idx, c_kv, k_rope, prefix_len, status,
                                 static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? DDT_OK
               : DDT_E_CUDA;
}

int ddt_tree_sample(const ddt_tree *tree, const float *logits, int vocab, float temperature, const float *u01,
                    int32_t *sample_tok, float *node_p, void *stream) {
    if (!tree || !logits || !sample_tok || !node_p) return DDT_E_INVAL;
    if (!tree->token || !tree->parent || !tree->n_nodes || !tree->status) return DDT_E_INVAL;
    if (tree->B < 1 || tree->Qc < 1 || tree->Qc > DDT_MAX_BUDGET + 1) return DDT_E_INVAL;
    if (!(temperature == temperature) || temperature == INFINITY || temperature == -INFINITY) return DDT_E_INVAL;
    if (temperature > 0.f && (temperature < 1e-30f || !u01)) return DDT_E_INVAL;
    if (vocab < 4 || (vocab & 3) || !aligned16(logits)) return DDT_E_INVAL;
    if (int rc = check_device()) return rc;
    const int max_c = ddt::sample_max_cluster();
    if (max_c == 0) return DDT_E_CUDA;
    const ddt::SamplePlan plan =
        ddt::plan_sample(vocab, static_cast<long long>(tree->B) * tree->Qc, device_info()->sms, max_c);
    if (plan.C == 0) return DDT_E_INVAL;
    const double kd = temperature > 0.f ? 1.4426950408889634 / static_cast<double>(temperature) : 0.0;
    return ddt::launch_tree_sample(*tree, logits, vocab, kd, u01, sample_tok, node_p, plan,
                                   static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? DDT_OK
               : DDT_E_CUDA;
}

const char *ddt_status_str(int code) {
    switch (code) {
        case DDT_OK: return "ok";
        case DDT_E_INVAL: return "invalid argument";
        case DDT_E_CUDA: return "CUDA launch or runtime error";
        case DDT_E_UNSUPPORTED: return "device is not sm_103";
        case DDT_E_BADINPUT: return "bad input data (drafter rows, token ids or prefix length)";
        case DDT_E_TIMEOUT: return "bounded on-chip wait expired";
        case DDT_E_SCRATCH_LIMIT: return "shape needs more scratch than the no-allocation entry point holds";
        default: return "unknown status";
    }
}

int ddt_read_device_status(const int32_t *dev_status, int B, int32_t *host_out) {
    if (!dev_status || !host_out || B < 1) return DDT_E_INVAL;
    return cudaMemcpy(host_out, dev_status, sizeof(int32_t) * static_cast<size_t>(B), cudaMemcpyDeviceToHost) ==
                   cudaSuccess
               ? DDT_OK
               : DDT_E_CUDA;
}

int ddt_selftest_bounded_wait(int32_t *dev_status, unsigned timeout_us, void *stream) {
    if (!dev_status || timeout_us == 0 || timeout_us > 10000000u) return DDT_E_INVAL;
    if (int rc = check_device()) return rc;
    return ddt::launch_selftest_wait(dev_status, timeout_us, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? DDT_OK
               : DDT_E_CUDA;
}

}  // extern "C"
