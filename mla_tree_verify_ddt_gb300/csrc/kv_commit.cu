// KV commit after acceptance: the accepted nodes' latent and rotary keys move
// into the committed prefix, on the device, with no host round-trip.
//
// Follows "The Architecture of a Thousand-Parameter Decision: Designing a
// Native DDTree Inference Engine for Kimi K2.6", section "What to Build New",
// items 4 and 5 (the step ends draft -> build -> verify -> accept -> append,
// the append writing the committed tokens' KV), with the key layout of "The
// Milestone Message", section "Architectural Abstraction" (node m's key at
// position L + m). For sequence b with prefix length T and accepted path
// a_0 = 0 (the root), a_1 < ... < a_{L-1}: rows T + a_k of c_kv and k_rope
// become rows T + k, and the prefix length becomes T + L.
//
// One block per sequence. A later source row can be an earlier destination
// (a_k = k' for some k' > k), so the block first stages all the path's rows in
// shared memory, then writes them. At most 17 rows of 1152 bytes.
#include <cuda_runtime.h>

#include <cstdint>

#include "ddt_internal.h"

namespace ddt {
namespace {

constexpr int kThreads = 128;
constexpr int kKvWords = 512 * 2 / 16;   // uint4 per latent row (1024 B)
constexpr int kKrWords = 64 * 2 / 16;    // uint4 per rotary row (128 B)
constexpr int kRowWords = kKvWords + kKrWords;
constexpr int kMaxPath = DDT_MAX_DEPTH + 1;

__global__ void __launch_bounds__(kThreads)
    kv_commit_kernel(int D, int Tcap, const int32_t *__restrict__ accept_len, const int32_t *__restrict__ accept_idx,
                     uint4 *__restrict__ c_kv, uint4 *__restrict__ k_rope, int32_t *__restrict__ prefix_len,
                     int32_t *__restrict__ status) {
    __shared__ uint4 rows[kMaxPath * kRowWords];
    __shared__ int path[kMaxPath];
    __shared__ int s_ok;
    const int b = blockIdx.x;
    const int T = prefix_len[b], L = accept_len[b];
    const int32_t *ai = accept_idx + static_cast<size_t>(b) * (D + 1);
    if (threadIdx.x < 32) {
        // the path in one load, checked by the warp: it starts at the root,
        // rises, and stays below Tcap
        const int lane = threadIdx.x;
        const bool in_path = lane < L && lane <= D;
        const int a = in_path ? ai[lane] : 0;
        const int prev = __shfl_up_sync(0xffffffffu, a, 1);
        const bool bad = in_path && (lane == 0 ? a != 0 : (a <= prev || static_cast<long long>(T) + a >= Tcap));
        const bool ok = L >= 1 && L <= D + 1 && T >= 0 && static_cast<long long>(T) + L <= Tcap &&
                        !__any_sync(0xffffffffu, bad);
        if (in_path) path[lane] = a;
        if (lane == 0) s_ok = ok;
    }
    __syncthreads();
    if (!s_ok) {
        if (threadIdx.x == 0) status[b] = DDT_E_BADINPUT;
        return;
    }
    uint4 *kv = c_kv + static_cast<size_t>(b) * Tcap * kKvWords;
    uint4 *kr = k_rope + static_cast<size_t>(b) * Tcap * kKrWords;
    // rows k = 1 .. L-1 (the root stays where it is)
    const int n = (L - 1) * kRowWords;
    for (int e = threadIdx.x; e < n; e += kThreads) {
        const int k = 1 + e / kRowWords, w = e % kRowWords;
        const size_t src = static_cast<size_t>(T) + path[k];
        rows[e] = w < kKvWords ? kv[src * kKvWords + w] : kr[src * kKrWords + (w - kKvWords)];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < n; e += kThreads) {
        const int k = 1 + e / kRowWords, w = e % kRowWords;
        const size_t dst = static_cast<size_t>(T) + k;
        if (w < kKvWords) kv[dst * kKvWords + w] = rows[e];
        else kr[dst * kKrWords + (w - kKvWords)] = rows[e];
    }
    if (threadIdx.x == 0) prefix_len[b] = T + L;
}

}  // namespace

cudaError_t launch_kv_commit(int B, int D, int Tcap, const int32_t *accept_len, const int32_t *accept_idx,
                             void *c_kv, void *k_rope, int32_t *prefix_len, int32_t *status, cudaStream_t s) {
    kv_commit_kernel<<<B, kThreads, 0, s>>>(D, Tcap, accept_len, accept_idx, static_cast<uint4 *>(c_kv),
                                             static_cast<uint4 *>(k_rope), prefix_len, status);
    return cudaGetLastError();
}

}  // namespace ddt
