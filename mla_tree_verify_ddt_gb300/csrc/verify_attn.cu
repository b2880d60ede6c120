// Tree-verify MLA-absorb attention on tcgen05 tensor cores (sm_103a).
//
// Computes, for every (sequence b, tree node i, head h) row,
//   s_j = scale * (q_lat . c_kv[j] + q_rope . k_rope[j])
// over the keys j the node may see — the whole committed prefix 0..T_b-1 and
// the keys T_b+m of its ancestors-or-self m — then
//   out = sum_j softmax(s)_j c_kv[j]   (the 512-wide latent, before w_vc)
//   lse = log sum_j exp(s_j).
// This is the absorbed-MLA verify attention of "The Architecture of a
// Thousand-Parameter Decision: Designing a Native DDTree Inference Engine for
// Kimi K2.6", section "What to Build New", item 2 (flash-style stream over the
// latent prefix plus a masked section over the tree nodes with a
// [q_len x q_len] visibility mask), with the key layout of "The Milestone
// Message", section "Architectural Abstraction" (nodes at positions L+depth,
// mask [ones | visibility]).
//
// Design (one CTA = 128 query rows x one half of the 512 output columns x one
// range of keys):
//  * rows are (node, head) pairs of one sequence, so every row of a tile
//    shares the sequence's KV: one 64-key KV tile feeds all 128 rows;
//  * S = Q K^T (M=128, N=64, K=576) and O += P V (M=128, N=256, K=64) run on
//    tcgen05 with fp32 accumulators in tensor memory. O for 128 rows x 512
//    columns would fill all 512 TMEM columns, leaving none for S, so each
//    CTA owns one 256-column half of O and recomputes S (the partner CTA of
//    the other half computes the same S bit for bit);
//  * the 512 latent query columns stay resident in shared memory (TMA,
//    128-byte swizzle); the 64 rotary query columns and the probabilities P
//    live in tensor memory and feed the MMA as its A operand;
//  * KV arrives by TMA in 64-column chunks: the four chunks that are this
//    half's V are double-buffered per tile and serve both S and PV; the other
//    five chunks stream through a 4-slot ring fed by a second producer warp,
//    so ring loads never queue behind V loads. S consumes the streamed chunks
//    first and the V chunks last, and a ready PV is slipped in between S
//    chunks;
//  * softmax runs on 4 warps, one thread per row, in fp32 in the log2 domain,
//    with a lazily moved reference max (O is rescaled only when a row's max
//    grows by more than 2^8);
//  * PV runs in fp16 (P rounded to fp16, 2^-11 relative, four times tighter
//    than bf16): after S of a tile has read its V chunks as bf16 K, the
//    softmax warps convert those chunks to fp16 in place;
//  * the softmax code is kept compact (visibility as one 64-bit word per
//    tile, rolled loops off the per-key path): the fully unrolled version
//    spent most of its time waiting for instruction fetch;
//  * when the key range is split over several CTAs, each writes a normalised
//    partial and its lse; a second kernel merges them.
// Every mbarrier wait is bounded; on expiry the CTA records DDT_E_TIMEOUT in
// the sequence's status word and leaves after draining its own copies.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "ddt_internal.h"
#include "ddt_ptx.cuh"

namespace ddt {
namespace {

constexpr int kRows = 128;        // query rows per CTA (MMA M)
constexpr int kKeys = 64;         // keys per tile (S MMA N)
constexpr int kChunkBytesQ = kRows * 128;   // 64 bf16 columns x 128 rows
constexpr int kChunkBytesKV = kKeys * 128;  // 64 bf16 columns x 64 keys
constexpr int kQChunks = 8;       // latent query: 512 columns
constexpr int kVChunks = 4;       // this CTA's half of the latent (256 columns)
constexpr int kStreamSlots = 4;
constexpr int kStreamPerTile = 5; // the other latent half (4) + rotary key (1)

// shared memory map (offsets from a 1024-aligned base)
constexpr int kOffQ = 0;
constexpr int kOffV = kOffQ + kQChunks * kChunkBytesQ;            // 131072
constexpr int kVSetBytes = kVChunks * kChunkBytesKV;              // 32768
constexpr int kOffStream = kOffV + 2 * kVSetBytes;                // 196608
constexpr int kOffBar = kOffStream + kStreamSlots * kChunkBytesKV; // 229376
constexpr int kSmemBytes = kOffBar + 256 + 1024;                  // + alignment slack

// tensor memory columns
constexpr uint32_t kColO = 0;     // 256 columns: this CTA's half of O
constexpr uint32_t kColS = 256;   // 2 x 64: S double buffer
constexpr uint32_t kColP = 384;   // 2 x 32: P (fp16 pairs) double buffer
constexpr uint32_t kColQR = 448;  // 32: rotary query (bf16 pairs)
constexpr uint32_t kTmemCols = 512;

constexpr float kRescaleThreshold = 8.0f;  // log2 units
// warps 0-3 softmax/epilogue, 4 TMA (Q, V), 5 MMA, 6 TMA (streamed chunks)
constexpr int kThreads = 224;

// barrier indices
enum {
    BAR_Q_FULL = 0,
    BAR_V_FULL = 1,      // 2
    BAR_V_EMPTY = 3,     // 2
    BAR_ST_FULL = 5,     // 4
    BAR_ST_EMPTY = 9,    // 4
    BAR_QR_READY = 13,
    BAR_S_FULL = 14,     // 2
    BAR_S_FREE = 16,     // 2
    BAR_P_FULL = 18,     // 2
    BAR_PV_DONE = 20,    // 2
    BAR_O_FINAL = 22,
    BAR_DRAIN = 23,
    NUM_BARS = 24
};

struct AttnArgs {
    int B, Qc, W, H, Tcap, nsplit;
    const uint64_t *mask;
    const int32_t *n_nodes;
    const int32_t *prefix_len;
    const uint16_t *q_rope;
    int32_t *status;
    float *o_dst;            // [nsplit][rows_total][512] (nsplit == 1: the final output)
    float *lse_dst;          // [nsplit][rows_total]
    size_t rows_total;       // B * Qc * H
    float scale_log2;        // scale * log2(e)
    unsigned long long wait_ns;
};

// Visibility of keys key0..key0+63 for a node with ancestor mask (m0, m1):
// every prefix key (< T) and the keys T+m of ancestors-or-self m < n. Only
// tiles that reach past the prefix need it; the loop stays rolled to keep
// the softmax code small.
__device__ __noinline__ uint64_t tile_visibility(int key0, int T, int n, uint64_t m0, uint64_t m1) {
    uint64_t vis = 0;
#pragma unroll 1
    for (int k = 0; k < 64; ++k) {
        const int key = key0 + k;
        bool v;
        if (key < T) {
            v = true;
        } else {
            const int m = key - T;
            v = m < n && (((m < 64 ? m0 : m1) >> (m & 63)) & 1ull);
        }
        vis |= static_cast<uint64_t>(v) << k;
    }
    return vis;
}

__global__ void __launch_bounds__(kThreads, 1)
    verify_attn_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_kv,
                       const __grid_constant__ CUtensorMap tm_kr, const AttnArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int mt = blockIdx.x >> 1;
    const int half = blockIdx.x & 1;
    const int chunk = blockIdx.y;
    const int b = blockIdx.z;

    // ---- per-sequence key range (uniform over the CTA)
    const int T = a.prefix_len[b];
    int n = a.n_nodes[b];
    n = n < 1 ? 1 : (n > a.Qc ? a.Qc : n);
    const bool seq_ok = (T >= 0) && (static_cast<long long>(T) + n <= a.Tcap);
    const int kend = seq_ok ? T + n : 0;
    const int ntiles = (kend + kKeys - 1) / kKeys;
    const int t0 = static_cast<int>((static_cast<long long>(ntiles) * chunk) / a.nsplit);
    const int t1 = static_cast<int>((static_cast<long long>(ntiles) * (chunk + 1)) / a.nsplit);
    const int nt = t1 - t0;
    const int rows_seq = a.Qc * a.H;
    const size_t row_base = static_cast<size_t>(b) * rows_seq;
    float *o_dst = a.o_dst + static_cast<size_t>(chunk) * a.rows_total * 512;
    float *lse_dst = a.lse_dst + static_cast<size_t>(chunk) * a.rows_total;

    if (!seq_ok && tid == 0 && mt == 0 && half == 0 && chunk == 0) a.status[b] = DDT_E_BADINPUT;

    if (nt <= 0) {
        // nothing visible in this range: zero rows, lse = -inf
        for (int idx = tid; idx < kRows * 64; idx += blockDim.x) {
            const int r = idx >> 6, c4 = idx & 63;
            const int g = mt * kRows + r;
            if (g >= rows_seq) continue;
            float4 *dst = reinterpret_cast<float4 *>(o_dst + (row_base + g) * 512 + half * 256) + c4;
            *dst = make_float4(0.f, 0.f, 0.f, 0.f);
            if (half == 0 && c4 == 0) lse_dst[row_base + g] = -INFINITY;
        }
        return;
    }

    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + kOffQ, sV = sbase + kOffV, sST = sbase + kOffStream;
    const uint32_t sBar = sbase + kOffBar;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffBar + NUM_BARS * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffBar + NUM_BARS * 8 + 4);
    auto bar = [&](int i) { return sBar + 8u * static_cast<uint32_t>(i); };

    if (tid == 0) {
        mbar_init(bar(BAR_Q_FULL), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(BAR_V_FULL + s), 1);
            mbar_init(bar(BAR_V_EMPTY + s), 1);
            mbar_init(bar(BAR_S_FULL + s), 1);
            mbar_init(bar(BAR_S_FREE + s), 4);
            mbar_init(bar(BAR_P_FULL + s), 4);
            mbar_init(bar(BAR_PV_DONE + s), 1);
        }
        for (int s = 0; s < kStreamSlots; ++s) {
            mbar_init(bar(BAR_ST_FULL + s), 1);
            mbar_init(bar(BAR_ST_EMPTY + s), 1);
        }
        mbar_init(bar(BAR_QR_READY), 4);
        mbar_init(bar(BAR_O_FINAL), 1);
        mbar_init(bar(BAR_DRAIN), 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint64_t deadline = globaltimer_ns() + a.wait_ns;

    auto fail = [&]() {
        *abort_flag = 1;
        a.status[b] = DDT_E_TIMEOUT;
    };

    if (warp == 4) {
        // ================= TMA producer: Q once, then this half's V chunks =================
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_kv);
            const int qrow = static_cast<int>(row_base) + mt * kRows;
            mbar_arrive_expect_tx(bar(BAR_Q_FULL), kQChunks * kChunkBytesQ);
            for (int c = 0; c < kQChunks; ++c)
                tma_load_2d(sQ + c * kChunkBytesQ, &tm_q, c * 64, qrow, bar(BAR_Q_FULL));
            int armed_v[2] = {0, 0};
            bool ok = true;
            for (int jj = 0; jj < nt; ++jj) {
                const int key_row = b * a.Tcap + (t0 + jj) * kKeys;
                const int vs = jj & 1;
                if (jj >= 2 && !mbar_wait(bar(BAR_V_EMPTY + vs), ((jj - 2) >> 1) & 1, deadline, abort_flag)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(bar(BAR_V_FULL + vs), kVSetBytes);
                ++armed_v[vs];
                for (int c = 0; c < kVChunks; ++c)
                    tma_load_2d(sV + vs * kVSetBytes + c * kChunkBytesKV, &tm_kv,
                                (kVChunks * half + c) * 64, key_row, bar(BAR_V_FULL + vs));
            }
            if (!ok) {
                fail();
                // let every copy this thread started land before the CTA leaves
                const uint64_t drain_deadline = globaltimer_ns() + 100000000ull;
                const int zero = 0;
                mbar_wait(bar(BAR_Q_FULL), 0, drain_deadline, &zero);
                for (int s = 0; s < 2; ++s)
                    if (armed_v[s]) mbar_wait(bar(BAR_V_FULL + s), (armed_v[s] - 1) & 1, drain_deadline, &zero);
            }
        }
    } else if (warp == 6) {
        // ====== TMA producer: the other latent half and the rotary key, through the ring ======
        if (lane == 0) {
            tma_prefetch_desc(&tm_kr);
            int armed_st[kStreamSlots] = {0, 0, 0, 0};
            int st_cnt = 0;
            bool ok = true;
            for (int jj = 0; jj < nt && ok; ++jj) {
                const int key_row = b * a.Tcap + (t0 + jj) * kKeys;
                for (int q = 0; q < kStreamPerTile; ++q) {
                    const int slot = st_cnt % kStreamSlots, use = st_cnt / kStreamSlots;
                    if (use >= 1 && !mbar_wait(bar(BAR_ST_EMPTY + slot), (use - 1) & 1, deadline, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(BAR_ST_FULL + slot), kChunkBytesKV);
                    ++armed_st[slot];
                    if (q < 4)
                        tma_load_2d(sST + slot * kChunkBytesKV, &tm_kv,
                                    (kVChunks * (1 - half) + q) * 64, key_row, bar(BAR_ST_FULL + slot));
                    else
                        tma_load_2d(sST + slot * kChunkBytesKV, &tm_kr, 0, key_row,
                                    bar(BAR_ST_FULL + slot));
                    ++st_cnt;
                }
            }
            if (!ok) {
                fail();
                const uint64_t drain_deadline = globaltimer_ns() + 100000000ull;
                const int zero = 0;
                for (int s = 0; s < kStreamSlots; ++s)
                    if (armed_st[s]) mbar_wait(bar(BAR_ST_FULL + s), (armed_st[s] - 1) & 1, drain_deadline, &zero);
            }
        }
    } else if (warp == 5) {
        // ======================= MMA issuer =======================
        if (lane == 0) {
            constexpr uint32_t idS = idesc_f32acc(kRows, kKeys, 1, 0, 0);   // bf16 Q, K
            constexpr uint32_t idPV = idesc_f32acc(kRows, 256, 0, 0, 1);  // fp16 P, V (MN-major)
            bool ok = mbar_wait(bar(BAR_Q_FULL), 0, deadline, abort_flag) &&
                      mbar_wait(bar(BAR_QR_READY), 0, deadline, abort_flag);
            tc_fence_after();
            int st_cnt = 0;
            int pv_next = 0;  // the next tile whose PV is still to be issued
            // O += P_j V_j once the softmax has published P_j. With block ==
            // false it only issues when P_j is already there, so a PV can slip
            // in between the chunks of the next S as soon as it is ready.
            auto issue_pv = [&](int j, bool block) -> int {
                const int pb = j & 1;
                if (block) {
                    if (!mbar_wait(bar(BAR_P_FULL + pb), (j >> 1) & 1, deadline, abort_flag)) return -1;
                } else if (!mbar_try_wait(bar(BAR_P_FULL + pb), (j >> 1) & 1)) {
                    return 0;
                }
                tc_fence_after();
                const uint32_t vb = sV + pb * kVSetBytes;
                for (int ks = 0; ks < kKeys / 16; ++ks)
                    mma_ts(tmem + kColO, tmem + kColP + pb * 32 + ks * 8,
                           desc_sw128(vb + ks * 2048, kChunkBytesKV, 1024), idPV,
                           (j > 0 || ks > 0) ? 1u : 0u);
                mma_commit(bar(BAR_PV_DONE + pb));
                mma_commit(bar(BAR_V_EMPTY + pb));
                return 1;
            };
            for (int jj = 0; jj < nt && ok; ++jj) {
                const int sb = jj & 1;
                if (jj >= 2 && !mbar_wait(bar(BAR_S_FREE + sb), ((jj - 2) >> 1) & 1, deadline, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t dS = tmem + kColS + sb * kKeys;
                // the streamed chunks first: the other latent half and the rotary part
                for (int q = 0; q < kStreamPerTile; ++q) {
                    const int slot = st_cnt % kStreamSlots, use = st_cnt / kStreamSlots;
                    if (!mbar_wait(bar(BAR_ST_FULL + slot), use & 1, deadline, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t kb = sST + slot * kChunkBytesKV;
                    if (q < 4) {
                        const uint32_t qa = sQ + (kVChunks * (1 - half) + q) * kChunkBytesQ;
                        for (int ks = 0; ks < 4; ++ks)
                            mma_ss(dS, desc_sw128(qa + ks * 32, 16, 1024), desc_sw128(kb + ks * 32, 16, 1024),
                                   idS, (q > 0 || ks > 0) ? 1u : 0u);
                    } else {
                        for (int ks = 0; ks < 4; ++ks)
                            mma_ts(dS, tmem + kColQR + ks * 8, desc_sw128(kb + ks * 32, 16, 1024), idS, 1u);
                    }
                    mma_commit(bar(BAR_ST_EMPTY + slot));
                    ++st_cnt;
                    if (pv_next < jj) {
                        const int r = issue_pv(pv_next, false);
                        if (r < 0) {
                            ok = false;
                            break;
                        }
                        pv_next += r;
                    }
                }
                if (!ok) break;
                // this half's latent columns last: the V chunks double as K
                if (!mbar_wait(bar(BAR_V_FULL + sb), (jj >> 1) & 1, deadline, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int c = 0; c < kVChunks; ++c) {
                    const uint32_t qa = sQ + (kVChunks * half + c) * kChunkBytesQ;
                    const uint32_t kb = sV + sb * kVSetBytes + c * kChunkBytesKV;
                    for (int ks = 0; ks < 4; ++ks)
                        mma_ss(dS, desc_sw128(qa + ks * 32, 16, 1024), desc_sw128(kb + ks * 32, 16, 1024), idS, 1u);
                }
                mma_commit(bar(BAR_S_FULL + sb));
                while (ok && pv_next < jj) {
                    if (issue_pv(pv_next, true) < 0) ok = false;
                    else ++pv_next;
                }
            }
            if (ok && issue_pv(nt - 1, true) < 0) ok = false;
            if (ok) {
                mma_commit(bar(BAR_O_FINAL));
            } else {
                fail();
                // wait for this thread's MMAs before tensor memory is released
                mma_commit(bar(BAR_DRAIN));
                const int zero = 0;
                mbar_wait(bar(BAR_DRAIN), 0, globaltimer_ns() + 100000000ull, &zero);
            }
        }
    } else {
        // ======================= softmax / epilogue (warps 0-3) =======================
        const int row = warp * 32 + lane;
        const int g = mt * kRows + row;           // row within the sequence
        const bool row_in_seq = g < rows_seq;
        const int node = g / a.H;
        const bool node_ok = row_in_seq && node < n && seq_ok;
        uint64_t m0 = 0, m1 = 0;
        if (node_ok) {
            const uint64_t *mk = a.mask + (static_cast<size_t>(b) * a.Qc + node) * a.W;
            m0 = mk[0];
            if (a.W > 1) m1 = mk[1];
        }
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        // rotary query row -> tensor memory (bf16 pairs, low half = even column)
        {
            uint32_t qr[32];
            if (row_in_seq) {
                const uint4 *src = reinterpret_cast<const uint4 *>(a.q_rope + (row_base + g) * 64);
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    const uint4 x = src[v];
                    qr[4 * v + 0] = x.x;
                    qr[4 * v + 1] = x.y;
                    qr[4 * v + 2] = x.z;
                    qr[4 * v + 3] = x.w;
                }
            } else {
#pragma unroll
                for (int v = 0; v < 32; ++v) qr[v] = 0;
            }
            tmem_st32(tmem + lane_base + kColQR, qr);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(BAR_QR_READY));
        }
        float m_ref = -INFINITY, l_sum = 0.f;
        bool ok = true;
        for (int jj = 0; jj < nt; ++jj) {
            const int sb = jj & 1;
            const int key0 = (t0 + jj) * kKeys;
            if (!mbar_wait(bar(BAR_S_FULL + sb), (jj >> 1) & 1, deadline, abort_flag)) {
                ok = false;
                break;
            }
            __syncwarp();
            tc_fence_after();
            uint32_t sv[64];
            {
                uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[0]);
                uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[32]);
                tmem_ld32(tmem + lane_base + kColS + sb * kKeys, lo);
                tmem_ld32(tmem + lane_base + kColS + sb * kKeys + 32, hi);
                tmem_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(BAR_S_FREE + sb));
            // scale, mask, tile max
            uint64_t vis = ~0ull;
            if (!node_ok) vis = 0;
            else if (key0 + kKeys > T) vis = tile_visibility(key0, T, n, m0, m1);
            const uint32_t vis_lo = static_cast<uint32_t>(vis), vis_hi = static_cast<uint32_t>(vis >> 32);
            float x[64];
            float mx = -INFINITY;
#pragma unroll
            for (int k = 0; k < 64; ++k) {
                const uint32_t bit = (k < 32 ? (vis_lo >> k) : (vis_hi >> (k - 32))) & 1u;
                x[k] = bit ? __uint_as_float(sv[k]) * a.scale_log2 : -INFINITY;
                mx = fmaxf(mx, x[k]);
            }
            // P buffer sb was last read by PV of tile jj-2
            if (jj >= 2 && !mbar_wait(bar(BAR_PV_DONE + sb), ((jj - 2) >> 1) & 1, deadline, abort_flag)) {
                ok = false;
                break;
            }
            const bool need = mx > m_ref + kRescaleThreshold;
            if (__any_sync(0xffffffffu, need)) {
                const float alpha = need ? ex2_approx(m_ref - mx) : 1.0f;
                if (need) {
                    m_ref = mx;
                    l_sum *= alpha;
                }
                if (jj >= 1) {
                    // O must be quiescent: PV of tile jj-1 complete
                    if (!mbar_wait(bar(BAR_PV_DONE + ((jj - 1) & 1)), ((jj - 1) >> 1) & 1, deadline, abort_flag)) {
                        ok = false;
                        break;
                    }
                    __syncwarp();
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 8; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tmem + lane_base + kColO + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int v = 0; v < 32; ++v) o[v] = __float_as_uint(__uint_as_float(o[v]) * alpha);
                        tmem_st32(tmem + lane_base + kColO + c * 32, o);
                    }
                    tmem_wait_st();
                }
            }
            // probabilities (fp16) into tensor memory. While no key has been
            // visible yet m_ref is -inf and every x is -inf: subtracting 0
            // instead keeps p = 0 without a per-element test. The row sum
            // adds the fp32 values (fp16 rounding is unbiased, 2^-11 each).
            uint32_t pk[32];
            const float mref = (m_ref == -INFINITY) ? 0.f : m_ref;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const float p0 = ex2_approx(x[2 * k] - mref);
                const float p1 = ex2_approx(x[2 * k + 1] - mref);
                pk[k] = pack_f16x2(p0, p1);
                l_sum += p0 + p1;
            }
            tmem_st32(tmem + lane_base + kColP + sb * 32, pk);
            // S of this tile is complete, so its V chunks (read as bf16 K by
            // S) can turn into the fp16 B operand of PV, in place. KV rows
            // past the last node may hold anything (NaN included): they become
            // zeros so that 0 * garbage cannot reach O.
            {
                uint4 *vset = reinterpret_cast<uint4 *>(smem + kOffV + sb * kVSetBytes);
                const int kvalid = kend - key0;  // keys of this tile that exist
#pragma unroll 1
                for (int e0 = row; e0 < kVSetBytes / 16; e0 += 4 * kRows) {
                    uint4 v[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) v[u] = vset[e0 + u * kRows];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int key = ((e0 + u * kRows) >> 3) & (kKeys - 1);  // 8 units of 16 B per key row
                        if (key < kvalid) {
                            v[u].x = bf16x2_to_f16x2(v[u].x);
                            v[u].y = bf16x2_to_f16x2(v[u].y);
                            v[u].z = bf16x2_to_f16x2(v[u].z);
                            v[u].w = bf16x2_to_f16x2(v[u].w);
                        } else {
                            v[u] = make_uint4(0, 0, 0, 0);
                        }
                        vset[e0 + u * kRows] = v[u];
                    }
                }
                fence_proxy_async_smem();
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(BAR_P_FULL + sb));
        }
        if (ok && !mbar_wait(bar(BAR_O_FINAL), 0, deadline, abort_flag)) ok = false;
        if (!ok) {
            fail();
        } else {
            __syncwarp();
            tc_fence_after();
            const float inv_l = l_sum > 0.f ? 1.0f / l_sum : 0.f;
            float *dst = o_dst + (row_base + g) * 512 + half * 256;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_base + kColO + c * 32, o);
                tmem_wait_ld();
                if (row_in_seq) {
                    float4 *d4 = reinterpret_cast<float4 *>(dst + c * 32);
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        d4[v] = make_float4(__uint_as_float(o[4 * v]) * inv_l, __uint_as_float(o[4 * v + 1]) * inv_l,
                                            __uint_as_float(o[4 * v + 2]) * inv_l,
                                            __uint_as_float(o[4 * v + 3]) * inv_l);
                }
            }
            if (half == 0 && row_in_seq)
                lse_dst[row_base + g] = l_sum > 0.f ? (m_ref + __log2f(l_sum)) * 0.69314718055994531f : -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Merge per-chunk normalised partials: lse = log sum_c exp(lse_c),
// out = sum_c exp(lse_c - lse) out_c. One 128-thread block per row.
__global__ void __launch_bounds__(128)
    merge_chunks_kernel(size_t rows_total, int nsplit, const float *__restrict__ ws_o,
                        const float *__restrict__ ws_lse, float *__restrict__ out,
                        float *__restrict__ lse) {
    const size_t r = blockIdx.x;
    if (r >= rows_total) return;
    float mx = -INFINITY;
    for (int c = 0; c < nsplit; ++c) mx = fmaxf(mx, ws_lse[c * rows_total + r]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float sum = 0.f;
    if (mx != -INFINITY) {
        for (int c = 0; c < nsplit; ++c) {
            const float lc = ws_lse[c * rows_total + r];
            if (lc == -INFINITY) continue;
            const float w = __expf(lc - mx);
            sum += w;
            const float4 v = reinterpret_cast<const float4 *>(ws_o + (c * rows_total + r) * 512)[threadIdx.x];
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        }
        const float inv = 1.0f / sum;
        acc.x *= inv;
        acc.y *= inv;
        acc.z *= inv;
        acc.w *= inv;
    }
    reinterpret_cast<float4 *>(out + r * 512)[threadIdx.x] = acc;
    if (threadIdx.x == 0) lse[r] = (mx == -INFINITY) ? -INFINITY : mx + __logf(sum);
}

// ---------------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool encode_2d(EncodeTiledFn enc, CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows,
               uint32_t box_cols, uint32_t box_rows) {
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

AttnPlan plan_attention(int B, int Qc, int H, int Tcap, int sms) {
    AttnPlan p{};
    p.mtiles = (Qc * H + kRows - 1) / kRows;
    const long long base = static_cast<long long>(B) * p.mtiles * 2;
    const int tiles_max = (Tcap + kKeys - 1) / kKeys;
    int nsplit = 1;
    if (base < 2LL * sms) {
        // spread the key range until the grid covers the GPU about twice, but
        // keep at least 4 key tiles per chunk
        nsplit = static_cast<int>((2LL * sms + base - 1) / base);
        const int max_split = tiles_max / 4 > 1 ? tiles_max / 4 : 1;
        if (nsplit > max_split) nsplit = max_split;
        if (nsplit < 1) nsplit = 1;
    }
    p.nsplit = nsplit;
    const size_t rows_total = static_cast<size_t>(B) * Qc * H;
    p.ws_bytes = nsplit > 1 ? static_cast<size_t>(nsplit) * rows_total * (512 + 1) * sizeof(float) : 0;
    return p;
}

int launch_verify_attn(const ddt_attn_in &in, const ddt_tree &tree, float scale,
                       const ddt_attn_out &out, void *workspace, size_t ws_bytes,
                       const AttnPlan &plan, cudaStream_t s) {
    EncodeTiledFn enc = get_encoder();
    if (!enc) return DDT_E_CUDA;
    const uint64_t rows_total = static_cast<uint64_t>(tree.B) * tree.Qc * in.H;
    const uint64_t kv_rows = static_cast<uint64_t>(tree.B) * in.Tcap;
    CUtensorMap tm_q, tm_kv, tm_kr;
    if (!encode_2d(enc, &tm_q, in.q_lat, 512, rows_total, 64, kRows) ||
        !encode_2d(enc, &tm_kv, in.c_kv, 512, kv_rows, 64, kKeys) ||
        !encode_2d(enc, &tm_kr, in.k_rope, 64, kv_rows, 64, kKeys))
        return DDT_E_INVAL;

    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(verify_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kSmemBytes);
    });
    if (attr_err != cudaSuccess) return DDT_E_CUDA;

    AttnArgs a{};
    a.B = tree.B;
    a.Qc = tree.Qc;
    a.W = tree.W;
    a.H = in.H;
    a.Tcap = in.Tcap;
    a.nsplit = plan.nsplit;
    a.mask = tree.mask;
    a.n_nodes = tree.n_nodes;
    a.prefix_len = in.prefix_len;
    a.q_rope = static_cast<const uint16_t *>(in.q_rope);
    a.status = tree.status;
    a.rows_total = rows_total;
    a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    a.wait_ns = kWaitLimitNs;
    float *ws_o = nullptr, *ws_lse = nullptr;
    if (plan.nsplit > 1) {
        if (!workspace || ws_bytes < plan.ws_bytes) return DDT_E_INVAL;
        ws_o = static_cast<float *>(workspace);
        ws_lse = ws_o + static_cast<size_t>(plan.nsplit) * rows_total * 512;
        a.o_dst = ws_o;
        a.lse_dst = ws_lse;
    } else {
        a.o_dst = out.out;
        a.lse_dst = out.lse;
    }
    dim3 grid(plan.mtiles * 2, plan.nsplit, tree.B);
    verify_attn_kernel<<<grid, kThreads, kSmemBytes, s>>>(tm_q, tm_kv, tm_kr, a);
    if (cudaGetLastError() != cudaSuccess) return DDT_E_CUDA;
    if (plan.nsplit > 1) {
        merge_chunks_kernel<<<static_cast<unsigned>(rows_total), 128, 0, s>>>(
            rows_total, plan.nsplit, ws_o, ws_lse, out.out, out.lse);
        if (cudaGetLastError() != cudaSuccess) return DDT_E_CUDA;
    }
    return DDT_OK;
}

// ---------------------------------------------------------------- self-test
namespace {
__global__ void selftest_wait_kernel(int32_t *status, unsigned long long wait_ns) {
    __shared__ __align__(8) uint64_t bar_storage;
    __shared__ int abort_flag;
    const uint32_t bar = smem_u32(&bar_storage);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // nothing ever arrives on this barrier: the wait must give up
        const bool ok = mbar_wait(bar, 0, globaltimer_ns() + wait_ns, &abort_flag);
        *status = ok ? DDT_OK : DDT_E_TIMEOUT;
    }
}
}  // namespace

cudaError_t launch_selftest_wait(int32_t *status, unsigned timeout_us, cudaStream_t s) {
    selftest_wait_kernel<<<1, 32, 0, s>>>(status, static_cast<unsigned long long>(timeout_us) * 1000ull);
    return cudaGetLastError();
}

}  // namespace ddt
