// Temperature sampling at every node of a verified draft tree, and each
// node's probability under its parent's distribution.
//
// Follows "The Architecture of a Thousand-Parameter Decision: Designing a
// Native DDTree Inference Engine for Kimi K2.6": section "What to Reuse",
// item 3 (temperature-based sampling from the verified token distribution
// over the tree) and section "What to Build New", item 2 (the
// sampling-probability path: the target's probabilities normalised over the
// tree nodes) and item 5 (greedy and temperature commit paths).
//
// Row (b, i) of the logits [B,Qc,V] is the target's logit vector after node
// i. Its distribution is p_j = 2^((x_j - M) kd) / S with kd = log2(e) / tau,
// M the row's largest logit and S the sum of the numerators. One uniform u
// per node draws the node's sample by inverse transform over token ids in
// increasing order: the first token of nonzero weight whose cumulative weight
// exceeds u * S; when none does (u >= 1, or rounding at the very top), the
// last token of nonzero weight. Following the verified tree with these
// samples in place of the greedy argmax (the accept walk) commits tokens
// distributed exactly as the target's temperature sampling would.
//
// Layout of the work. A persistent grid of clusters of C CTAs; cluster g
// takes rows g, g + G, g + 2G, ... (G clusters). In a row, CTA c owns tokens
// [c * NREG * R * 128, (c + 1) * NREG * R * 128), cut into NREG regions of
// 128 R tokens; warp w takes the contiguous regions w Q .. w Q + Q - 1
// (Q = NREG / 8) and streams them, row after row, through a two-stage ring
// of bulk copies into shared memory; the logits are read from HBM once. In a region lane l owns the R consecutive
// float4 l R .. l R + R - 1 (R odd: the 8 lanes of a 128-bit shared-memory
// phase then hit 8 different bank groups). C is the smallest cluster that
// still fills the GPU (two CTAs per SM): every row ends with block-wide (and,
// for C > 1, cluster-wide) synchronisation, so the longer a CTA's share of a
// row, the smaller that fixed cost against its streaming time.
//
// Per region (one warp):
//   pass 1  largest logit (NaN-propagating max; the greedy kernel then finds
//           its first index);
//   pass 2  weights against the region's largest logit, 4 at a time (a quad
//           sum), a sequential sum per lane, an inclusive scan over the
//           lanes (its last entry is the region total); the warp folds the
//           total into its running float-pair prefix over its regions, kept
//           in units of its running maximum (a new maximum rescales the
//           prefix: an exact power of two times a hardware exp2 of the
//           fraction).
// Per row:
//   CTA      the 8 warps' prefixes scaled to the CTA's maximum and scanned in
//           warp order;
//   cluster  every CTA writes its (max, first index, total) into every CTA
//           of the cluster (distributed shared memory stores); after a
//           cluster barrier each reads the C summaries locally and computes
//           the same row maximum, float-pair scan, total and winning CTA;
//   locate   the winning CTA descends warp -> region -> lane -> float4 ->
//           element over the sums it built (a region's prefix brought to its
//           warp's final maximum); for the float4 level it reloads the chosen
//           lane's R float4 from memory and recomputes their quad sums, which
//           come out bit-identical (one fixed sequence of correctly rounded
//           operations). A threshold past a level's total takes that level's
//           last entry of nonzero weight.
// Rank 0 of the cluster writes the greedy result and the children's node
// probabilities (the child token's weight against the row maximum over the
// row total). No float64: this GPU's float64 rate is a small fraction of
// float32's, so the sums above a lane are float pairs (hi + lo).
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "ddt_internal.h"
#include "ddt_ptx.cuh"

namespace ddt {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kStages = 2;  // ring depth per warp
constexpr int kFlagNan = 1, kFlagTimeout = 2, kFlagNoDist = 4;
constexpr int kMaxNodes = DDT_MAX_BUDGET + 1;

struct Ctrl {
    uint64_t bar[kWarps][kStages];
    // per region; warp w owns regions w Q .. w Q + Q - 1 (contiguous tokens)
    float rmax[kSampleMaxRegions];     // region maximum
    float rtot[kSampleMaxRegions];     // region total, units of 2^((x - rmax) kd)
    unsigned lpos[kSampleMaxRegions];  // lanes of the region with nonzero weight
    float rref[kSampleMaxRegions];     // the warp's running maximum W after this region
    float rp_hi[kSampleMaxRegions], rp_lo[kSampleMaxRegions];  // running prefix, units of 2^((x - W) kd)
    // per warp: maximum (greedy: its first index), flags, total, and the
    // CTA-level scale, mass and inclusive scan
    float wmax[kWarps], wp_hi[kWarps], wp_lo[kWarps];
    int widx[kWarps], wflag[kWarps];
    float wfs[kWarps], wmass[kWarps], wscan_hi[kWarps], wscan_lo[kWarps];
    float quads[32];  // the located lane's quad sums
    // the cluster's CTA summaries, written by each CTA into every CTA of the
    // cluster (slot = writer's rank), double-buffered by row parity
    float xm[2][16], xhi[2][16], xlo[2][16];
    int xidx[2][16], xflag[2][16];
    // the row's result, identical in every CTA of the cluster
    int row_flag, row_idx, cstar;
    float row_m, row_s, t_hi, t_lo;
    // the cluster's rows that hold a node (padding slots left out), in order
    int nlist;
    int wcount[kWarps];
    int list_row[kSampleListCap];
    int list_n[kSampleListCap];
    float list_u[kSampleListCap];
    // node i's children (thread c holds node c): parent, token, logit
    int cpar[kMaxNodes], ctok[kMaxNodes];
    float cx[kMaxNodes];
};

struct SampleArgs {
    const float *logits;
    const float *u01;
    const int32_t *token;
    const int32_t *parent;
    const int32_t *n_nodes;
    int32_t *sample_tok;
    float *node_p;
    int32_t *status;
    float kh, kl;        // log2(e) / temperature = kh + kl, kl > 0 (unused by the greedy kernel)
    int row0, rows_end;  // this launch's rows: cluster g takes row0 + g + t * G < rows_end
    int Qc, V, C, nreg, G;
};

// Bulk copy global -> this CTA's shared memory, credited to `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Store into the same shared-memory location of CTA `rank` of the cluster.
__device__ __forceinline__ void st_peer_f32(float *p, uint32_t rank, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(mapa_shared(smem_u32(p), rank)), "f"(v) : "memory");
}
__device__ __forceinline__ void st_peer_s32(int *p, uint32_t rank, int v) {
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(mapa_shared(smem_u32(p), rank)), "r"(v) : "memory");
}

// 4 bytes global -> shared without holding a register; cp.async.wait_all
// makes them visible to the issuing thread.
__device__ __forceinline__ void cp_async_4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// max that returns NaN when either operand is NaN
__device__ __forceinline__ float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity) {
    const uint64_t deadline = globaltimer_ns() + kWaitLimitNs;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 63u && globaltimer_ns() > deadline) return false;
    }
}

// Weights of two logits x against the reference m: 2^((x - m) kd), kd
// carried as kh + kl with kl > 0 (so x = -inf gives -inf * kl = -inf, weight
// 0, and a NaN propagates), computed with packed float32x2 instructions.
// Every operation is explicitly rounded to nearest (no contraction), so the
// same inputs give the same bits wherever this is evaluated.
__device__ __forceinline__ void weight2(float x0, float x1, float m, float kh, float kl, float &e0, float &e1) {
    float d0, d1, t0, t1, a0, a1;
    sub_f32x2(x0, x1, m, m, d0, d1);
    mul_f32x2(d0, d1, kl, kl, t0, t1);
    fma_f32x2_vv(d0, d1, kh, kh, t0, t1, a0, a1);
    e0 = ex2_approx(a0);
    e1 = ex2_approx(a1);
}

__device__ __forceinline__ float quad_sum(const float4 v, float m, float kh, float kl) {
    float e0, e1, e2, e3;
    weight2(v.x, v.y, m, kh, kl, e0, e1);
    weight2(v.z, v.w, m, kh, kl, e2, e3);
    return __fadd_rn(__fadd_rn(__fadd_rn(e0, e1), e2), e3);
}

// NaN-propagating maximum of three
__device__ __forceinline__ float max_nan3(float a, float b, float c) {
    float r;
    asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// 2^((a - b) kd) for a <= b with an exponent good to far below float32
// rounding: a - b as an exact float pair (two-sum), its product with
// kd = kh + kl as a float pair (the fma residual), the integer part of the
// exponent applied exactly (ldexpf) and only the fraction through exp2.
__device__ __forceinline__ float exp2_diff(float a, float b, float kh, float kl) {
    if (a == -INFINITY) return 0.f;
    const float nb = -b;
    const float s = __fadd_rn(a, nb);
    const float bv = __fsub_rn(s, a);
    const float av = __fsub_rn(s, bv);
    const float err = __fadd_rn(__fsub_rn(a, av), __fsub_rn(nb, bv));  // s + err == a - b exactly
    const float ph = __fmul_rn(s, kh);
    if (ph < -250.f) return 0.f;
    const float pl = __fmaf_rn(s, kh, -ph);
    const float rest = __fadd_rn(pl, __fadd_rn(__fmul_rn(s, kl), __fmul_rn(err, kh)));
    const float n = rintf(ph);
    const float frac = __fadd_rn(__fsub_rn(ph, n), rest);
    // times 2^n, -251 <= n <= 0, as products with exact powers of two built
    // from their bits (2^n = 2^(n + 126) 2^-126 below the normal range)
    const int ni = static_cast<int>(n);
    const float r = ex2_approx(frac);
    return ni >= -126 ? __fmul_rn(r, __int_as_float((ni + 127) << 23))
                      : __fmul_rn(__fmul_rn(r, __int_as_float((ni + 253) << 23)), __int_as_float(1 << 23));
}

// ---- float pairs (hi + lo, |lo| <= ulp(hi) / 2): sums of up to a few
// thousand terms with about 44 significant bits, all in float32
struct ff {
    float hi, lo;
};
__device__ __forceinline__ ff ff_norm(float s, float e) {  // |s| >= |e|
    const float hi = __fadd_rn(s, e);
    return {hi, __fsub_rn(e, __fsub_rn(hi, s))};
}
__device__ __forceinline__ ff ff_add(ff a, ff b) {
    const float s = __fadd_rn(a.hi, b.hi);
    const float bv = __fsub_rn(s, a.hi);
    const float err = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bv)), __fsub_rn(b.hi, bv));
    return ff_norm(s, __fadd_rn(err, __fadd_rn(a.lo, b.lo)));
}
__device__ __forceinline__ ff ff_neg(ff a) { return {-a.hi, -a.lo}; }
__device__ __forceinline__ ff ff_mul(ff a, float f) {
    const float p = __fmul_rn(a.hi, f);
    return ff_norm(p, __fmaf_rn(a.lo, f, __fmaf_rn(a.hi, f, -p)));
}
// a / f: the quotient from the hardware reciprocal, then one correction
// step with the exact remainder (f > 0; below 2^-100 the plain division,
// where the reciprocal would overflow or flush)
__device__ __forceinline__ ff ff_div(ff a, float f) {
    const float r = f < 7.9e-31f ? 0.f : rcp_approx(f);
    const float q1 = f < 7.9e-31f ? __fdiv_rn(a.hi, f) : __fmul_rn(a.hi, r);
    const float rem = __fadd_rn(__fmaf_rn(-q1, f, a.hi), a.lo);
    return ff_norm(q1, f < 7.9e-31f ? __fdiv_rn(rem, f) : __fmul_rn(rem, r));
}
__device__ __forceinline__ bool ff_gt(ff a, ff b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }
__device__ __forceinline__ ff ff_shfl(ff a, int src) {
    return {__shfl_sync(0xffffffffu, a.hi, src), __shfl_sync(0xffffffffu, a.lo, src)};
}
// inclusive scan over the lanes, fixed association
__device__ __forceinline__ ff ff_scan(ff v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const ff u = {__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
        if (lane >= o) v = ff_add(u, v);
    }
    return v;
}

// inclusive scan over the lanes in float32, fixed association
__device__ __forceinline__ float warp_scan(float v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v = __fadd_rn(u, v);
    }
    return v;
}

// Larger value, or the lower index among equal values; flags OR-ed; the
// same result lands in every lane.
__device__ __forceinline__ void warp_argmax(float &v, int &idx, int &flag) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, o);
        const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
        flag |= __shfl_xor_sync(0xffffffffu, flag, o);
        if (ov > v || (ov == v && oi < idx)) {
            v = ov;
            idx = oi;
        }
    }
}

// First lane of `pick`, else the highest lane of `pos` (0 if neither: the
// callers only reach a level whose total is positive).
__device__ __forceinline__ int choose(unsigned pick, unsigned pos) {
    if (pick) return __ffs(pick) - 1;
    return pos ? 31 - __clz(pos) : 0;
}

// Node count of sequence b, clamped to [1, Qc].
__device__ __forceinline__ int node_count(const SampleArgs &a, int b) {
    const int n = a.n_nodes[b];
    return n < 1 ? 1 : (n > a.Qc ? a.Qc : n);
}

// R (float4 per lane in a region) is a template parameter so that the
// region passes unroll: every load and exp2 of a lane's run can be in flight
// at once.
template <bool kGreedy, int R>
__global__ void __launch_bounds__(kThreads, 2) tree_sample_kernel(const SampleArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int C = a.C, V = a.V, Qc = a.Qc, NREG = a.nreg, G = a.G;
    const int Q = NREG / kWarps;  // regions per warp per row
    const int g = blockIdx.x / C;
    const int rank = static_cast<int>(cluster_ctarank());
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned full = 0xffffffffu;
    const float kh = a.kh, kl = a.kl;
    const int rtok = R * 128;  // tokens per region
    const long long cta0 = static_cast<long long>(rank) * NREG * rtok;
    float *stages = reinterpret_cast<float *>(smem);  // [warp][stage][rtok]
    float *lscan = stages + kWarps * kStages * rtok;  // [region][32] inclusive scan of the lane sums
    Ctrl &ct = *reinterpret_cast<Ctrl *>(lscan + NREG * 32);

    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&ct.bar[warp][s]), 1);
        mbar_fence_init();
    }
    // ---- the cluster's rows that hold a node, compacted in order (every CTA
    // of the cluster builds the same list); padding slots get their outputs
    // here; each row's uniform is fetched now, not at the end of the row
    {
        const int span = (a.rows_end - a.row0 - g + G - 1) / G;
        int base = 0;
        for (int t0 = 0; t0 < span; t0 += kThreads) {
            const int t = t0 + threadIdx.x;
            const int row = a.row0 + g + t * G;
            bool valid = false;
            int n = 0;
            float u = 0.f;
            if (t < span) {
                const int b = row / Qc;
                n = node_count(a, b);
                valid = row - b * Qc < n;
                if (!kGreedy && valid) u = a.u01[row];
                if (!valid && rank == 0) {
                    a.sample_tok[row] = -1;
                    a.node_p[row] = 0.f;
                }
            }
            const unsigned bal = __ballot_sync(full, valid);
            if (lane == 0) ct.wcount[warp] = __popc(bal);
            __syncthreads();
            int off = base;
            for (int w = 0; w < warp; ++w) off += ct.wcount[w];
            if (valid) {
                const int pos = off + __popc(bal & ((1u << lane) - 1u));
                ct.list_row[pos] = row;
                ct.list_n[pos] = n;
                ct.list_u[pos] = u;
            }
            for (int w = 0; w < kWarps; ++w) base += ct.wcount[w];
            __syncthreads();
        }
        if (threadIdx.x == 0) ct.nlist = base;
        __syncthreads();
    }
    const int nlist = ct.nlist;

    // ---- producer (lane 0 of each warp): this warp's regions of the
    // cluster's rows, in order, two in flight
    int pl = 0, pq = 0;
    uint32_t issued = 0;
    auto issue = [&]() {
        if (pl >= nlist) return;
        const int prow = ct.list_row[pl];
        const int stage = static_cast<int>(issued & 1u);
        const uint32_t bar = smem_u32(&ct.bar[warp][stage]);
        const long long reg0 = cta0 + static_cast<long long>(warp * Q + pq) * rtok;
        const long long left = static_cast<long long>(V) - reg0;
        const int nvalid = left <= 0 ? 0 : (left >= rtok ? rtok : static_cast<int>(left));
        if (nvalid > 0) {
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nvalid) * 4u);
            bulk_load(smem_u32(stages + (warp * kStages + stage) * rtok),
                      a.logits + static_cast<size_t>(prow) * V + reg0, static_cast<uint32_t>(nvalid) * 4u, bar);
        } else {
            mbar_arrive(bar);  // an empty region still completes its phase
        }
        ++issued;
        if (++pq == Q) {
            pq = 0;
            ++pl;
        }
    };
    if (lane == 0) {
        issue();
        issue();
    }
    __syncwarp();
    // every CTA of the cluster is running before any writes into another
    if (C > 1) cluster_sync();

    uint32_t used = 0;  // regions consumed by this warp
    int parity = 0;     // row count parity (publication buffer)
    for (int li = 0; li < nlist; ++li) {
        const int row = ct.list_row[li], n = ct.list_n[li];
        const int b = row / Qc, i = row - b * Qc;
        const size_t tb = static_cast<size_t>(b) * Qc;
        // what the end of the row needs from memory is copied into shared
        // memory while the regions stream (a load left for the end of the row
        // would queue behind the other CTAs' streams): node i's children,
        // their tokens, then (once the tokens are in) their logits (rank 0)
        const float u = ct.list_u[li];
        const int c = threadIdx.x;
        const bool cslot = rank == 0 && c >= 1 && c < n;
        if (cslot) {
            cp_async_4(&ct.cpar[c], a.parent + tb + c);
            cp_async_4(&ct.ctok[c], a.token + tb + c);
        }
        bool child = false, tok_ok = false;
        int c_tok = -1;

        // ---- this warp's regions of the row, in token order: a running
        // maximum W and (sampling) a running float-pair prefix P of the
        // regions' totals in units of 2^((x - W) kd)
        float W = -INFINITY;
        int widx = INT_MAX, wflag = 0;
        ff P = {0.f, 0.f};
        for (int q = 0; q < Q; ++q) {
            const int j = warp * Q + q;
            const int stage = static_cast<int>(used & 1u);
            const long long reg0 = cta0 + static_cast<long long>(j) * rtok;
            const long long left = static_cast<long long>(V) - reg0;
            const int nq = (left <= 0 ? 0 : (left >= rtok ? rtok : static_cast<int>(left))) >> 2;
            int flag = 0;
            if (!wait_bar(smem_u32(&ct.bar[warp][stage]), (used >> 1) & 1u)) flag |= kFlagTimeout;
            // the lane's run into registers (past V: -inf, weight 0), then the
            // stage goes straight back to the producer
            const int q0 = lane * R;  // this lane's first float4 of the region
            const float4 *reg4 = reinterpret_cast<const float4 *>(stages + (warp * kStages + stage) * rtok) + q0;
            float4 x[R];
#pragma unroll
            for (int k = 0; k < R; ++k)
                x[k] = (q0 + k < nq && !(flag & kFlagTimeout)) ? reg4[k]
                                                               : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            __syncwarp();  // every lane has its run
            ++used;
            if (lane == 0) issue();
            if (q == 0 && cslot) {
                cp_async_wait_all();
                child = ct.cpar[c] == i;
                c_tok = ct.ctok[c];
                tok_ok = c_tok >= 0 && c_tok < V;
                if (child && tok_ok && !kGreedy) cp_async_4(&ct.cx[c], a.logits + static_cast<size_t>(row) * V + c_tok);
            }
            // region maximum (NaN-propagating)
            float best = -INFINITY;
#pragma unroll
            for (int k = 0; k < R; ++k)
                best = max_nan3(best, max_nan3(x[k].x, x[k].y, x[k].z), x[k].w);
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                best = max_nan(best, __shfl_xor_sync(full, best, o));
                flag |= __shfl_xor_sync(full, flag, o);
            }
            if (best != best) flag |= kFlagNan;
            if (!kGreedy && best == INFINITY) flag |= kFlagNoDist;
            wflag |= flag;
            if (kGreedy) {
                // its first index: the lanes' first element equal to it, lowest lane
                int bidx = INT_MAX;
#pragma unroll
                for (int k = R - 1; k >= 0; --k) {
                    const int t = static_cast<int>(reg0) + 4 * (q0 + k);
                    bidx = x[k].w == best ? t + 3 : bidx;
                    bidx = x[k].z == best ? t + 2 : bidx;
                    bidx = x[k].y == best ? t + 1 : bidx;
                    bidx = x[k].x == best ? t : bidx;
                }
                bidx = static_cast<int>(__reduce_min_sync(full, static_cast<unsigned>(bidx)));
                if (best > W || (best == W && bidx < widx)) {
                    W = best;
                    widx = bidx;
                }
            } else {
                // weights: quad sums, a sequential sum per lane, a scan over lanes
                float tot = 0.f;
                if (wflag == 0 && best > -INFINITY) {
                    float qs[R];
#pragma unroll
                    for (int k = 0; k < R; ++k) qs[k] = quad_sum(x[k], best, kh, kl);
                    float s = 0.f;
#pragma unroll
                    for (int k = 0; k < R; ++k) s = __fadd_rn(s, qs[k]);
                    const float inc = warp_scan(s, lane);
                    lscan[j * 32 + lane] = inc;
                    const unsigned lp = __ballot_sync(full, s > 0.f);
                    if (lane == 0) ct.lpos[j] = lp;
                    tot = __shfl_sync(full, inc, 31);
                    // into the running prefix (a new maximum rescales it first)
                    if (best > W) {
                        P = ff_mul(P, exp2_diff(W, best, kh, kl));
                        W = best;
                    }
                    P = ff_add(P, ff_mul({tot, 0.f}, exp2_diff(best, W, kh, kl)));
                }
                if (lane == 0) {
                    ct.rmax[j] = best;
                    ct.rtot[j] = tot;
                    ct.rref[j] = W;
                    ct.rp_hi[j] = P.hi;
                    ct.rp_lo[j] = P.lo;
                }
            }
        }
        if (lane == 0) {
            ct.wmax[warp] = W;
            ct.widx[warp] = widx;
            ct.wflag[warp] = wflag;
            ct.wp_hi[warp] = P.hi;
            ct.wp_lo[warp] = P.lo;
        }
        __syncthreads();

        // ---- CTA summary (warp 0): the 8 warps' maxima, their totals scaled
        // to the CTA's maximum and scanned in warp (token) order
        if (warp == 0) {
            const bool wl = lane < kWarps;
            float m = wl ? ct.wmax[lane] : -INFINITY;
            int idx = wl ? ct.widx[lane] : INT_MAX;
            int f = wl ? ct.wflag[lane] : 0;
            const float wm = m;
            warp_argmax(m, idx, f);
            ff total = {0.f, 0.f};
            if (!kGreedy && f == 0 && m > -INFINITY) {
                const float fs = wl ? exp2_diff(wm, m, kh, kl) : 0.f;
                const ff mass = wl ? ff_mul({ct.wp_hi[lane], ct.wp_lo[lane]}, fs) : ff{0.f, 0.f};
                const ff sc = ff_scan(mass, lane);
                if (wl) {
                    ct.wfs[lane] = fs;
                    ct.wmass[lane] = mass.hi;
                    ct.wscan_hi[lane] = sc.hi;
                    ct.wscan_lo[lane] = sc.lo;
                }
                total = ff_shfl(sc, 31);
            }
            // the CTA's summary into every CTA of the cluster
            if (lane < C) {
                st_peer_f32(&ct.xm[parity][rank], lane, m);
                st_peer_f32(&ct.xhi[parity][rank], lane, total.hi);
                st_peer_f32(&ct.xlo[parity][rank], lane, total.lo);
                st_peer_s32(&ct.xidx[parity][rank], lane, idx);
                st_peer_s32(&ct.xflag[parity][rank], lane, f);
            }
        }
        if (C > 1) cluster_sync();
        else __syncthreads();

        // ---- cluster exchange (warp 0 of every CTA computes the same result)
        if (warp == 0) {
            float pm = -INFINITY;
            ff ps = {0.f, 0.f};
            int pi = INT_MAX, pf = 0;
            if (lane < C) {
                pm = ct.xm[parity][lane];
                ps = {ct.xhi[parity][lane], ct.xlo[parity][lane]};
                pi = ct.xidx[parity][lane];
                pf = ct.xflag[parity][lane];
            }
            float M = pm;
            int idx = pi, f = pf;
            warp_argmax(M, idx, f);
            if (!kGreedy && !(M > -INFINITY && M < INFINITY)) f |= kFlagNoDist;
            int cstar = 0;
            ff S = {0.f, 0.f}, t = {0.f, 0.f};
            if (!kGreedy && f == 0) {
                // the CTA holding M has a weight-1 element: S >= 1
                const float fc = lane < C ? exp2_diff(pm, M, kh, kl) : 0.f;
                const ff mass = ff_mul(ps, fc);
                const ff sc = ff_scan(mass, lane);
                S = ff_shfl(sc, 31);
                const ff thr = ff_mul(S, u);
                cstar = choose(__ballot_sync(full, mass.hi > 0.f && ff_gt(sc, thr)), __ballot_sync(full, mass.hi > 0.f));
                const ff pre = ff_shfl(sc, cstar > 0 ? cstar - 1 : 0);
                t = ff_div(ff_add(thr, ff_neg(cstar > 0 ? pre : ff{0.f, 0.f})), __shfl_sync(full, fc, cstar));
            }
            if (lane == 0) {
                ct.row_flag = f;
                ct.row_idx = idx;
                ct.row_m = M;
                ct.row_s = S.hi;
                ct.cstar = cstar;
                ct.t_hi = t.hi;
                ct.t_lo = t.lo;
            }
        }
        __syncthreads();
        const int rflag = ct.row_flag;

        // ---- locate the sample inside the winning CTA (warp 0)
        if (!kGreedy && rflag == 0 && rank == ct.cstar && warp == 0) {
            const ff tc = {ct.t_hi, ct.t_lo};
            // warp: first of positive mass whose scan passes tc, else the last
            // of positive mass
            const bool wpos = lane < kWarps && ct.wmass[lane] > 0.f;
            const bool wpick = wpos && ff_gt({ct.wscan_hi[lane], ct.wscan_lo[lane]}, tc);
            const int wst = choose(__ballot_sync(full, wpick), __ballot_sync(full, wpos));
            const ff pre_w = wst > 0 ? ff{ct.wscan_hi[wst - 1], ct.wscan_lo[wst - 1]} : ff{0.f, 0.f};
            const ff tw = ff_div(ff_add(tc, ff_neg(pre_w)), ct.wfs[wst]);  // units of 2^((x - W) kd)
            const float Ww = ct.wmax[wst];
            // region of the warp: its running prefix, brought to the warp's
            // final maximum
            const int j = wst * Q + lane;
            const bool rl = lane < Q;
            const bool rpos = rl && ct.rtot[j] > 0.f;
            const ff pconv = rl ? ff_mul({ct.rp_hi[j], ct.rp_lo[j]}, exp2_diff(ct.rref[j], Ww, kh, kl)) : ff{0.f, 0.f};
            const int qst = choose(__ballot_sync(full, rpos && ff_gt(pconv, tw)), __ballot_sync(full, rpos));
            const ff pre_q = qst > 0 ? ff_shfl(pconv, qst - 1) : ff{0.f, 0.f};
            const int jst = wst * Q + qst;
            const float mr = ct.rmax[jst];
            const ff tjf = ff_div(ff_add(tw, ff_neg(qst > 0 ? pre_q : ff{0.f, 0.f})), exp2_diff(mr, Ww, kh, kl));
            const float tj = __fadd_rn(tjf.hi, tjf.lo);  // units of 2^((x - rmax) kd)
            // lane: the region's lane scan, among the lanes of nonzero weight
            // (the scan's fixed tree need not rise by an empty lane's zero)
            const float inc = lscan[jst * 32 + lane];
            const unsigned lposm = ct.lpos[jst];
            const bool lpos = (lposm >> lane) & 1u;
            const int lst = choose(__ballot_sync(full, lpos && inc > tj), lposm);
            const float tl = __fsub_rn(tj, lst > 0 ? lscan[jst * 32 + lst - 1] : 0.f);
            // float4 of the lane: its quad sums again, from the logits in
            // memory, and their sequential prefix (the sequence that made the
            // lane sum)
            const long long ltok0 = cta0 + static_cast<long long>(jst) * rtok + 4LL * lst * R;
            const long long mytok = ltok0 + 4LL * lane;
            const bool inb = lane < R && mytok + 4 <= V;
            const float4 v = inb ? *reinterpret_cast<const float4 *>(a.logits + static_cast<size_t>(row) * V + mytok)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            const float own = inb ? quad_sum(v, mr, kh, kl) : 0.f;
            ct.quads[lane] = own;
            __syncwarp();
            float p = 0.f;
#pragma unroll
            for (int k = 0; k < R; ++k) {
                const float qv = ct.quads[k];
                if (k <= lane) p = __fadd_rn(p, qv);
            }
            const int kst = choose(__ballot_sync(full, own > 0.f && p > tl), __ballot_sync(full, own > 0.f));
            const float before = __shfl_sync(full, p, kst > 0 ? kst - 1 : 0);
            const float tk = __fsub_rn(tl, kst > 0 ? before : 0.f);
            if (lane == kst) {
                // element: the float4's own partial sums
                float e[4];
                weight2(v.x, v.y, mr, kh, kl, e[0], e[1]);
                weight2(v.z, v.w, mr, kh, kl, e[2], e[3]);
                float acc = 0.f;
                int pick = -1, lastpos = 0;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    acc = jj == 0 ? e[0] : __fadd_rn(acc, e[jj]);
                    if (e[jj] > 0.f) {
                        lastpos = jj;
                        if (pick < 0 && acc > tk) pick = jj;
                    }
                }
                a.sample_tok[row] = static_cast<int>(mytok) + (pick >= 0 ? pick : lastpos);
            }
        }

        // ---- greedy result, flagged rows, node probabilities (rank 0)
        if (rank == 0) {
            const int idx = ct.row_idx == INT_MAX ? 0 : ct.row_idx;
            if (threadIdx.x == 0) {
                if (rflag != 0) {
                    a.sample_tok[row] = -1;
                    a.status[b] = (rflag & kFlagTimeout) ? DDT_E_TIMEOUT : DDT_E_BADINPUT;
                } else if (kGreedy) {
                    a.sample_tok[row] = idx;
                }
                if (i == 0) a.node_p[tb] = 1.f;
            }
            if (child) {
                cp_async_wait_all();
                const float c_x = ct.cx[c];
                float p = 0.f;
                if (!tok_ok) {
                    a.status[b] = DDT_E_BADINPUT;
                } else if (rflag == 0) {
                    p = kGreedy ? (c_tok == idx ? 1.f : 0.f) : __fdividef(exp2_diff(c_x, ct.row_m, kh, kl), ct.row_s);
                }
                a.node_p[tb + c] = p;
            }
        }
        parity ^= 1;
        __syncthreads();  // the next row overwrites the region summaries
    }
    // (no CTA touches another's shared memory after a row's cluster barrier,
    // so a CTA may leave as soon as its last row is done)
}

size_t smem_bytes(int R, int nreg) {
    return static_cast<size_t>(kWarps * kStages * R * 128 + nreg * 32) * 4 + sizeof(Ctrl);
}

}  // namespace

SamplePlan plan_sample(int V, long long rows, int sms, int max_cluster) {
    SamplePlan p{};
    if (V < 4 || (V & 3) || rows < 1 || rows >= (1LL << 31)) return p;
    // Pick C for the shortest makespan: rows go round-robin over the G = 2 *
    // sms / C clusters that fit at once (two CTAs per SM); a round costs a
    // CTA its share of a row plus the row's fixed synchronisation, counted as
    // the streaming time of about 60 (one CTA) or 120 (a cluster: barrier and
    // exchange on top) 128-token rows. Ties go to the smaller C.
    const long long slots = 2LL * sms;
    double best = 0.0;
    for (int C = 1; C <= max_cluster; C <<= 1) {
        const long long per_cta = (V + C - 1) / C;  // tokens
        if (C > 1 && per_cta < 2048) break;         // too little of a row to split further
        const long long rows128 = (per_cta + 127) / 128;
        // region shape: R odd, 8..128 regions (a multiple of 8); the least
        // capacity past the CTA's share, slightly preferring longer regions
        int bR = 0, bN = 0;
        double bscore = 0.0;
        for (int R = kSampleMaxRows; R >= 1; R -= 2) {
            const long long nreg = (rows128 + 8LL * R - 1) / (8LL * R) * 8;
            if (nreg > kSampleMaxRegions) continue;
            const double score = static_cast<double>(nreg * R) * (1.0 + 0.01 * (kSampleMaxRows - R));
            if (bR == 0 || score < bscore) {
                bscore = score;
                bR = R;
                bN = static_cast<int>(nreg);
            }
        }
        if (bR == 0) continue;
        const long long G = slots / C > 0 ? slots / C : 1;
        const double t = static_cast<double>((rows + G - 1) / G) * static_cast<double>(bN * bR + (C > 1 ? 120 : 60));
        if (p.C == 0 || t < best * 0.999) {
            best = t;
            p.C = C;
            p.R = bR;
            p.nreg = bN;
        }
    }
    if (p.C != 0) p.smem = smem_bytes(p.R, p.nreg);
    return p;
}

namespace {
using SampleKernel = void (*)(SampleArgs);
// [greedy][R / 2] for R = 1, 3, ..., kSampleMaxRows
const SampleKernel kKernels[2][6] = {
    {tree_sample_kernel<false, 1>, tree_sample_kernel<false, 3>, tree_sample_kernel<false, 5>,
     tree_sample_kernel<false, 7>, tree_sample_kernel<false, 9>, tree_sample_kernel<false, 11>},
    {tree_sample_kernel<true, 1>, tree_sample_kernel<true, 3>, tree_sample_kernel<true, 5>,
     tree_sample_kernel<true, 7>, tree_sample_kernel<true, 9>, tree_sample_kernel<true, 11>}};
static_assert(kSampleMaxRows == 11, "one kernel per odd R up to kSampleMaxRows");
}  // namespace

// The largest cluster the sampling kernels may use on the current device (0
// if their attributes could not be set: tried again on the next call), found
// once per device.
int sample_max_cluster() {
    constexpr int kDevices = 64;
    static std::mutex mu;
    static int known[kDevices];  // 0: not yet found
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevices) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (known[dev] > 0) return known[dev];
    const int smem_max = static_cast<int>(smem_bytes(kSampleMaxRows, kSampleMaxRegions));
    for (auto &row : kKernels)
        for (SampleKernel k : row)
            if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max) != cudaSuccess) {
                cudaGetLastError();
                return 0;
            }
    int max_c = 8;
    bool nonportable = true;
    for (auto &row : kKernels)
        for (SampleKernel k : row)
            if (nonportable && cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
                cudaGetLastError();
                nonportable = false;
            }
    if (nonportable) {
        // a cluster of 16 CTAs of the size the 16-CTA plans use
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(16);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem_bytes(kSampleMaxRows, 16);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 16;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kKernels[0][kSampleMaxRows / 2], &cfg) == cudaSuccess && n > 0)
            max_c = 16;
        cudaGetLastError();
    }
    known[dev] = max_c;
    return max_c;
}

cudaError_t launch_tree_sample(const ddt_tree &tree, const float *logits, int V, double kd, const float *u01,
                               int32_t *sample_tok, float *node_p, const SamplePlan &plan, cudaStream_t s) {
    const bool greedy = kd == 0.0;
    if (plan.R < 1 || plan.R > kSampleMaxRows || !(plan.R & 1)) return cudaErrorInvalidValue;
    const SampleKernel kernel = kKernels[greedy ? 1 : 0][plan.R / 2];
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(plan.C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // as many clusters as fit on the device at once (a persistent grid), at
    // most one per row; the occupancy answer is cached per shape
    static std::mutex mu;
    static int cached_c = 0, cached_g = 0, cached_dev = -1;
    static size_t cached_smem = 0;
    int dev = 0, G = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (cached_c == plan.C && cached_smem == plan.smem && cached_dev == dev) {
            G = cached_g;
        } else {
            cfg.gridDim = dim3(static_cast<unsigned>(plan.C));
            if (cudaOccupancyMaxActiveClusters(&G, kKernels[0][plan.R / 2], &cfg) != cudaSuccess || G < 1) {
                cudaGetLastError();
                return cudaErrorInvalidConfiguration;
            }
            cached_c = plan.C;
            cached_smem = plan.smem;
            cached_dev = dev;
            cached_g = G;
        }
    }
    const long long rows = static_cast<long long>(tree.B) * tree.Qc;
    SampleArgs a{};
    a.logits = logits;
    a.u01 = u01;
    a.token = tree.token;
    a.parent = tree.parent;
    a.n_nodes = tree.n_nodes;
    a.sample_tok = sample_tok;
    a.node_p = node_p;
    a.status = tree.status;
    if (!greedy) {
        // kd = kh + kl with kl > 0: kh the largest float below kd
        float kh = static_cast<float>(kd);
        if (static_cast<double>(kh) >= kd) kh = nextafterf(kh, 0.f);
        a.kh = kh;
        a.kl = static_cast<float>(kd - static_cast<double>(kh));
    }
    a.Qc = tree.Qc;
    a.V = V;
    a.C = plan.C;
    a.nreg = plan.nreg;
    // each launch gives a cluster at most kSampleListCap rows
    const long long per_launch = static_cast<long long>(G) * kSampleListCap;
    for (long long r0 = 0; r0 < rows; r0 += per_launch) {
        const long long r1 = r0 + per_launch < rows ? r0 + per_launch : rows;
        a.row0 = static_cast<int>(r0);
        a.rows_end = static_cast<int>(r1);
        a.G = static_cast<int>(r1 - r0 < G ? r1 - r0 : G);
        cfg.gridDim = dim3(static_cast<unsigned>(a.G * plan.C));
        if (cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a)) return e;
    }
    return cudaSuccess;
}

}  // namespace ddt
