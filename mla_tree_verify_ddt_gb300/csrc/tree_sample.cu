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
// Layout of the work. One cluster of C CTAs per row; CTA c holds tokens
// [c * 1024 r, (c + 1) * 1024 r), split into 8 warp regions of r rows of 128
// tokens (a row is one float4 per lane). Each warp fetches its region with
// one bulk copy into shared memory, so the logits are read from HBM once:
//   pass 1  largest logit (and its first index), NaN check, per warp -> CTA;
//   pass 2  weights relative to the CTA's own maximum; per row a sum over the
//           32 lanes in lane order, per warp a prefix over its rows (float32),
//           per CTA a float64 sum over its warps;
//   exchange  each CTA publishes (max, first index, sum) in its shared memory;
//           after a cluster barrier every CTA reads all C summaries through
//           distributed shared memory and computes the same row maximum, the
//           same total and the same winning CTA;
//   locate  the winning CTA descends warp -> row -> lane -> element using the
//           very sums it built in pass 2 (recomputed weights are bit-identical:
//           one fixed sequence of correctly rounded operations), so every level
//           agrees with the level above it up to the rounding of that level's
//           prefix (float32 inside a CTA, float64 across CTAs); a threshold
//           that falls past a level's total takes that level's last nonzero
//           entry.
// Rank 0 of the cluster writes the greedy result and the children's node
// probabilities (the child token's weight against the row maximum over the
// row total). Float64 arithmetic runs only in single threads: its rate on
// this GPU is a small fraction of float32's.
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
constexpr int kRowTokens = 128;           // one float4 per lane
constexpr int kFlagNan = 1, kFlagTimeout = 2;

struct Ctrl {
    uint64_t bar[kWarps];         // one bulk copy per warp region
    float incl[kWarps][32];       // inclusive prefix over each region's row sums
    float rsum[kWarps][32];       // row sums (lane order)
    float wsum[kWarps];           // region totals
    float wmax[kWarps];
    int widx[kWarps];
    int wflag[kWarps];
    // published to the cluster
    double pub_s;
    float pub_m;
    int pub_idx;
    int pub_flag;
    // the row's result, identical in every CTA of the cluster
    int row_flag;                 // kFlag* bits; 4: no distribution
    int row_idx;                  // first index of the largest logit
    int cstar;                    // CTA holding the sample
    float row_m;
    float row_s;                  // the row's total weight (in units of 2^((x - row_m) kd))
    float t_cta;                  // threshold inside CTA cstar, in its own weight units
    double s_c;                   // this CTA's total (float64 sum of the region totals)
    double xps[16];               // the cluster's CTA totals and scales, for one thread
    float xfc[16];
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
    double kd;  // log2(e) / temperature; 0 selects the greedy limit
    int Qc, V, C, r;
};

// Bulk copy global -> this CTA's shared memory, credited to `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t a) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ int ld_cluster_s32(uint32_t a) {
    int v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ double ld_cluster_f64(uint32_t a) {
    double v;
    asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint64_t deadline) {
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, 0)) return true;
        if ((it & 63u) == 63u && globaltimer_ns() > deadline) return false;
    }
}

// Weight of logit x against the reference m: 2^((x - m) kd), kd carried as a
// float pair (kh + kl) so the product keeps about 48 bits of it. Every
// operation is explicitly rounded (no contraction), so the same inputs give
// the same bits wherever this is evaluated.
__device__ __forceinline__ float weight(float x, float m, float kh, float kl) {
    const float d = __fsub_rn(x, m);
    const float arg = __fmaf_rn(d, kh, __fmul_rn(d, kl));
    return x == -INFINITY ? 0.f : ex2_approx(arg);
}

__device__ __forceinline__ void quad_weights(const float4 v, float m, float kh, float kl, float (&e)[4]) {
    e[0] = weight(v.x, m, kh, kl);
    e[1] = weight(v.y, m, kh, kl);
    e[2] = weight(v.z, m, kh, kl);
    e[3] = weight(v.w, m, kh, kl);
}

__device__ __forceinline__ float quad_sum(const float (&e)[4]) {
    return __fadd_rn(__fadd_rn(__fadd_rn(e[0], e[1]), e[2]), e[3]);
}

__device__ __forceinline__ void consider(float x, int j, float &best, int &bidx, int &flag) {
    if (x != x) flag |= kFlagNan;
    else if (x > best) {
        best = x;
        bidx = j;
    }
}

// First set bit of `pick`, else the highest set bit of `pos` (-1 if none).
__device__ __forceinline__ int choose(unsigned pick, unsigned pos) {
    if (pick) return __ffs(pick) - 1;
    return pos ? 31 - __clz(pos) : -1;
}

__global__ void __launch_bounds__(kThreads, 2) tree_sample_kernel(const SampleArgs a) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int r = a.r, C = a.C, V = a.V, Qc = a.Qc;
    const int row = blockIdx.x / C;
    const int rank = static_cast<int>(cluster_ctarank());
    const int b = row / Qc, i = row - b * Qc;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned full = 0xffffffffu;
    int n = a.n_nodes[b];
    n = n < 1 ? 1 : (n > Qc ? Qc : n);
    if (i >= n) {  // a padding slot: the whole cluster leaves before any exchange
        if (rank == 0 && threadIdx.x == 0) {
            a.sample_tok[row] = -1;
            a.node_p[row] = 0.f;
        }
        return;
    }
    const bool greedy = a.kd == 0.0;
    float *data = reinterpret_cast<float *>(smem);
    float *tiles = data + kWarps * r * kRowTokens;
    Ctrl &ct = *reinterpret_cast<Ctrl *>(smem + static_cast<size_t>(r) * 5120);

    // ---- fetch this warp's region
    const long long cta0 = static_cast<long long>(rank) * r * (kWarps * kRowTokens);
    const long long reg0 = cta0 + static_cast<long long>(warp) * r * kRowTokens;
    const long long left = static_cast<long long>(V) - reg0;
    const int nvalid = left <= 0 ? 0 : (left >= r * kRowTokens ? r * kRowTokens : static_cast<int>(left));
    const int nq = nvalid >> 2;
    float *reg = data + warp * r * kRowTokens;
    const float4 *reg4 = reinterpret_cast<const float4 *>(reg);
    const uint32_t bar = smem_u32(&ct.bar[warp]);
    if (lane == 0) {
        mbar_init(bar, 1);
        mbar_fence_init();
        if (nvalid > 0) {
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nvalid) * 4u);
            bulk_load(smem_u32(reg), a.logits + static_cast<size_t>(row) * V + reg0,
                      static_cast<uint32_t>(nvalid) * 4u, bar);
        }
    }
    __syncwarp();
    int flag = 0;
    if (nvalid > 0 && !wait_bar(bar, globaltimer_ns() + kWaitLimitNs)) flag |= kFlagTimeout;

    // ---- pass 1: largest logit, its first index, NaN check
    float best = -INFINITY;
    int bidx = INT_MAX;
    if (!(flag & kFlagTimeout)) {
        for (int k = 0; k < r; ++k) {
            const int q = k * 32 + lane;
            if (q < nq) {
                const float4 v = reg4[q];
                const int j = static_cast<int>(reg0) + 4 * q;
                consider(v.x, j, best, bidx, flag);
                consider(v.y, j + 1, best, bidx, flag);
                consider(v.z, j + 2, best, bidx, flag);
                consider(v.w, j + 3, best, bidx, flag);
            }
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float ob = __shfl_xor_sync(full, best, o);
        const int oi = __shfl_xor_sync(full, bidx, o);
        flag |= __shfl_xor_sync(full, flag, o);
        if (ob > best || (ob == best && oi < bidx)) {
            best = ob;
            bidx = oi;
        }
    }
    if (lane == 0) {
        ct.wmax[warp] = best;
        ct.widx[warp] = bidx;
        ct.wflag[warp] = flag;
    }
    __syncthreads();
    float m_c = -INFINITY;
    int idx_c = INT_MAX, flag_c = 0;
    for (int w = 0; w < kWarps; ++w) {
        const float v = ct.wmax[w];
        const int ix = ct.widx[w];
        flag_c |= ct.wflag[w];
        if (v > m_c || (v == m_c && ix < idx_c)) {
            m_c = v;
            idx_c = ix;
        }
    }

    // ---- pass 2: weights against m_c; row sums in lane order; float64 prefix over rows
    const bool weigh = !greedy && flag_c == 0 && m_c > -INFINITY && m_c < INFINITY;
    float *tile = tiles + warp * r * 32;
    const float kh = static_cast<float>(a.kd);
    const float kl = static_cast<float>(a.kd - static_cast<double>(kh));
    if (weigh) {
        for (int k = 0; k < r; ++k) {
            const int q = k * 32 + lane;
            float s = 0.f;
            if (q < nq) {
                float e[4];
                quad_weights(reg4[q], m_c, kh, kl, e);
                s = quad_sum(e);
            }
            // row k, lane l at column (l + k) mod 32: the row sums below read
            // a different bank in every lane
            tile[k * 32 + ((lane + k) & 31)] = s;
        }
        __syncwarp();
        float s = 0.f;
        if (lane < r) {
            const float *t = tile + lane * 32;
            for (int l = 0; l < 32; ++l) s = __fadd_rn(s, t[(l + lane) & 31]);
        }
        ct.rsum[warp][lane] = s;
        __syncwarp();
        if (lane == 0) {
            float acc = 0.f;
            for (int k = 0; k < r; ++k) {
                acc = __fadd_rn(acc, ct.rsum[warp][k]);
                ct.incl[warp][k] = acc;
            }
            ct.wsum[warp] = acc;
        }
    } else if (lane == 0) {
        ct.wsum[warp] = 0.f;
    }
    __syncthreads();

    // ---- exchange through distributed shared memory (float64 only in
    // single threads: this GPU's float64 rate is low)
    if (threadIdx.x == 0) {
        double s_c = 0.0;
        for (int w = 0; w < kWarps; ++w) s_c = __dadd_rn(s_c, static_cast<double>(ct.wsum[w]));
        ct.s_c = s_c;
        ct.pub_s = s_c;
        ct.pub_m = m_c;
        ct.pub_idx = idx_c;
        ct.pub_flag = flag_c;
    }
    cluster_sync();
    if (warp == 0) {
        float pm = -INFINITY;
        int pi = INT_MAX, pf = 0;
        double ps = 0.0;
        if (lane < C) {
            pm = ld_cluster_f32(mapa_shared(smem_u32(&ct.pub_m), lane));
            pi = ld_cluster_s32(mapa_shared(smem_u32(&ct.pub_idx), lane));
            pf = ld_cluster_s32(mapa_shared(smem_u32(&ct.pub_flag), lane));
            ps = ld_cluster_f64(mapa_shared(smem_u32(&ct.pub_s), lane));
        }
        float M = pm;
        int idx = pi, f = pf;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float ob = __shfl_xor_sync(full, M, o);
            const int oi = __shfl_xor_sync(full, idx, o);
            f |= __shfl_xor_sync(full, f, o);
            if (ob > M || (ob == M && oi < idx)) {
                M = ob;
                idx = oi;
            }
        }
        if (!greedy && !(M > -INFINITY && M < INFINITY)) f |= 4;
        // CTA c's scale 2^((m_c - M) kd): the exponent in float64 (exact
        // difference), its fraction through the hardware exp2, the integer
        // part applied exactly
        float fc = 0.f;
        if (!greedy && f == 0 && lane < C && pm > -INFINITY) {
            const double e = (static_cast<double>(pm) - static_cast<double>(M)) * a.kd;
            const double fl = floor(e);
            fc = fl < -126.0 ? 0.f : ldexpf(ex2_approx(static_cast<float>(e - fl)), static_cast<int>(fl));
        }
        if (lane < C) {
            ct.xfc[lane] = fc;
            ct.xps[lane] = ps;
        }
        __syncwarp();
        if (lane == 0) {
            int cstar = 0;
            float S_f = 0.f, t = 0.f;
            if (!greedy && f == 0) {
                // the CTA holding M has a weight-1 element: S >= 1, and some
                // CTA has positive mass
                double S = 0.0;
                for (int c = 0; c < C; ++c) S = __dadd_rn(S, static_cast<double>(ct.xfc[c]) * ct.xps[c]);
                const double thr = static_cast<double>(a.u01[row]) * S;
                double pre = 0.0, pre_star = 0.0;
                int last = -1, pick = -1;
                for (int c = 0; c < C; ++c) {
                    const double mc = static_cast<double>(ct.xfc[c]) * ct.xps[c];
                    if (mc > 0.0) {
                        last = c;
                        pre_star = pre;
                        if (__dadd_rn(pre, mc) > thr) {
                            pick = c;
                            break;
                        }
                    }
                    pre = __dadd_rn(pre, mc);
                }
                cstar = pick >= 0 ? pick : last;
                t = static_cast<float>((thr - pre_star) / static_cast<double>(ct.xfc[cstar]));
                S_f = static_cast<float>(S);
            }
            ct.row_flag = f;
            ct.row_idx = idx;
            ct.row_m = M;
            ct.row_s = S_f;
            ct.cstar = cstar;
            ct.t_cta = t;
        }
    }
    cluster_arrive_release();  // done reading the other CTAs' shared memory
    __syncthreads();
    const int rflag = ct.row_flag;

    // ---- locate the sample inside the winning CTA
    if (!greedy && rflag == 0 && rank == ct.cstar && warp == 0) {
        const float tc = ct.t_cta;
        // warp region: prefix over the region totals in the order that made s_c
        int wst = -1, lastw = -1;
        float pre = 0.f, prel = 0.f;
        for (int w = 0; w < kWarps; ++w) {
            const float m = ct.wsum[w];
            if (m > 0.f) {
                lastw = w;
                prel = pre;
                if (__fadd_rn(pre, m) > tc) {
                    wst = w;
                    break;
                }
            }
            pre = __fadd_rn(pre, m);
        }
        if (wst < 0) wst = lastw < 0 ? 0 : lastw;  // (lastw >= 0: this CTA's total is positive)
        const float tw = __fsub_rn(tc, prel);
        // row: incl[k] = incl[k-1] + rsum[k], exactly as pass 2 built it
        const float rs = lane < r ? ct.rsum[wst][lane] : 0.f;
        const float inc = lane < r ? ct.incl[wst][lane] : 0.f;
        const int kst =
            max(0, choose(__ballot_sync(full, rs > 0.f && inc > tw), __ballot_sync(full, rs > 0.f)));
        const float tk = __fsub_rn(tw, kst > 0 ? ct.incl[wst][kst - 1] : 0.f);
        // lane: prefix over lanes in lane order, the sequence that made rsum[kst]
        const float *t = tiles + wst * r * 32 + kst * 32;
        float p = 0.f, own = 0.f;
        for (int l = 0; l < 32; ++l) {
            const float v = t[(l + kst) & 31];
            if (l <= lane) p = __fadd_rn(p, v);
            if (l == lane) own = v;
        }
        const int lst = max(0, choose(__ballot_sync(full, own > 0.f && p > tk), __ballot_sync(full, own > 0.f)));
        const float before = __shfl_sync(full, p, lst > 0 ? lst - 1 : 0);
        const float tl = __fsub_rn(tk, lst > 0 ? before : 0.f);
        if (lane == 0) {
            // element: the float4's own partial sums
            const int q = kst * 32 + lst;
            const float4 v = reinterpret_cast<const float4 *>(data + wst * r * kRowTokens)[q];
            float e[4];
            quad_weights(v, m_c, kh, kl, e);
            float acc = 0.f;
            int pick = -1, lastpos = -1;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc = j == 0 ? e[0] : __fadd_rn(acc, e[j]);
                if (e[j] > 0.f) {
                    lastpos = j;
                    if (pick < 0 && acc > tl) pick = j;
                }
            }
            const int j = pick >= 0 ? pick : (lastpos >= 0 ? lastpos : 0);
            a.sample_tok[row] = static_cast<int>(cta0) + wst * r * kRowTokens + 4 * q + j;
        }
    }

    // ---- greedy result, flagged rows, node probabilities (rank 0)
    if (rank == 0) {
        const size_t tb = static_cast<size_t>(b) * Qc;
        const int idx = ct.row_idx == INT_MAX ? 0 : ct.row_idx;
        if (threadIdx.x == 0) {
            if (rflag != 0) {
                a.sample_tok[row] = -1;
                a.status[b] = (rflag & kFlagTimeout) ? DDT_E_TIMEOUT : DDT_E_BADINPUT;
            } else if (greedy) {
                a.sample_tok[row] = idx;
            }
            if (i == 0) a.node_p[tb] = 1.f;
        }
        const int c = threadIdx.x;
        if (c >= 1 && c < n && a.parent[tb + c] == i) {
            const int tk = a.token[tb + c];
            float p = 0.f;
            if (tk < 0 || tk >= V) {
                a.status[b] = DDT_E_BADINPUT;
            } else if (rflag == 0) {
                if (greedy) {
                    p = tk == idx ? 1.f : 0.f;
                } else {
                    const float x = a.logits[static_cast<size_t>(row) * V + tk];
                    p = __fdiv_rn(weight(x, ct.row_m, kh, kl), ct.row_s);
                }
            }
            a.node_p[tb + c] = p;
        }
    }
    cluster_wait();  // no CTA leaves while another may still read its summary
}

}  // namespace

SamplePlan plan_sample(int V, long long rows, int sms, int max_cluster) {
    SamplePlan p{0, 0, 0};
    if (V < 4 || (V & 3) || rows < 1) return p;
    int C = 1;
    // about 20K tokens (80 KB) per CTA; more CTAs when few rows would leave SMs idle
    while (C < max_cluster && static_cast<long long>(C) * 20480 < V) C <<= 1;
    while (C < max_cluster && rows * C < sms && static_cast<long long>(C) * 2048 <= V) C <<= 1;
    int r = static_cast<int>((V + C * 1024LL - 1) / (C * 1024LL));
    while (r > kSampleMaxRows && C < max_cluster) {
        C <<= 1;
        r = static_cast<int>((V + C * 1024LL - 1) / (C * 1024LL));
    }
    if (r > kSampleMaxRows || rows * C >= (1LL << 31)) return p;
    p.C = C;
    p.r = r;
    p.smem = static_cast<size_t>(r) * 5120 + sizeof(Ctrl);
    return p;
}

int sample_max_cluster() {
    static std::once_flag once;
    static int max_c = 0;
    std::call_once(once, [] {
        const size_t smem_max = static_cast<size_t>(kSampleMaxRows) * 5120 + sizeof(Ctrl);
        if (cudaFuncSetAttribute(tree_sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem_max)) != cudaSuccess)
            return;
        max_c = 8;
        if (cudaFuncSetAttribute(tree_sample_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess) {
            cudaGetLastError();
            return;
        }
        // a cluster of 16 CTAs of the largest size this library launches
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(16);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = static_cast<size_t>(10) * 5120 + sizeof(Ctrl);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 16;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, tree_sample_kernel, &cfg) == cudaSuccess && n > 0) max_c = 16;
        cudaGetLastError();
    });
    return max_c;
}

cudaError_t launch_tree_sample(const ddt_tree &tree, const float *logits, int V, double kd, const float *u01,
                               int32_t *sample_tok, float *node_p, const SamplePlan &plan, cudaStream_t s) {
    SampleArgs a{};
    a.logits = logits;
    a.u01 = u01;
    a.token = tree.token;
    a.parent = tree.parent;
    a.n_nodes = tree.n_nodes;
    a.sample_tok = sample_tok;
    a.node_p = node_p;
    a.status = tree.status;
    a.kd = kd;
    a.Qc = tree.Qc;
    a.V = V;
    a.C = plan.C;
    a.r = plan.r;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(static_cast<long long>(tree.B) * tree.Qc * plan.C));
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
    return cudaLaunchKernelEx(&cfg, tree_sample_kernel, a);
}

}  // namespace ddt
