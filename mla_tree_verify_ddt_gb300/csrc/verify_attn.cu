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
// Design. A cluster of two CTAs (ranks r = 0, 1) owns 128 (node, head) rows
// of one sequence and one range of its keys. All rows share the sequence's
// KV, so one 64-key KV tile feeds 128 rows.
//  * Split along the 576-wide contraction: CTA r holds the query columns of
//    latent dims [256r, 256r+256) and rotary dims [32r, 32r+32), loads the
//    same columns of every KV tile, and computes a partial S (M=128 rows,
//    N=64 keys, K=288) into tensor memory. Its 256 latent KV columns are also
//    the V of its half of the output, so O += P V (M=128, N=256, K=64) needs
//    no further load. Nothing is loaded or multiplied twice and each CTA
//    keeps only part of Q and half of each KV row (36 KB per 64-key tile) in
//    shared memory: four latent tiles in flight, and two of the small
//    rotary parts (free as soon as their S is done).
//  * Tensor memory: O (256 columns) and four S/P buffers of 64 columns; the
//    query is in shared memory. Each thread overwrites its own lane of S with
//    the P of that tile once it has read S, so S and P share buffers and a
//    buffer is reused four tiles later, after its PV.
//  * Four shipper warps send each tile's partial S to the partner as soon as
//    it is done, block-scaled to 16 bits per score, with st.async (bytes
//    credited to the partner's mbarrier on arrival) into a ring of two
//    half-tile units, and leave the same scaled values in place of their own
//    partial. Each softmax thread adds the partner's unit to its own. Both
//    CTAs then hold the same full S and run the same softmax, each for its
//    own half of O: no probabilities cross the cluster.
//  * Softmax in fp32, log2 domain, two threads per row: lanes t and t+16 of
//    one warp read the same tensor-memory lane (the 16x32bx2 access shape),
//    32 keys each, and combine their tile max and, at the end, their row sums
//    with one shuffle; visibility as one 32-bit word per half tile (all ones
//    inside the prefix). Scores stay unscaled until the
//    exponent's FFMA (the scale is positive); packed float32x2 arithmetic.
//    The reference max moves lazily: O is rescaled only when a row's max
//    grows by more than 8 (log2 units), so probabilities stay <= 256.
//  * P goes to the tensor core as two bf16 terms, hi = bf16(p) and
//    lo = bf16(p - hi), each an A operand from tensor memory against the same
//    bf16 V; together they carry p to about 2^-17 relative.
//  * KV rows past the last node may hold anything; the tail tile's V rows
//    there are zeroed in shared memory before the PV product reads them.
//  * When the key range is split over several clusters, each writes a
//    normalised partial and its lse; a second kernel merges them (and, inside
//    the verify step, also runs the accept walk).
// Every on-chip wait is bounded; on expiry the CTA records DDT_E_TIMEOUT in
// the sequence's status word, drains its own copies and MMAs and leaves.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "accept_walk.cuh"
#include "ddt_internal.h"
#include "ddt_ptx.cuh"

namespace ddt {
namespace {

constexpr int kRows = 128;          // rows per cluster (MMA M)
constexpr int kKeys = 64;           // keys per tile (S MMA N)
constexpr int kQChunks = 4;         // latent query/KV chunks per CTA: 4 x 64 columns
constexpr int kQSmemChunks = 4;     // the query's latent chunks, in shared memory
constexpr int kChunkBytesQ = kRows * 128;    // 64 bf16 x 128 rows, 128-byte swizzle
constexpr int kChunkBytesKV = kKeys * 128;   // 64 bf16 x 64 keys
constexpr int kKRopeBytes = kKeys * 64;      // 32 bf16 x 64 keys, 64-byte swizzle
constexpr int kQRopeBytes = kRows * 64;      // 32 bf16 x 128 rows, 64-byte swizzle
constexpr int kLatBytes = kQChunks * kChunkBytesKV;  // 32768: a tile's latent keys (and its V)
constexpr int kTileBytes = kLatBytes + kKRopeBytes;  // 36864: a tile's bytes in shared memory
constexpr int kSlots = 4;           // latent KV tiles in flight
constexpr int kSPBufs = 4;          // S / P buffers in tensor memory
constexpr int kRopeSlots = 2;       // rotary key tiles in flight: the slot of tile j (j % 2) is
                                    // free again once S of tile j - 2 is done
// The partner's partial S arrives in units of one key half of a tile (128
// rows x 32 keys) in a ring of two units (tile j's key half h is unit
// 2j + h, slot h). A unit row is block-scaled: 32 16-bit
// integers q (offset by 32768) and the scale d, the score being q d (see
// quantize_unit); the 16-byte groups of the 128 rows come first, then the
// rows' scales.
constexpr int kSXMantBytes = kRows * 64;                  // 8192
constexpr int kSXUnitBytes = kSXMantBytes + kRows * 4;    // 8704
constexpr int kSXUnits = 2;

// shared memory map (offsets from the dynamic shared memory base, which is
// 1024-aligned: checked at run time)
constexpr int kOffQ = 0;
constexpr int kOffQR = kOffQ + kQSmemChunks * kChunkBytesQ;       // 65536: rotary query
constexpr int kOffRing = kOffQR + kQRopeBytes;                    // 73728: latent ring
constexpr int kOffRope = kOffRing + kSlots * kLatBytes;           // 204800: rotary ring
constexpr int kOffSX = kOffRope + kRopeSlots * kKRopeBytes;       // 212992: exchange ring
constexpr int kOffBar = kOffSX + kSXUnits * kSXUnitBytes;         // 230400: barriers and flags (288 B)
constexpr int kOffTree = kOffBar + 288;                           // 230688: the tree as this CTA needs it
constexpr int kMaxTileNodes = DDT_MAX_BUDGET + 1;                 // nodes a 128-row tile can span (<= Qc)
constexpr int kTreeBytes = 16 + kMaxTileNodes * 16;               // node count, then 2 mask words per node
constexpr int kSmemBytes = kOffTree + kTreeBytes;
static_assert(kOffRing % 1024 == 0 && kOffQR % 1024 == 0 && kOffRope % 512 == 0, "swizzle atom alignment");
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
constexpr int kOutBoxBytes = kRows * 128;                         // output staging: 128 rows x 32 fp32
static_assert(8 * kOutBoxBytes <= kSlots * kLatBytes, "output staging must fit in the latent ring");

// tensor memory columns
constexpr uint32_t kColO = 0;       // 256: this CTA's half of O
constexpr uint32_t kColSP = 256;    // 4 x 64: partial S of a tile, overwritten in place (lane by
                                    // lane, once read) by its P: 32 hi words then 32 lo words
constexpr uint32_t kTmemCols = 512;
static_assert(kColSP + kSPBufs * 64 <= kTmemCols, "tensor memory");

constexpr float kRescaleThreshold = 8.0f;  // log2 units
// warps 0-7 softmax group (two threads per row), 8 TMA producer, 9 S-MMA
// issuer (and tensor-memory owner), 10 tree fetch (it waits for the tree
// build, which stalls its whole warp), 11 PV-MMA issuer, 12-15 partial-S
// shippers (warp 12 + q: rows 32q..32q+31, its tensor-memory lane quadrant).
// A thread issues one tcgen05.mma every ~46 cycles at most, which is slower
// than an N=64 S MMA executes; two issuing threads keep the tensor pipe fed
// (S and PV share it).
constexpr int kThreads = 512;
constexpr int kProducerWarp = 8, kMmaWarp = 9, kTreeWarp = 10, kPvWarp = 11, kShipWarp0 = 12;

enum {
    BAR_Q_FULL = 0,      // the query (latent chunks and rotary part) is in shared memory
    BAR_RING_FULL = 1,   // kSlots
    BAR_RING_EMPTY = 5,  // kSlots
    BAR_S_FULL = 9,      // kSPBufs
    BAR_P_FULL = 13,     // kSPBufs
    BAR_PV_DONE = 17,    // kSPBufs
    BAR_O_FINAL = 21,
    BAR_DRAIN = 22,      // the S issuer's MMAs, after a failure
    BAR_TREE = 23,       // the tree's node count and this tile's node masks are in shared memory
    BAR_DRAIN_PV = 24,   // the PV issuer's MMAs, after a failure
    BAR_S_READ = 25,     // kSPBufs: the shippers have sent S of the buffer and left its block-scaled values
    // exchange ring, one barrier per unit slot
    BAR_SX_FULL = 29,    // kSXUnits: the partner's unit is in my slot (its bytes come from the partner)
    BAR_SX_EMPTY = 31,   // kSXUnits: the partner has read the unit my shippers wrote into its slot
    NUM_BARS = 33
};
static_assert(NUM_BARS * 8 + 12 <= kOffTree - kOffBar, "barrier region");
static_assert(BAR_SX_EMPTY + kSXUnits == NUM_BARS, "barrier numbering");

// arrival count of barrier i (see the enum); with a block-table cache the
// ring is filled by the 64 lanes of two gather warps instead of TMA
__device__ __forceinline__ uint32_t bar_count(int i, bool gathered) {
    if (gathered && i >= BAR_RING_FULL && i < BAR_RING_FULL + kSlots) return 64;  // two gather warps
    if (i >= BAR_P_FULL && i < BAR_P_FULL + kSPBufs) return 8;                            // one per softmax warp
    if (i >= BAR_S_READ && i < BAR_S_READ + kSPBufs) return 4;                          // one per shipper warp
    if (i >= BAR_SX_EMPTY && i < BAR_SX_EMPTY + kSXUnits) return kRows;  // the partner's threads of one key half
    return 1;  // one arrival (SX_FULL: the arming thread; its bytes come from the partner's st.async)
}

struct AttnArgs {
    int B, Qc, W, H, Tcap, nsplit;
    const uint64_t *mask;
    const int32_t *n_nodes;
    const int32_t *prefix_len;
    int32_t *status;
    float *o_dst;            // [nsplit][rows_total][512] (nsplit == 1: the final output)
    float *lse_dst;          // [nsplit][rows_total]
    size_t rows_total;       // B * Qc * H
    float scale_log2;        // scale * log2(e)
    unsigned long long wait_ns;
    // block-table cache: key position p of sequence b is row kv_index[b*Tcap + p]
    // of the pools c_kv [pool_rows][512] and k_rope [pool_rows][64]; null for
    // the contiguous cache read by TMA
    const int32_t *kv_index;
    const uint8_t *pool_kv;
    const uint8_t *pool_kr;
    int pool_rows;
    // the output is stored as bfloat16 (only when the key range is not split;
    // split partials stay float32 and the merge kernel rounds)
    int out_bf16;
};

// Visibility of keys key0..key0+31 (half a tile) for a node with ancestor
// mask (m0, m1), as a 32-bit word (bit k: key key0+k): every prefix key
// (< T) and the keys T+m of its ancestors-or-self m < n. Only tiles that reach
// past the prefix need it (key0 + 32 > T). With o = key0 - T, bit k is a
// prefix key for k < -o, else node o+k: bits o..o+31 of the 128-bit mask,
// kept for nodes below n. Shifts instead of a per-key loop (which cost the
// one sequence range holding the nodes about 1.9 us on the single-stream
// workload).
__device__ __noinline__ uint32_t half_tile_visibility(int key0, int T, int n, uint64_t m0, uint64_t m1) {
    const int o = key0 - T;  // > -32
    const uint32_t pre = o < 0 ? (1u << (-o)) - 1u : 0u;
    uint64_t w;
    if (o < 0) w = m0 << (-o);
    else if (o == 0) w = m0;
    else if (o < 64) w = (m0 >> o) | (m1 << (64 - o));
    else if (o < 128) w = m1 >> (o - 64);
    else w = 0;
    const int lim = n - o;  // keys k < lim are nodes below n
    const uint32_t valid = lim >= 32 ? ~0u : (lim > 0 ? (1u << lim) - 1u : 0u);
    return pre | (static_cast<uint32_t>(w) & valid);
}

// The epilogue's staging of one 32-column chunk c (0..3) of a thread's 128
// output columns (tensor-memory columns o_col + 128 half + 32c .. +31 of its
// lane, read with the 16x32bx2 shape whose second range starts 128 columns
// on; times inv_l, or zeros) in the KV ring as the boxes the tensor store
// reads: 128-row x 32-column float32 boxes (box 4 half + c), or 128-row x
// 64-column bfloat16 boxes (box 2 half + c/2, its half c%2), rounded to
// nearest even, in the 128-byte swizzle (16-byte group j of row r at
// j ^ (r % 8)). Written this way each warp store is conflict-free, where
// direct row-strided global stores cost a transaction per lane. Out of line,
// so its temporaries do not weigh on the register allocation of the kernel's
// main loop.
__device__ __noinline__ void stage_chunk(uint32_t o_col, uint8_t *ring, int half, int row, bool zero_row,
                                         float inv_l, bool bf16, int c) {
    uint32_t o[32];
    tmem_ld16x2_32<128>(o_col + c * 32, o);
    tmem_wait_ld();
    if (!bf16) {
        uint8_t *box_row = ring + (half * 4 + c) * kOutBoxBytes + row * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 v = zero_row ? make_float4(0.f, 0.f, 0.f, 0.f)
                                      : make_float4(__uint_as_float(o[4 * j]) * inv_l,
                                                    __uint_as_float(o[4 * j + 1]) * inv_l,
                                                    __uint_as_float(o[4 * j + 2]) * inv_l,
                                                    __uint_as_float(o[4 * j + 3]) * inv_l);
            *reinterpret_cast<float4 *>(box_row + ((j ^ (row & 7)) << 4)) = v;
        }
    } else {
        uint8_t *box_row = ring + (half * 2 + (c >> 1)) * kOutBoxBytes + row * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t w[4];
#pragma unroll
            for (int v = 0; v < 4; ++v)
                w[v] = zero_row ? 0u
                                : pack_bf16x2(__uint_as_float(o[8 * j + 2 * v]) * inv_l,
                                              __uint_as_float(o[8 * j + 2 * v + 1]) * inv_l);
            const int grp = (c & 1) * 4 + j;
            *reinterpret_cast<uint4 *>(box_row + ((grp ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// Partial scores cross the cluster block-scaled: the 32 scores x_k of a row
// and key half with m = max |x_k| become q_k = round(x_k 32767 / m), integers
// in [-32767, 32767], sent as q_k + 32768 in 16 bits, and the scale
// d = m / 32767; the score used is q_k d (float32 products). The CTA that
// owns the scores uses the same q_k d in place of its own, so both CTAs add
// the same two terms. |x_k - q_k d| <= m / 65534 (plus float32 rounding), and
// the keys that decide a softmax have the largest scores, for which that is
// the float32 value rounded to about 16 significant bits. (The scale factor
// 32767 / m may be approximate: |x_k| 32767 / m stays below 32767.5, and the
// products use d alone.) q_k + 32768 is the low 16 bits of the float32
// x_k (32767 / m) + 2^23 + 2^15, a number in [2^23, 2^24) rounded to an
// integer by the fused multiply-add, whose high 16 bits are 0x4B00; the
// receiver rebuilds that float from the 16 bits and subtracts 2^23 + 2^15
// exactly.
constexpr float kQBias = 8421376.0f;  // 2^23 + 2^15

// The 32 partial scores x (float32 patterns) of a row and key half: their
// packed 16-bit codes (value 2p in the low half of word p) and their scale.
// The maximum is taken as a tree (a chain of 32 dependent maxima would cost
// its full latency).
__device__ __forceinline__ float quantize_unit(const uint32_t (&x)[32], uint32_t (&code)[16]) {
    float a[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) a[k] = fmaxf(fabsf(__uint_as_float(x[2 * k])), fabsf(__uint_as_float(x[2 * k + 1])));
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
        for (int k = 0; k < w; ++k) a[k] = fmaxf(a[k], a[k + w]);
    const float m = a[0];
    const float c = m > 1e-30f ? __fdividef(32767.0f, m) : 0.f;
#pragma unroll
    for (int p = 0; p < 16; ++p) {
        float y0, y1;
        fma_f32x2(__uint_as_float(x[2 * p]), __uint_as_float(x[2 * p + 1]), c, kQBias, y0, y1);
        code[p] = __byte_perm(__float_as_uint(y0), __float_as_uint(y1), 0x5410);
    }
    return m * (1.0f / 32767.0f);
}

// The two values q d of code word w (scale d).
__device__ __forceinline__ void dequantize_pair(uint32_t w, float d, float &v0, float &v1) {
    float q0, q1;
    sub_f32x2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7610)), __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7632)),
              kQBias, kQBias, q0, q1);
    mul_f32x2(q0, q1, d, d, v0, v1);
}

// kPaged: the instantiation launched for a block-table cache (a.kv_index set),
// whose gather warps read the block table two tiles ahead; the contiguous
// instantiation runs the tensor-map loads.
template <bool kPaged>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    verify_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qr,
                       const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_kr,
                       const __grid_constant__ CUtensorMap tm_o, const AttnArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int mt = blockIdx.x >> 1;
    const uint32_t rank = cluster_ctarank();  // == blockIdx.x & 1
    const uint32_t peer = rank ^ 1u;
    const int chunk = blockIdx.y;
    const int b = blockIdx.z;

    // ---- per-sequence key range (uniform over the cluster). The two loads
    // are issued here and first used after the barrier / tensor-memory /
    // cluster setup below, which hides their latency.
    const int T_in = a.prefix_len[b];
    uint8_t *smem = smem_raw;
    const uint32_t sbase = smem_u32(smem);
    // The swizzled operand layouts need a 1024-aligned base, which the
    // declaration asks for; shared memory has no room to align it here.
    if (sbase & 1023u) {
        if (tid == 0 && rank == 0 && mt == 0 && chunk == 0) a.status[b] = DDT_E_CUDA;
        return;
    }
    const uint32_t sQ = sbase + kOffQ, sQR = sbase + kOffQR, sRing = sbase + kOffRing, sRope = sbase + kOffRope;
    const uint32_t sBar = sbase + kOffBar;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffBar + NUM_BARS * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffBar + NUM_BARS * 8 + 4);
    // (the word after it is a scratch target for dependency stores)
    auto bar = [&](int i) { return sBar + 8u * static_cast<uint32_t>(i); };

    // Setup. The producer warp initialises the barriers (one per lane) and
    // starts the query load at once; the MMA warp allocates tensor memory
    // meanwhile. A CTA barrier publishes both locally. The cluster barrier
    // that makes this CTA's barriers safe for the partner to touch is only
    // arrived on here (relaxed: the init fence already releases the inits);
    // the softmax threads wait on it just before their first remote store.
    if (warp == kProducerWarp) {
        for (int i = lane; i < NUM_BARS; i += 32) mbar_init(bar(i), bar_count(i, a.kv_index != nullptr));
        if (lane == 0) *abort_flag = 0;
        mbar_fence_init();
        __syncwarp();
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_kv);
            tma_prefetch_desc(&tm_kr);
            tma_prefetch_desc(&tm_qr);
            const int qrow = b * a.Qc * a.H + mt * kRows;
            mbar_arrive_expect_tx(bar(BAR_Q_FULL), kQSmemChunks * kChunkBytesQ + kQRopeBytes);
            for (int c = 0; c < kQSmemChunks; ++c)
                tma_load_2d(sQ + c * kChunkBytesQ, &tm_q, static_cast<int>(rank) * 256 + c * 64, qrow,
                            bar(BAR_Q_FULL));
            tma_load_2d(sQR, &tm_qr, static_cast<int>(rank) * 32, qrow, bar(BAR_Q_FULL));
        }
    } else if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_arrive_relaxed();
    const uint32_t tmem = *tmem_slot;
    const uint64_t deadline = globaltimer_ns() + a.wait_ns;
    // Key ranges are cut from the prefix length and the node capacity alone,
    // not from the tree's node count. The tiles wholly inside the prefix are
    // then known at once and can be streamed while the previous kernel (the
    // tree build, under programmatic dependent launch) is still running; the
    // tree is read between the two phases of each role's tile loop: the
    // tiles known without it, then the rest.
    const int T = T_in;
    const bool t_ok = T >= 0 && T < a.Tcap;
    const int kcap = t_ok ? (a.Tcap - T < a.Qc ? a.Tcap : T + a.Qc) : 0;
    const int ntiles = (kcap + kKeys - 1) / kKeys;
    const int t0 = static_cast<int>((static_cast<long long>(ntiles) * chunk) / a.nsplit);
    const int t1 = static_cast<int>((static_cast<long long>(ntiles) * (chunk + 1)) / a.nsplit);
    const int nrange = t1 - t0;
    const int rows_seq = a.Qc * a.H;
    const size_t row_base = static_cast<size_t>(b) * rows_seq;
    float *o_dst = a.o_dst + static_cast<size_t>(chunk) * a.rows_total * 512;
    float *lse_dst = a.lse_dst + static_cast<size_t>(chunk) * a.rows_total;

    auto fail = [&]() {
        *abort_flag = 1;
        grid_dep_wait();  // after the tree build's own status write
        a.status[b] = DDT_E_TIMEOUT;
    };

    // Known once the tree is: the node count, whether prefix + nodes fit the
    // key capacity, and the sequence's key end. Only the softmax needs them
    // (for tiles that reach past the prefix, and at the end); the tree-fetch
    // warp copies the node count and the ancestor masks of this tile's nodes
    // into shared memory once the tree build has finished. Tiles of the range
    // past the key end (at most one, when the tree is not full) are processed
    // fully masked.
    const volatile int *tree_n = reinterpret_cast<const volatile int *>(smem + kOffTree);
    const uint64_t *tree_mask = reinterpret_cast<const uint64_t *>(smem + kOffTree + 16);
    const int node_lo = (mt * kRows) / a.H;  // first node of the tile's rows
    int n = 1, kend = 0;
    bool seq_ok = false, resolved = false;
    // (tree_ready false: a bounded wait for the tree ran out; the CTA stops)
    auto resolve = [&](bool tree_ready, int n_in) {
        if (!tree_ready) fail();
        n = n_in < 1 ? 1 : (n_in > a.Qc ? a.Qc : n_in);
        seq_ok = tree_ready && t_ok && static_cast<long long>(T) + n <= a.Tcap;
        kend = seq_ok ? T + n : 0;
        resolved = true;
    };


    // Block-table cache: each tile's 64 keys come from arbitrary pool rows.
    // Two warps (the producer and, after its fetch, the tree warp; on
    // different SM sub-partitions) each copy 32 of them, 16 bytes per lane,
    // one key's contiguous half-row per instruction, into the same swizzled
    // layout the tensor-map loads produce; each lane arrives on the slot's
    // barrier once its copies have landed. Block-table entries are checked for
    // keys below the sequence's key end (the tree is known first); a bad entry
    // reads row 0 and flags the sequence; entries past the key end are not
    // used for anything.
    auto gather_keys = [&](int k_lo) {
        grid_dep_wait();
        const int n_g = a.n_nodes[b] < 1 ? 1 : (a.n_nodes[b] > a.Qc ? a.Qc : a.n_nodes[b]);
        const int kend_g = (t_ok && static_cast<long long>(T) + n_g <= a.Tcap) ? T + n_g : 0;
        const int32_t *kvi = a.kv_index + static_cast<size_t>(b) * a.Tcap;
        bool ok = true, bad_index = false;
        // Block-table entries are loaded two tiles ahead and checked only
        // when their tile is copied, so a load's latency overlaps the slot
        // waits instead of sitting between a slot's release and its copies.
        auto entry = [&](int jj) {
            const int key = (t0 + jj) * kKeys + k_lo + lane;
            return (jj < nrange && key < a.Tcap) ? kvi[key] : 0;
        };
        int e_next = 0, e_next2 = 0;
        if constexpr (kPaged) {
            e_next = entry(0);
            e_next2 = entry(1);
        }
        for (int jj = 0; jj < nrange; ++jj) {
            const int slot = jj % kSlots, use = jj / kSlots, rs = jj % kRopeSlots;
            if (!__all_sync(0xffffffffu,
                            (use < 1 || mbar_wait(bar(BAR_RING_EMPTY + slot), (use - 1) & 1, deadline, abort_flag)) &&
                                (jj < kRopeSlots || mbar_wait(bar(BAR_S_FULL + (jj - kRopeSlots) % kSPBufs),
                                                              ((jj - kRopeSlots) / kSPBufs) & 1,
                                                              deadline, abort_flag)))) {
                ok = false;
                break;
            }
            const uint32_t dst = sRing + slot * kLatBytes, rdst = sRope + rs * kKRopeBytes;
            // pool row of key k_lo + lane of the tile
            const int key = (t0 + jj) * kKeys + k_lo + lane;
            int phys;
            if constexpr (kPaged) {
                phys = e_next;
                e_next = e_next2;
                e_next2 = entry(jj + 2);
            } else {
                phys = key < a.Tcap ? kvi[key] : 0;
            }
            if (phys < 0 || phys >= a.pool_rows) {
                if (key < kend_g) bad_index = true;
                phys = 0;
            }
            // latent half-rows: lane l copies its 16 bytes (4 chunks x 8
            // groups, 128-byte swizzle)
#pragma unroll 4
            for (int i = 0; i < 32; ++i) {
                const int r = k_lo + i;
                const int pr = __shfl_sync(0xffffffffu, phys, i);
                cp_async_16(dst + (lane >> 3) * kChunkBytesKV + r * 128 + (((lane & 7) ^ (r & 7)) << 4),
                            a.pool_kv + static_cast<size_t>(pr) * 1024 + rank * 512 + lane * 16);
            }
            // rotary rows: 8 keys per instruction, 4 lanes each (64-byte swizzle)
#pragma unroll
            for (int i0 = 0; i0 < 32; i0 += 8) {
                const int i = i0 + (lane >> 2), q = lane & 3, r = k_lo + i;
                const int pr = __shfl_sync(0xffffffffu, phys, i);
                cp_async_16(rdst + r * 64 + ((q ^ ((r >> 1) & 3)) << 4),
                            a.pool_kr + static_cast<size_t>(pr) * 128 + rank * 64 + q * 16);
            }
            cp_async_arrive_noinc(bar(BAR_RING_FULL + slot));
        }
        if (!ok && lane == 0) fail();
        if (__any_sync(0xffffffffu, bad_index) && lane == 0) a.status[b] = DDT_E_BADINPUT;
        cp_async_wait_all();  // every copy has landed before the CTA can leave
    };

    bool stored = false;  // this thread issued tensor stores of the output block
    if (nrange <= 0) {
        // nothing visible in this range: zero rows (this CTA's half), lse = -inf
        // (this CTA's 256 columns of a row: 64 float4, or 32 uint4 of bfloat16)
        const int per_row = a.out_bf16 ? 32 : 64;
        for (int idx = tid; idx < kRows * per_row; idx += kThreads) {
            const int r = idx / per_row, c4 = idx % per_row;
            const int g = mt * kRows + r;
            if (g >= rows_seq) continue;
            if (a.out_bf16)
                reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(o_dst) + (row_base + g) * 512 + rank * 256)[c4] =
                    make_uint4(0u, 0u, 0u, 0u);
            else
                reinterpret_cast<float4 *>(o_dst + (row_base + g) * 512 + rank * 256)[c4] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (rank == 0 && c4 == 0) lse_dst[row_base + g] = -INFINITY;
        }
        if (warp == kProducerWarp && lane == 0) {
            const int zero = 0;
            mbar_wait(bar(BAR_Q_FULL), 0, globaltimer_ns() + 100000000ull, &zero);
        }
    } else if (warp == kProducerWarp && a.kv_index) {
        // ======================= KV gather, keys 0-31 of each tile =======================
        gather_keys(0);
    } else if (warp == kProducerWarp) {
        // ======================= TMA producer =======================
        if (lane == 0) {
            int armed[kSlots] = {0, 0, 0, 0};
            bool ok = true;
            for (int jj = 0; jj < nrange; ++jj) {
                const int slot = jj % kSlots, use = jj / kSlots, rs = jj % kRopeSlots;
                // latent slot: PV of tile jj - 4 done; rotary slot: S of tile jj - 2 done
                if ((use >= 1 && !mbar_wait(bar(BAR_RING_EMPTY + slot), (use - 1) & 1, deadline, abort_flag)) ||
                    (jj >= kRopeSlots &&
                     !mbar_wait(bar(BAR_S_FULL + (jj - kRopeSlots) % kSPBufs), ((jj - kRopeSlots) / kSPBufs) & 1,
                                deadline, abort_flag))) {
                    ok = false;
                    break;
                }
                const int key_row = b * a.Tcap + (t0 + jj) * kKeys;
                const uint32_t dst = sRing + slot * kLatBytes;
                mbar_arrive_expect_tx(bar(BAR_RING_FULL + slot), kTileBytes);
                ++armed[slot];
                for (int c = 0; c < kQChunks; ++c)
                    tma_load_2d(dst + c * kChunkBytesKV, &tm_kv, static_cast<int>(rank) * 256 + c * 64, key_row,
                                bar(BAR_RING_FULL + slot));
                tma_load_2d(sRope + rs * kKRopeBytes, &tm_kr, static_cast<int>(rank) * 32, key_row,
                            bar(BAR_RING_FULL + slot));
            }
            if (!ok) {
                fail();
                // let every copy this thread started land before the CTA leaves
                const uint64_t drain_deadline = globaltimer_ns() + 100000000ull;
                const int zero = 0;
                mbar_wait(bar(BAR_Q_FULL), 0, drain_deadline, &zero);
                for (int s = 0; s < kSlots; ++s)
                    if (armed[s]) mbar_wait(bar(BAR_RING_FULL + s), (armed[s] - 1) & 1, drain_deadline, &zero);
            }
        }
    } else if (warp == kTreeWarp) {
        // ======================= tree fetch =======================
        // the node count and the ancestor masks of this tile's nodes, once
        // the tree build has finished
        grid_dep_wait();
        const int node_hi = min((mt * kRows + kRows - 1) / a.H, a.Qc - 1);
        const uint64_t *src = a.mask + (static_cast<size_t>(b) * a.Qc + node_lo) * a.W;
        uint64_t *dst = reinterpret_cast<uint64_t *>(smem + kOffTree + 16);
        const int words = (node_hi - node_lo + 1) * a.W;
        for (int w = lane; w < words; w += 32) dst[(w / a.W) * 2 + (w % a.W)] = src[w];
        if (lane == 0) *reinterpret_cast<volatile int *>(smem + kOffTree) = a.n_nodes[b];
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_TREE));
        if (a.kv_index) gather_keys(32);  // ======== KV gather, keys 32-63 of each tile
    } else if (warp == kMmaWarp) {
        // ======================= S issuer =======================
        // S_j = Q K_j^T (this CTA's half of the contraction) into S/P buffer
        // j % kSPBufs, once the buffer's previous PV (tile j - kSPBufs) is done
        // and KV tile j is in the ring. The whole warp runs the loop, so its
        // operands stay warp-uniform; one elected lane issues the MMAs and
        // commits.
        const bool leader = elect_one();
        constexpr uint32_t idS = idesc_f32acc(kRows, kKeys, 1, 0, 0);   // bf16 Q, K (K-major)
        // operand descriptors of the query's latent chunk 0 and rotary part,
        // of latent slot 0's chunk 0 and of rotary slot 0; the loop adds
        // offsets / 16
        const uint64_t dq = desc_sw128(sQ, 16, 1024), dqr = desc_sw64(sQR, 512), dk = desc_sw128(sRing, 16, 1024),
                       dr = desc_sw64(sRope, 512);
        const uint32_t dq_lo = static_cast<uint32_t>(dq), dq_hi = static_cast<uint32_t>(dq >> 32);
        const uint32_t dqr_lo = static_cast<uint32_t>(dqr), dqr_hi = static_cast<uint32_t>(dqr >> 32);
        const uint32_t dk_lo = static_cast<uint32_t>(dk), dk_hi = static_cast<uint32_t>(dk >> 32);
        const uint32_t dr_lo = static_cast<uint32_t>(dr), dr_hi = static_cast<uint32_t>(dr >> 32);
        bool ok = __all_sync(0xffffffffu, mbar_wait(bar(BAR_Q_FULL), 0, deadline, abort_flag));
        tc_fence_after();
        for (int jj = 0; jj < nrange && ok; ++jj) {
            const int sb = jj % kSPBufs, slot = jj % kSlots;
            if (!__all_sync(0xffffffffu, (jj < kSPBufs || mbar_wait(bar(BAR_PV_DONE + sb), ((jj - kSPBufs) / kSPBufs) & 1,
                                                                   deadline, abort_flag)) &&
                                             mbar_wait(bar(BAR_RING_FULL + slot), (jj / kSlots) & 1, deadline,
                                                       abort_flag))) {
                ok = false;
                break;
            }
            // gathered tiles were written by ordinary (generic-proxy)
            // copies: order them before the tensor core's reads
            if constexpr (kPaged) fence_proxy_async_smem();
            tc_fence_after();
            const uint32_t dS = tmem + kColSP + sb * 64;
            const uint32_t k_lo = dk_lo + ((slot * kLatBytes) >> 4),
                           r_lo = dr_lo + (((jj % kRopeSlots) * kKRopeBytes) >> 4);
            if (leader) {
#pragma unroll
                for (int c = 0; c < kQSmemChunks; ++c)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_ss_w(dS, dq_lo + ((c * kChunkBytesQ + ks * 32) >> 4), dq_hi,
                                 k_lo + ((c * kChunkBytesKV + ks * 32) >> 4), dk_hi, idS, (c > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
                    mma_ss_w(dS, dqr_lo + ((ks * 32) >> 4), dqr_hi, r_lo + ((ks * 32) >> 4), dr_hi, idS, 1u);
                mma_commit(bar(BAR_S_FULL + sb));
            }
            __syncwarp();
        }
        if (!ok && leader) {
            fail();
            // wait for this thread's MMAs before tensor memory is released
            mma_commit(bar(BAR_DRAIN));
            const int zero = 0;
            mbar_wait(bar(BAR_DRAIN), 0, globaltimer_ns() + 100000000ull, &zero);
        }
    } else if (warp == kPvWarp) {
        // ======================= PV issuer =======================
        // O += P_j V_j (both bf16 terms of P) once P_j is in tensor memory;
        // then S/P buffer j % kSPBufs and ring slot j % kSlots are free. The
        // whole warp runs the loop; one elected lane issues and commits.
        const bool leader = elect_one();
        constexpr uint32_t idPV = idesc_f32acc(kRows, 256, 1, 0, 1);  // bf16 P (TMEM), V (MN-major)
        // latent slot 0's V descriptor; the loop adds offsets / 16
        const uint64_t dv = desc_sw128(sRing, kChunkBytesKV, 1024);
        const uint32_t dv_lo = static_cast<uint32_t>(dv), dv_hi = static_cast<uint32_t>(dv >> 32);
        bool ok = true;
        for (int j = 0; j < nrange && ok; ++j) {
            const int pb = j % kSPBufs, slot = j % kSlots;
            if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_P_FULL + pb), (j / kSPBufs) & 1, deadline, abort_flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t v_lo = dv_lo + ((slot * kLatBytes) >> 4);
            // keys 32c..32c+31 of P sit in columns 32c..32c+31 of the
            // buffer: 16 hi words, then 16 lo words
            const uint32_t pcol = tmem + kColSP + pb * 64;
            if (leader) {
#pragma unroll
                for (int ks = 0; ks < kKeys / 16; ++ks)
                    mma_ts_w(tmem + kColO, pcol + (ks >> 1) * 32 + (ks & 1) * 8, v_lo + ((ks * 2048) >> 4), dv_hi, idPV,
                             (j > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
                for (int ks = 0; ks < kKeys / 16; ++ks)
                    mma_ts_w(tmem + kColO, pcol + (ks >> 1) * 32 + 16 + (ks & 1) * 8, v_lo + ((ks * 2048) >> 4), dv_hi,
                             idPV, 1u);
                mma_commit(bar(BAR_PV_DONE + pb));
                mma_commit(bar(BAR_RING_EMPTY + slot));
            }
            __syncwarp();
        }
        if (leader) {
            if (ok) {
                mma_commit(bar(BAR_O_FINAL));
            } else {
                fail();
                mma_commit(bar(BAR_DRAIN_PV));
                const int zero = 0;
                mbar_wait(bar(BAR_DRAIN_PV), 0, globaltimer_ns() + 100000000ull, &zero);
            }
        }
    } else if (warp >= kShipWarp0) {
        // ======================= partial-S shippers =======================
        // Once S of tile j is done, lane l of warp 12 + q reads row 32q + l
        // of it (this CTA's partial scores of the row's 64 keys), block-scales
        // each key half and sends it to the partner as unit 2j + h of its
        // exchange ring, as soon as the partner has read the unit its slot
        // held before (two units back); then it writes the scaled values
        // back in place of its own scores and releases the buffer to the
        // softmax. Dedicated warps make the transfer independent of the
        // softmax: it starts as soon as S is done and runs while the softmax
        // of earlier tiles does.
        const int q = warp - kShipWarp0;
        const int srow = q * 32 + lane;
        const uint32_t quad_base = static_cast<uint32_t>(q * 32) << 16;
        const int t_tree = (T / kKeys) - t0;  // first tile of the range that can hold node keys
        const uint32_t r_sx = mapa_shared(sbase + kOffSX, peer);
        const uint32_t r_sx_full = mapa_shared(bar(BAR_SX_FULL), peer);
        // the partner's barriers exist before the first remote store
        cluster_wait();
        bool ok = true;
        int sb = 0;
        uint32_t sph = 0;
        for (int jj = 0; jj < nrange && ok; ++jj) {
            if (!__all_sync(0xffffffffu, mbar_wait(bar(BAR_S_FULL + sb), sph, deadline, abort_flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t v[2][32];
            tmem_ld32(tmem + quad_base + kColSP + sb * 64, v[0]);
            tmem_ld32(tmem + quad_base + kColSP + sb * 64 + 32, v[1]);
            tmem_wait_ld();
            // KV rows past the sequence's key end may hold anything: their
            // scores are set to 0 so they cannot widen a unit's scale (the
            // softmax hides those keys). Only tiles that reach past the prefix
            // can hold such keys; the key end is known once the tree is.
            if (jj >= t_tree) {
                if (!resolved) {
                    const bool ready = __all_sync(0xffffffffu, mbar_wait(bar(BAR_TREE), 0, deadline, abort_flag));
                    resolve(ready, ready ? *tree_n : 0);
                    if (!ready) {
                        ok = false;
                        break;
                    }
                }
                const int kbase = (t0 + jj) * kKeys;
#pragma unroll
                for (int k = 0; k < kKeys; ++k)
                    if (kbase + k >= kend) v[k >> 5][k & 31] = 0u;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t code[16];
                const float dsc = quantize_unit(v[h], code);
                const int un = 2 * jj + h, u = un % kSXUnits, use = un / kSXUnits;
                if (use >= 1 && !__all_sync(0xffffffffu, mbar_wait_cluster(bar(BAR_SX_EMPTY + u), (use - 1) & 1,
                                                                           deadline, abort_flag))) {
                    ok = false;
                    break;
                }
                // unit layout: [4 stores][128 rows] of 16 bytes (code words 4st..4st+3), then the scales
                const uint32_t dst = r_sx + u * kSXUnitBytes, ubar = r_sx_full + 8u * static_cast<uint32_t>(u);
#pragma unroll
                for (int st = 0; st < 4; ++st)
                    st_async_v4(dst + (st * kRows + srow) * 16,
                                make_uint4(code[4 * st], code[4 * st + 1], code[4 * st + 2], code[4 * st + 3]), ubar);
                st_async_b32(dst + kSXMantBytes + srow * 4, __float_as_uint(dsc), ubar);
                // the values both CTAs use for this key half of this CTA's partial, in place of it
#pragma unroll
                for (int p = 0; p < 16; ++p) {
                    float v0, v1;
                    dequantize_pair(code[p], dsc, v0, v1);
                    v[h][2 * p] = __float_as_uint(v0);
                    v[h][2 * p + 1] = __float_as_uint(v1);
                }
                tmem_st32(tmem + quad_base + kColSP + sb * 64 + 32 * h, v[h]);
            }
            if (!ok) break;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(BAR_S_READ + sb));
            sb = sb == kSPBufs - 1 ? 0 : sb + 1;
            sph = sb == 0 ? sph ^ 1u : sph;
        }
        if (!ok) fail();
        // this warp's remote stores are over (each lands on the partner's
        // barrier, which the partner waits for before it leaves)
        cluster_arrive_release();
    } else {
        // ======================= softmax group (warps 0-7) =======================
        // Warp w serves 16 rows: tensor-memory lanes 32(w%4) + 16(w/4) ..
        // +15 of its lane quadrant. Lanes t and t+16 share a row and take its
        // key halves c = t/16 of every tile, keys [32c, 32c+32), through the
        // 16x32bx2 access shape. Per tile a thread adds the partner's partial
        // scores of its row and key half (one unit of the exchange ring) to
        // its own, both block-scaled, and runs the softmax of its row and key
        // half. Both CTAs then hold the same full S and compute the
        // same P (fp32 addition commutes), each for its own half of O. The two
        // threads of a row agree on the row max with a shuffle.
        const int quad = warp & 3, sub = warp >> 2, half = lane >> 4;
        const int row = quad * 32 + sub * 16 + (lane & 15);   // TMEM lane of this thread
        const int g = mt * kRows + row;              // row within the sequence
        const bool row_in_seq = g < rows_seq;
        const int node = g / a.H;
        // Until the tree is known every in-sequence row is treated as a node:
        // the tiles processed before that are pure prefix, visible to all
        // nodes, and rows of absent nodes come out zero in the end.
        bool node_ok = row_in_seq;
        const int t_tree = (T / kKeys) - t0;  // first tile of the range that can hold node keys
        const bool lead = row == 0;  // arms the byte count of its key half's units (warp 0, lanes 0 and 16)
        uint64_t m0 = 0, m1 = 0;
        auto resolve_s = [&]() -> bool {
            const bool ready = __all_sync(0xffffffffu, mbar_wait(bar(BAR_TREE), 0, deadline, abort_flag));
            resolve(ready, ready ? *tree_n : 0);
            node_ok = row_in_seq && node < n && seq_ok;
            if (node_ok) {
                m0 = tree_mask[(node - node_lo) * 2];
                if (a.W > 1) m1 = tree_mask[(node - node_lo) * 2 + 1];
            }
            return ready;
        };
        // this warp's 16 lanes; the S/P buffer columns of key half 1 start 32
        // columns on, those of O's second half 128 columns on
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32 + sub * 16) << 16;
        const uint4 *sx = reinterpret_cast<const uint4 *>(smem + kOffSX);  // units: [4][128 rows] x 16 B, then scales
        const uint32_t r_bar_sx_empty = mapa_shared(bar(BAR_SX_EMPTY), peer);

        // waits of the softmax group are made warp-uniform, so a lane that
        // gives up can never leave its warp split before a .sync.aligned op
        auto wwait = [&](uint32_t barrier, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait(barrier, parity, deadline, abort_flag));
        };
        auto wwait_cluster = [&](uint32_t barrier, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait_cluster(barrier, parity, deadline, abort_flag));
        };
        // the row sum of this thread's keys, as the sums of its even and odd
        // keys (one packed add per key pair)
        float m_ref = -INFINITY, l_even = 0.f, l_odd = 0.f;
        bool ok = true;
        // the partner's barriers exist before this CTA's first remote operation
        cluster_wait();
        // tile jj's S/P buffer (jj % kSPBufs) and phase parity ((jj / kSPBufs) & 1),
        // kept as running counters
        int sb = 0;
        uint32_t sph = 0;
        for (int jj = 0; jj < nrange && ok; ++jj) {
            const int nb = sb == kSPBufs - 1 ? 0 : sb + 1;
            const uint32_t nph = sb == kSPBufs - 1 ? sph ^ 1u : sph;
            const int key0 = (t0 + jj) * kKeys + half * 32;
            // this key half's unit of the partner's partial: unit 2jj + half
            const int un = 2 * jj + half, u = un % kSXUnits;
            if (lead) mbar_arrive_expect_tx(bar(BAR_SX_FULL + u), kSXUnitBytes);
            // this CTA's partial of tile jj as the shippers left it, block-scaled
            // (loaded while the partner's is awaited)
            if (!wwait(bar(BAR_S_READ + sb), sph)) {
                ok = false;
                break;
            }
            __syncwarp();
            tc_fence_after();
            uint32_t sv[32];
            tmem_ld16x2_32<32>(tmem + lane_base + kColSP + sb * 64, sv);
            const bool got = wwait_cluster(bar(BAR_SX_FULL + u), (un / kSXUnits) & 1);
            tmem_wait_ld();
            if (!got) {
                ok = false;
                break;
            }
            // the unit's 16 code words and scale of this row; read_dep depends
            // on every load (a 128-bit load completes as a whole, so one word
            // of each is enough)
            uint32_t w[16];
            const uint4 *ux = sx + u * (kSXUnitBytes / 16) + row;
            const uint32_t dbits = reinterpret_cast<const uint32_t *>(smem + kOffSX + u * kSXUnitBytes + kSXMantBytes)[row];
            uint32_t read_dep = dbits;
#pragma unroll
            for (int st = 0; st < 4; ++st) {
                const uint4 o = ux[st * kRows];
                read_dep ^= o.x;
                w[4 * st] = o.x;
                w[4 * st + 1] = o.y;
                w[4 * st + 2] = o.z;
                w[4 * st + 3] = o.w;
            }
            // hand the slot back once every read of it is done (the arrive
            // waits for read_dep)
            mbar_arrive_remote_relaxed_after(r_bar_sx_empty + 8u * static_cast<uint32_t>(u), read_dep,
                                             sBar + NUM_BARS * 8 + 8);
            float s[32];
#pragma unroll
            for (int p = 0; p < 16; ++p) {
                float v0, v1;
                dequantize_pair(w[p], __uint_as_float(dbits), v0, v1);
                add_f32x2(__uint_as_float(sv[2 * p]), __uint_as_float(sv[2 * p + 1]), v0, v1, s[2 * p], s[2 * p + 1]);
            }
            // ---- masked online softmax, log2 domain
            if (!resolved && jj >= t_tree && !resolve_s()) {
                ok = false;
                break;
            }
            uint32_t vis = ~0u;
            if (!node_ok) vis = 0;
            else if (key0 + 32 > T) vis = half_tile_visibility(key0, T, n, m0, m1);
            // The scores stay unscaled: the scale (positive, checked on the
            // host) is applied to their maximum here and folded into the
            // exponent's FFMA below. Hidden keys become -inf, only in tiles
            // where some lane has one.
            if (!__all_sync(0xffffffffu, vis == ~0u)) {
#pragma unroll
                for (int k = 0; k < 32; ++k) s[k] = ((vis >> k) & 1u) ? s[k] : -INFINITY;
            }
            // two three-input max chains over the 32 scores
            float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
            for (int k = 0; k < 32; k += 4) {
                mxa = fmax3(mxa, s[k], s[k + 1]);
                mxb = fmax3(mxb, s[k + 2], s[k + 3]);
            }
            float mx = fmaxf(mxa, mxb);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16)) * a.scale_log2;  // the row's other key half
            float alpha = 1.0f;  // rescale factor of this row's O for this tile
            if (mx > m_ref + kRescaleThreshold) {
                alpha = ex2_approx(m_ref - mx);  // 0 while nothing was visible before
                m_ref = mx;
                l_even *= alpha;
                l_odd *= alpha;
            }
            // P = hi + lo, both bf16. While no key has been visible yet
            // m_ref is -inf and every s is -inf: subtracting 0 keeps p = 0.
            const float nmref = (m_ref == -INFINITY) ? 0.f : -m_ref;
            uint32_t pw[32];  // 16 hi words, then 16 lo words
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                float e0, e1, r0, r1;
                fma_f32x2(s[2 * k], s[2 * k + 1], a.scale_log2, nmref, e0, e1);
                const float p0 = ex2_approx(e0);
                const float p1 = ex2_approx(e1);
                const uint32_t h = pack_bf16x2(p0, p1);
                pw[k] = h;
                sub_f32x2(p0, p1, bf16lo_to_f32(h), bf16hi_to_f32(h), r0, r1);
                pw[16 + k] = pack_bf16x2(r0, r1);
                add_f32x2(l_even, l_odd, p0, p1, l_even, l_odd);
            }
            // ---- rescale this thread's half of the row's O (needs PV of the
            // previous tile done), then publish P over the S it replaces
            if (__any_sync(0xffffffffu, alpha != 1.0f) && jj >= 1) {
                if (!wwait(bar(BAR_PV_DONE + ((jj - 1) % kSPBufs)), ((jj - 1) / kSPBufs) & 1)) {
                    ok = false;
                    break;
                }
                __syncwarp();
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    const uint32_t col = kColO + c * 32;  // (+128 for key half 1)
                    uint32_t o[32];
                    tmem_ld16x2_32<128>(tmem + lane_base + col, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int v = 0; v < 32; ++v) o[v] = __float_as_uint(__uint_as_float(o[v]) * alpha);
                    tmem_st16x2_32<128>(tmem + lane_base + col, o);
                }
            }
            // KV rows past the last node may hold anything (NaN included) and
            // P is 0 there, but 0 * NaN is NaN: zero those V rows of the tail
            // tile (S, which read them as K, is already complete)
            if (jj >= t_tree && (t0 + jj) * kKeys + kKeys > kend) {  // (jj >= t_tree: the tree is known)
                uint4 *vset = reinterpret_cast<uint4 *>(smem + kOffRing + (jj % kSlots) * kLatBytes);
                const int kvalid = kend - (t0 + jj) * kKeys;
#pragma unroll 1
                for (int e = half * kRows + row; e < kQChunks * kChunkBytesKV / 16; e += 2 * kRows)
                    if (((e >> 3) & (kKeys - 1)) >= kvalid) vset[e] = make_uint4(0, 0, 0, 0);
                fence_proxy_async_smem();
            }
            tmem_st16x2_32<32>(tmem + lane_base + kColSP + sb * 64, pw);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(BAR_P_FULL + sb));
            sb = nb;
            sph = nph;
        }
        if (ok && !resolved && !resolve_s()) ok = false;
        // the row sum is the two halves' sums (same reference max)
        float l_sum = l_even + l_odd;
        l_sum += __shfl_xor_sync(0xffffffffu, l_sum, 16);
        if (ok && !wwait(bar(BAR_O_FINAL), 0)) ok = false;
        if (!ok) fail();
        __syncwarp();
        tc_fence_after();
        // This thread's remote operations are over (the last exchange unit
        // handed back; a release arrival orders them first): arrive on the
        // cluster barrier that lets the partner leave.
        // It is waited on only at the very end, so the staging and stores
        // below hold neither CTA. (Arriving right after the tile loop instead
        // measured 0.9% slower on the max-budget workload.)
        cluster_arrive_release();
        // rows of absent nodes, and every row of a range with no tile of
        // this sequence's keys, are zero (tensor memory was not written)
        const bool zero_row = !node_ok;
        const float inv_l = (l_sum > 0.f && !zero_row) ? 1.0f / l_sum : 0.f;
        // Stage this thread's 128 output columns in the KV ring (idle once
        // every PV is done), 32 at a time; as soon as the eight softmax warps
        // have staged a chunk, one thread stores the boxes it completes, so
        // the stores overlap the rest of the staging. The tensor map has the
        // sequence's rows as one dimension: rows past the sequence are not
        // written. Every softmax warp takes part in each barrier, failed or
        // not (a failure is in the abort flag before the first one).
        const int box_cols = a.out_bf16 ? 64 : 32;
        for (int c = 0; c < 4; ++c) {
            if (ok) stage_chunk(tmem + lane_base + kColO, smem + kOffRing, half, row, zero_row, inv_l,
                                a.out_bf16 != 0, c);
            fence_proxy_async_smem();
            named_bar_sync(1, 8 * 32);
            if (tid == 0 && !*abort_flag && (!a.out_bf16 || (c & 1))) {
                // float32: boxes c and 4 + c; bfloat16: boxes c/2 and 2 + c/2
                const int box0 = a.out_bf16 ? (c >> 1) : c, box1 = box0 + (a.out_bf16 ? 2 : 4);
                tma_store_3d(&tm_o, sRing + box0 * kOutBoxBytes, static_cast<int>(rank) * 256 + box0 * box_cols,
                             mt * kRows, b + a.B * chunk);
                tma_store_3d(&tm_o, sRing + box1 * kOutBoxBytes, static_cast<int>(rank) * 256 + box1 * box_cols,
                             mt * kRows, b + a.B * chunk);
                bulk_commit_group();
                stored = true;
            }
        }
        // both CTAs hold the same row sum and max; one writes the lse
        if (ok && rank == 0 && half == 0 && row_in_seq)
            lse_dst[row_base + g] =
                (l_sum > 0.f && !zero_row) ? (m_ref + __log2f(l_sum)) * 0.69314718055994531f : -INFINITY;
    }

    // The producer, MMA and tree warps wait on the setup's cluster barrier
    // now and arrive on the final one (they made no remote access).
    if ((warp >= kProducerWarp && warp < kShipWarp0) || nrange <= 0) {
        cluster_wait();
        cluster_arrive_relaxed();
    }
    // Every thread has waited for the tree build by now (or does so here);
    // only then may the next kernel of the step start.
    grid_dep_wait();
    grid_dep_launch();
    if (tid == 0) {
        if (!resolved) {
            if (nrange > 0) {
                const bool r = mbar_wait(bar(BAR_TREE), 0, deadline, abort_flag);
                resolve(r, r ? *tree_n : 0);
            } else {
                grid_dep_wait();
                resolve(true, a.n_nodes[b]);
            }
        }
        if (!seq_ok && mt == 0 && rank == 0 && chunk == 0 && !*abort_flag) a.status[b] = DDT_E_BADINPUT;
    }
    // every tensor-memory access of the CTA is complete before it is freed
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    // the tensor stores have read the staged block before shared memory is
    // released, and neither CTA leaves while its partner can still access it
    if (stored) bulk_wait_read_all();
    cluster_wait();
}

// Merge per-chunk normalised partials: lse = log sum_c exp(lse_c),
// out = sum_c exp(lse_c - lse) out_c. One 128-thread block per row; each
// thread owns one float4 of the row. The float4 of the first kAhead chunks
// are loaded before the weights are known, together with the row's lse
// values, so one memory round trip serves both; a chunk of weight 0 (no
// visible key) contributes nothing, whatever its partial holds. Chunks past
// kAhead are read in batches of 8 once the weights are known. kAhead (4, 8
// or 16) follows the chunk count: registers held for loads that are never
// issued would only lower the occupancy.
// Inside a verify step the grid has ceil(B / 4) blocks more, whose warps run
// the accept walk of one sequence each (it needs only the tree, complete
// before the attention kernel let this grid start), so the step needs no
// launch of its own for the accept.
// The partials are read through plain pointers, not const __restrict__ ones:
// this grid starts while the attention grid still writes them, so they are
// not read-only for its lifetime, and a restrict-qualified load may be
// hoisted above the dependency wait or served by the non-coherent cache.
template <int kAhead>
__global__ void __launch_bounds__(128)
    merge_chunks_kernel(size_t rows_total, int nsplit, const float *ws_o, const float *ws_lse,
                        void *__restrict__ out, int out_bf16, float *__restrict__ lse, const AcceptArgs walk) {
    __shared__ float wsh[64];
    __shared__ float stat[2];
    // work later on the stream may start now; the partials are complete once
    // the attention grid is
    grid_dep_launch();
    const size_t r = blockIdx.x;
    const int t = threadIdx.x;
    if (r >= rows_total) {
        const int b = static_cast<int>(r - rows_total) * 4 + (t >> 5);
        if (b < walk.B) accept_walk(walk, b, t & 31);
        return;
    }
    grid_dep_wait();
    const float4 *src = reinterpret_cast<const float4 *>(ws_o) + r * 128 + t;
    float4 ahead[kAhead];
#pragma unroll
    for (int u = 0; u < kAhead; ++u)
        ahead[u] = u < nsplit ? src[u * rows_total * 128] : make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < 32) {
        // lse of chunks t and t + 32 (nsplit <= 64), their maximum, weights, sum
        const float l0 = t < nsplit ? ws_lse[t * rows_total + r] : -INFINITY;
        const float l1 = t + 32 < nsplit ? ws_lse[(t + 32) * rows_total + r] : -INFINITY;
        float mx = fmaxf(l0, l1);
#pragma unroll
        for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float w0 = (mx == -INFINITY || l0 == -INFINITY) ? 0.f : __expf(l0 - mx);
        const float w1 = (mx == -INFINITY || l1 == -INFINITY) ? 0.f : __expf(l1 - mx);
        float sum = w0 + w1;
#pragma unroll
        for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        wsh[t] = w0;
        wsh[t + 32] = w1;
        if (t == 0) {
            stat[0] = mx;
            stat[1] = sum;
        }
    }
    __syncthreads();
    const float mx = stat[0], sum = stat[1];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [&](float w, const float4 &v) {
        if (w != 0.f) {
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        }
    };
    if (mx != -INFINITY) {
#pragma unroll
        for (int u = 0; u < kAhead; ++u)
            if (u < nsplit) add(wsh[u], ahead[u]);
        for (int c0 = kAhead; c0 < nsplit; c0 += 8) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                v[u] = (c0 + u < nsplit && wsh[c0 + u] != 0.f) ? src[(c0 + u) * rows_total * 128]
                                                             : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (c0 + u < nsplit) add(wsh[c0 + u], v[u]);
        }
        const float inv = 1.0f / sum;
        acc.x *= inv;
        acc.y *= inv;
        acc.z *= inv;
        acc.w *= inv;
    }
    if (out_bf16)
        reinterpret_cast<uint2 *>(static_cast<uint16_t *>(out) + r * 512)[t] =
            make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    else
        reinterpret_cast<float4 *>(static_cast<float *>(out) + r * 512)[t] = acc;
    if (t == 0) lse[r] = (mx == -INFINITY) ? -INFINITY : mx + __logf(sum);
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

// The kernels' dynamic shared-memory size, set once per device (and tried
// again on the next call if setting it failed).
cudaError_t set_attn_attributes() {
    constexpr int kDevices = 64;
    static std::mutex mu;
    static bool done[kDevices];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(verify_attn_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(verify_attn_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess) done[dev] = true;
    return e;
}

// bf16 matrix [rows, cols] row-major, box [box_rows, box_cols]
bool encode_2d(EncodeTiledFn enc, CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows,
               uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz) {
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 tensor [dim2][dim1][cols] row-major, box [box_rows, 32 columns] (128 bytes,
// 128-byte swizzle), for tile stores
// (or bfloat16 with 64-column boxes: 128 bytes either way)
bool encode_3d_store(EncodeTiledFn enc, CUtensorMap *m, void *ptr, uint64_t cols, uint64_t dim1, uint64_t dim2,
                     uint32_t box_rows, bool bf16) {
    const uint64_t es = bf16 ? 2 : 4;
    cuuint64_t dims[3] = {cols, dim1, dim2};
    cuuint64_t strides[2] = {cols * es, dim1 * cols * es};
    cuuint32_t box[3] = {bf16 ? 64u : 32u, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

AttnPlan plan_attention(int B, int Qc, int H, int Tcap, int sms) {
    AttnPlan p{};
    p.mtiles = (Qc * H + kRows - 1) / kRows;
    // each row tile is a cluster of two CTAs, one per SM
    const long long base = static_cast<long long>(B) * p.mtiles * 2;
    const int tiles = (Tcap + kKeys - 1) / kKeys;
    const size_t rows_total = static_cast<size_t>(B) * Qc * H;
    // Pick the split of each sequence's keys that minimises a simple cost:
    // waves of CTAs x key tiles per CTA (about 1 us each, plus 2 for the
    // prologue and epilogue), plus the partial outputs the merge writes and
    // reads (about 1 us per 4 MB at HBM rate). At least 4 key tiles per range.
    int best = 1;
    double best_cost = 1e30;
    const int max_split = tiles / 4 > 1 ? tiles / 4 : 1;
    for (int s = 1; s <= max_split && s <= 64; ++s) {
        const long long ctas = base * s;
        const long long waves = (ctas + sms - 1) / sms;
        const double per_cta = static_cast<double>((tiles + s - 1) / s) + 2.0;
        const double merge = s > 1 ? static_cast<double>(s + 1) * rows_total * 2048.0 / 4.0e6 : 0.0;
        const double cost = waves * per_cta + merge;
        if (cost < best_cost * 0.98) {
            best_cost = cost;
            best = s;
        }
    }
    p.nsplit = best;
    p.ws_bytes = best > 1 ? static_cast<size_t>(best) * rows_total * (512 + 1) * sizeof(float) : 0;
    return p;
}

int launch_verify_attn(const ddt_attn_in &in, const ddt_tree &tree, float scale,
                       const ddt_attn_out &out, void *workspace, size_t ws_bytes,
                       const AttnPlan &plan, cudaStream_t s, bool after_prev, const int32_t *kv_index,
                       int pool_rows, bool out_bf16, const AcceptArgs *fused_accept, bool *accepted) {
    if (accepted) *accepted = false;
    EncodeTiledFn enc = get_encoder();
    if (!enc) return DDT_E_CUDA;
    const uint64_t rows_total = static_cast<uint64_t>(tree.B) * tree.Qc * in.H;
    // (with a block table the KV maps cover the pools; the gather path does
    // not use them)
    const uint64_t kv_rows = kv_index ? static_cast<uint64_t>(pool_rows) : static_cast<uint64_t>(tree.B) * in.Tcap;
    CUtensorMap tm_q, tm_qr, tm_kv, tm_kr;
    if (!encode_2d(enc, &tm_q, in.q_lat, 512, rows_total, 64, kRows, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(enc, &tm_qr, in.q_rope, 64, rows_total, 32, kRows, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !encode_2d(enc, &tm_kv, in.c_kv, 512, kv_rows, 64, kKeys, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(enc, &tm_kr, in.k_rope, 64, kv_rows, 32, kKeys, CU_TENSOR_MAP_SWIZZLE_64B))
        return DDT_E_INVAL;

    if (set_attn_attributes() != cudaSuccess) return DDT_E_CUDA;

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
    a.status = tree.status;
    a.rows_total = rows_total;
    a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    a.wait_ns = kWaitLimitNs;
    a.kv_index = kv_index;
    a.pool_kv = static_cast<const uint8_t *>(in.c_kv);
    a.pool_kr = static_cast<const uint8_t *>(in.k_rope);
    a.pool_rows = pool_rows;
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
    // the output (or the key-range partials) as [splits x B][Qc*H rows][512]
    a.out_bf16 = (out_bf16 && plan.nsplit == 1) ? 1 : 0;
    CUtensorMap tm_o;
    if (!encode_3d_store(enc, &tm_o, a.o_dst, 512, static_cast<uint64_t>(tree.Qc) * in.H,
                         static_cast<uint64_t>(tree.B) * plan.nsplit, kRows, a.out_bf16 != 0))
        return DDT_E_INVAL;
    dim3 grid(plan.mtiles * 2, plan.nsplit, tree.B);
    if (launch_kernel(kv_index ? verify_attn_kernel<true> : verify_attn_kernel<false>, grid, dim3(kThreads), kSmemBytes,
                      s, after_prev, tm_q, tm_qr, tm_kv, tm_kr, tm_o, a) != cudaSuccess)
        return DDT_E_CUDA;
    if (plan.nsplit > 1) {
        auto merge = plan.nsplit <= 4 ? merge_chunks_kernel<4>
                     : plan.nsplit <= 8 ? merge_chunks_kernel<8> : merge_chunks_kernel<16>;
        AcceptArgs acc{};  // B = 0: no accept blocks
        if (fused_accept) acc = *fused_accept;
        const uint64_t blocks = rows_total + (static_cast<uint64_t>(acc.B) + 3) / 4;
        if (launch_kernel(merge, dim3(static_cast<unsigned>(blocks)), dim3(128), 0, s, after_prev,
                          static_cast<size_t>(rows_total), plan.nsplit, static_cast<const float *>(ws_o),
                          static_cast<const float *>(ws_lse), static_cast<void *>(out.out), out_bf16 ? 1 : 0,
                          out.lse, acc) != cudaSuccess)
            return DDT_E_CUDA;
        if (accepted && fused_accept) *accepted = true;
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
