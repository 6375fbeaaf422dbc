// bkv_ragged_tc.cu -- tensor-core (tcgen05 + TMA) prefill kernel of the
// mixed-step attention: bf16, head_dim 128, query tiles of 128 rows, two
// query tiles per unit of work.
//
// Operation ("Padding and Batching with Block KV", Batching with Block KV
// and Cache Masking; see bkv_ragged.cu): each query token of a request
// attends, at its own position, over the request's paged keys.
//
// Design (sm_103a):
// * Work unit = (request r, KV head g, pair p of query tiles): tile A is the
//   request's query tile 2p and tile B tile 2p + 1 (absent when the request
//   has an odd number of tiles; a decode token has one), each the T = 128 / G
//   query tokens of the tile times the G query heads of g, 128 rows ordered
//   (token, head) -- exactly the box a 3-D TMA load of q (head_dim, H_q,
//   tokens) delivers.  Both tiles read the same key tiles [0, nk), nk
//   covering the causal bound of the unit's last token, so every K and V
//   tile is loaded once for two MMAs.  Persistent CTAs, one per SM.
// * Warp roles: warp 0 loads Q and gathers K tiles, the last warp gathers V
//   tiles (2-slot rings of 32 KB), warp 1 issues tcgen05.mma from one thread
//   and owns the tensor memory; sixteen softmax warps, four warpgroups: for
//   each query tile one per half of every key tile (keys 0..63, 64..127),
//   one query row (TMEM lane) per thread.  The two halves of a row exchange
//   their partial tile max (and at the end their weight sums) through shared
//   memory at a bounded two-warp barrier, so both take the same rescaling
//   decision.
// * Units are ranked by cost (key tiles, one or two query tiles) and dealt
//   to the CTAs back and forth, largest first.
// * Tensor memory (512 columns): S_A, S_B (128 fp32 columns each) and the
//   accumulators O_A, O_B (128 each).  Each key half writes its P (bf16, two
//   per 32-bit column) over the first 32 of its own 64 S columns, and P V
//   takes P from tensor memory (tcgen05.mma with A in TMEM), so P never goes
//   through shared memory.
// * MMA order per key tile j: O_A += P_A(j-1) V(j-1); S_A(j) = Q_A K(j)^T;
//   O_B += P_B(j-1) V(j-1); S_B(j) = Q_B K(j)^T.  While softmax A works on
//   S_A(j) the tensor cores run O_B and S_B, and the other way round, so the
//   two softmax warpgroups overlap each other and the MMAs.  The MMA that
//   overwrites S_X's columns is issued after the one that reads P_X from
//   them (one thread's tcgen05 MMAs run in issue order), and a commit after
//   S_X(j) completes only once O_X(j-1) has, so when softmax X sees S_X(j)
//   its O_X is settled and may be rescaled.
// * Softmax: S read from TMEM in 32-column chunks (max pass, then
//   exponentials); per-row key limit (cache end and causal bound) and a
//   null-segment mask; a tile fully visible to every row of a warp skips the
//   per-key tests.  The running max is a lazy reference that moves only when
//   a tile's max passes it by more than 8 (log2 units), so O in TMEM is
//   rescaled only on those tiles.
// * Keys are gathered through the block table with one TMA load per block
//   segment and head_dim half; null and out-of-range entries are not loaded,
//   positions past the causal bound of the unit's last token are not loaded,
//   and V rows loaded past the cache end are zeroed (by softmax A) before P V.
// * Every wait is bounded (~2 s), after which the CTA records 1 << 24 in
//   err_count, frees its TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "bkv_ragged.cuh"
#include "bkv_tc_ptx.cuh"

namespace bkv {
namespace rtc {

using namespace tc;

constexpr int kTile = 128;                   // keys per tile; query rows per tile
constexpr int kD = 128;                      // head_dim handled
constexpr int kStages = 2;                   // K ring and V ring depth
constexpr int kHalfBytes = kTile * 128;      // 128 rows x 64 bf16: one head_dim (or key) half
constexpr int kTileBytes = 2 * kHalfBytes;   // 32 KB
constexpr int kThreads = 608;                // K producer, MMA, 4 x 4 softmax warps, V producer
constexpr int kWarpV = kThreads / 32 - 1;
constexpr int kTmemCols = 512;               // S_A, S_B, O_A, O_B (128 columns each)
constexpr int kTimeoutErr = 1 << 24;
constexpr int kMaxReqs = 2048;

constexpr int kOffQ = 0;                                 // Q_A, Q_B
constexpr int kOffK = kOffQ + 2 * kTileBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffMask = kOffV + kStages * kTileBytes;   // 8 words: loaded segments per tile (ring)
constexpr int kOffBar = kOffMask + 64;
constexpr int kNumBars = 4 * kStages + 2 + 8 + 8 + 8;
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
constexpr int kOffPre = (kOffAbort + 4 + 15) / 16 * 16;  // [kMaxReqs + 1] units before request r
// the two key halves of a query tile exchange, per row, their partial tile max
// ([tile][half][tile parity][row]) and at the end their partial row sums ([tile][half][row])
constexpr int kOffXmax = (kOffPre + (kMaxReqs + 1) * 4 + 15) / 16 * 16;
constexpr int kOffXsum = kOffXmax + 2 * 2 * 2 * kTile * 4;
// the unit schedule: each unit's cost, a histogram of costs, this CTA's units
constexpr int kSchedUnits = 4096;            // launches with more units are dealt round robin
constexpr int kBuckets = 1024;
constexpr int kMaxMine = 64;
constexpr int kOffCost = kOffXsum + 2 * 2 * kTile * 4;
constexpr int kOffHist = kOffCost + kSchedUnits * 2;
constexpr int kOffMine = kOffHist + kBuckets * 4;
constexpr int kOffUnits = kOffMine + kMaxMine * 4;      // this CTA's units, decoded once
constexpr int kSmemUsed = kOffUnits + kMaxMine * 48;
constexpr int kSmemBytes = kSmemUsed + 1024;             // slack for 1024 alignment
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA exceeds the sm_103a limit");

__host__ __device__ constexpr uint32_t col_s(int x) { return 128u * (uint32_t)x; }         // S_A, S_B
__host__ __device__ constexpr uint32_t col_o(int x) { return 256u + 128u * (uint32_t)x; }  // O_A, O_B

// One unit of work and the facts every role derives from it.
struct Unit {
    int r, g;
    int64_t t0;          // first packed token of the request
    int32_t ql, L;       // query tokens and cache length of the request
    int32_t tok0;        // tile A's first token (of the request); tile B starts T later
    int32_t ntok[2];     // tokens of tile A and B (B: 0 when absent)
    int32_t kend;        // keys [0, kend) may be visible to some row of the unit
    int32_t nk;          // key tiles
};

static_assert(sizeof(Unit) <= 48 && alignof(Unit) <= 16, "the shared-memory unit list holds 48 bytes per unit");

__device__ __forceinline__ int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

constexpr float kSlack = 8.f;   // lazy-rescale slack of the running max (log2 units)

// Max and sum of 32 values as trees (depth 5, not a 32-long chain).
__device__ __forceinline__ float tree_max32(const float (&v)[32]) {
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) t[i] = fmaxf(v[2 * i], v[2 * i + 1]);
#pragma unroll
    for (int w = 8; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) t[i] = fmaxf(t[2 * i], t[2 * i + 1]);
    return t[0];
}

__device__ __forceinline__ float tree_sum32(const float (&v)[32]) {
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) t[i] = v[2 * i] + v[2 * i + 1];
#pragma unroll
    for (int w = 8; w > 0; w >>= 1)
#pragma unroll
        for (int i = 0; i < w; ++i) t[i] = t[2 * i] + t[2 * i + 1];
    return t[0];
}

// Units of request r: H_kv KV heads times its pairs of query tiles.
__device__ __forceinline__ int pairs_of(int32_t ql, int T) { return ceil_div_i(ceil_div_i(ql, T), 2); }

// Unit u of the launch (pre[] in shared memory holds the units before each
// request; T tokens per tile).
__device__ __forceinline__ Unit unit_at(const RaggedArgs &a, const int32_t *pre, int64_t u, int T) {
    int lo = 0, hi = a.num_reqs;   // last request with pre[r] <= u
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid] <= u) lo = mid;
        else hi = mid;
    }
    Unit x;
    x.r = lo;
    const RaggedReq q = ragged_req(a, lo);
    x.t0 = q.t0;
    x.ql = q.ql;
    x.L = q.L;
    const int np = pairs_of(q.ql, T);
    const int64_t v = u - pre[lo];
    x.g = (int)(v / np);
    const int p = (int)(v - (int64_t)x.g * np);
    x.tok0 = 2 * p * T;
    x.ntok[0] = min(T, q.ql - x.tok0);
    x.ntok[1] = max(0, min(T, q.ql - x.tok0 - T));
    const int32_t last = x.ntok[1] > 0 ? x.tok0 + T + x.ntok[1] - 1 : x.tok0 + x.ntok[0] - 1;
    const int32_t plast = q.L - q.ql + last;   // position of the unit's last token
    const int32_t kend = a.mask_mode == 0 ? min(q.L, plast + 1) : q.L;
    x.kend = kend > 0 ? kend : 0;
    x.nk = ceil_div_i(x.kend, kTile);
    return x;
}

template <int kDummy = 0>
__global__ void __launch_bounds__(kThreads, 1)
    ragged_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmQ, const RaggedArgs a, int seg_rows, int T) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint32_t *mask_words = reinterpret_cast<uint32_t *>(smem + kOffMask);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffTmemSlot);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffAbort);
    int32_t *pre = reinterpret_cast<int32_t *>(smem + kOffPre);
    const uint32_t bar0 = sbase + kOffBar;
    auto bar_kfull = [&](int s) { return bar0 + 8u * s; };
    auto bar_kempty = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto bar_vfull = [&](int s) { return bar0 + 8u * (2 * kStages + s); };
    auto bar_vempty = [&](int s) { return bar0 + 8u * (3 * kStages + s); };
    const uint32_t bar_qfull = bar0 + 8u * (4 * kStages);
    const uint32_t bar_qempty = bar0 + 8u * (4 * kStages + 1);
    // per query tile x (0: A, 1: B): S ready, P ready (4 warps), O ready, O read out (4 warps)
    auto bar_sfull = [&](int x) { return bar0 + 8u * (4 * kStages + 2 + x); };
    auto bar_pfull = [&](int x) { return bar0 + 8u * (4 * kStages + 4 + x); };
    auto bar_ofull = [&](int x) { return bar0 + 8u * (4 * kStages + 6 + x); };
    auto bar_oempty = [&](int x) { return bar0 + 8u * (4 * kStages + 8 + x); };
    auto bar_mask = [&](int m) { return bar0 + 8u * (4 * kStages + 10 + m); };
    // the two warps (one per key half) that share TMEM lane quarter qw of query tile x
    auto bar_pair = [&](int x, int qw) { return bar0 + 8u * (4 * kStages + 18 + 4 * x + qw); };
    const uint32_t sm_q = sbase + kOffQ;
    const uint32_t sm_k = sbase + kOffK;
    const uint32_t sm_v = sbase + kOffV;

    // ---- set-up (no global memory) ----
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar_kfull(s), 1);
            mbar_init(bar_kempty(s), 1);
            mbar_init(bar_vfull(s), 1);
            mbar_init(bar_vempty(s), 1);
        }
        mbar_init(bar_qfull, 1);
        mbar_init(bar_qempty, 1);
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar_sfull(x), 1);
            mbar_init(bar_pfull(x), 8);
            mbar_init(bar_ofull(x), 1);
            mbar_init(bar_oempty(x), 8);
            for (int qw = 0; qw < 4; ++qw) mbar_init(bar_pair(x, qw), 2);
        }
        for (int m = 0; m < 8; ++m) mbar_init(bar_mask(m), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmQ);
    }
    {
        // the V ring starts at zero: a row no TMA load writes must never hold
        // uninitialised bits (NaN) that P V could read
        const uint4 z = make_uint4(0, 0, 0, 0);
        uint4 *v = reinterpret_cast<uint4 *>(smem + kOffV);
        for (int i = threadIdx.x; i < kStages * kTileBytes / 16; i += kThreads) v[i] = z;
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();   // global memory is read from here on
    pdl_trigger();
    // units per request (H_kv * pairs of query tiles), then their exclusive prefix sum
    for (int r = threadIdx.x; r < a.num_reqs; r += kThreads) {
        const RaggedReq q = ragged_req(a, r);
        pre[r] = q.ql > 0 ? a.H_kv * pairs_of(q.ql, T) : 0;
        if (q.bad && blockIdx.x == 0 && a.err) atomicAdd(a.err, 1);
    }
    __syncthreads();
    if (warp == 0) {
        const int n = a.num_reqs;
        const int per = (n + 31) / 32;
        const int lo = min(n, lane * per), hi = min(n, lo + per);
        int32_t sum = 0;
        for (int r = lo; r < hi; ++r) sum += pre[r];
        int32_t inc = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t x = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += x;
        }
        int32_t run = inc - sum;
        for (int r = lo; r < hi; ++r) {
            const int32_t t = pre[r];
            pre[r] = run;
            run += t;
        }
        if (lane == 31) pre[n] = inc;
    }
    __syncthreads();
    const uint32_t tmem = *tmem_slot;
    const int64_t U = pre[a.num_reqs];
    const int G = a.G;
    const int nseg = kTile / seg_rows;
    const int seg_shift = 31 - __clz(seg_rows);
    const uint32_t all_seg = nseg >= 32 ? 0xffffffffu : ((1u << nseg) - 1u);   // every segment loaded

    // ---- the unit schedule ----
    // Units differ in cost (key tiles, one or two query tiles).  Every CTA ranks all units by
    // cost, largest first (a counting sort over cost buckets, ties in unit order, so every CTA
    // computes the same ranking), and takes the ranks it gets when they are dealt over the
    // CTAs back and forth (0 .. grid-1, grid-1 .. 0, ...): the largest units are spread first
    // and the per-CTA sums come out close.  Beyond kSchedUnits units, round robin.
    const int64_t grid = gridDim.x;
    const bool lpt = U > grid && U <= kSchedUnits && (U + grid - 1) / grid <= kMaxMine;
    int32_t *mine = reinterpret_cast<int32_t *>(smem + kOffMine);
    if (lpt) {
        uint16_t *cost = reinterpret_cast<uint16_t *>(smem + kOffCost);
        int32_t *hist = reinterpret_cast<int32_t *>(smem + kOffHist);
        for (int b = threadIdx.x; b < kBuckets; b += kThreads) hist[b] = 0;
        __syncthreads();
        for (int u = threadIdx.x; u < U; u += kThreads) {
            const Unit x = unit_at(a, pre, u, T);
            // a unit's time follows its key tiles: with two query tiles the second softmax runs
            // beside the first, and measured pairs take about as long per key tile as singles
            const int c = min(x.nk, kBuckets - 1);
            cost[u] = (uint16_t)c;
            atomicAdd(&hist[kBuckets - 1 - c], 1);   // bucket order = descending cost
        }
        __syncthreads();
        if (warp == 0) {
            // exclusive prefix sum of the buckets: lane l owns buckets [32 l, 32 l + 32)
            int32_t sum = 0;
            for (int b = 32 * lane; b < 32 * lane + 32; ++b) sum += hist[b];
            int32_t inc = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += y;
            }
            int32_t run = inc - sum;
            for (int b = 32 * lane; b < 32 * lane + 32; ++b) {
                const int32_t t = hist[b];
                hist[b] = run;
                run += t;
            }
            __syncwarp();
            // ranks in unit order, 32 units at a time; rank -> CTA by the back-and-forth deal
            for (int base = 0; base < U; base += 32) {
                const int u = base + lane;
                const int b = u < U ? kBuckets - 1 - cost[u] : -1 - lane;
                const unsigned same = __match_any_sync(0xffffffffu, b);
                const int before = __popc(same & ((1u << lane) - 1u));
                const int start = u < U ? hist[b] : 0;
                __syncwarp();
                if (u < U && before == 0) hist[b] = start + __popc(same);
                __syncwarp();
                if (u < U) {
                    const int rank = start + before;
                    const int k = rank / (int)grid, c = rank - k * (int)grid;
                    if (((k & 1) ? (int)grid - 1 - c : c) == (int)blockIdx.x) mine[k] = u;
                }
            }
        }
        __syncthreads();
    }
    // this CTA's units, in the order it runs them: one per full round of the deal, and one in the
    // last, partial round if the deal reaches it there
    int n_mine;
    if (lpt) {
        const int full = (int)(U / grid), rem = (int)(U - full * grid);
        const int c = (int)blockIdx.x;
        n_mine = full + ((full & 1) ? ((int)grid - 1 - c < rem) : (c < rem));
    } else {
        n_mine = U > blockIdx.x ? (int)((U - 1 - blockIdx.x) / grid + 1) : 0;
    }
    auto unit_id = [&](int i) -> int64_t { return lpt ? mine[i] : blockIdx.x + i * grid; };
    // every role walks the same units: decode them once into shared memory
    Unit *units_s = reinterpret_cast<Unit *>(smem + kOffUnits);
    const bool cached = n_mine <= kMaxMine;
    if (cached) {
        for (int i = threadIdx.x; i < n_mine; i += kThreads) units_s[i] = unit_at(a, pre, unit_id(i), T);
        __syncthreads();
    }
    auto unit_i = [&](int i) -> Unit { return cached ? units_s[i] : unit_at(a, pre, unit_id(i), T); };

    if (warp == 0 || warp == kWarpV) {
        // ================= TMA producers (warp 0: Q and K, last warp: V) =================
        const bool is_v = warp == kWarpV;
        int64_t j = 0;   // key-tile sequence number in this CTA
        int uq = 0;      // units with key tiles
        for (int i = 0; i < n_mine && !*abort_flag; ++i) {
            const Unit x = unit_i(i);
            if (x.nk == 0) continue;
            if (!is_v) {
                if (!mbar_wait_warp(bar_qempty, (uint32_t)(uq & 1) ^ 1u, abort_flag)) break;
                if (lane == 0) {
                    const bool has_b = x.ntok[1] > 0;
                    mbar_arrive_expect_tx(bar_qfull, (has_b ? 2u : 1u) * (uint32_t)kTileBytes);
                    for (int xb = 0; xb < (has_b ? 2 : 1); ++xb) {
                        const int tq = (int)(x.t0 + x.tok0 + xb * T);
                        const uint32_t dq = sm_q + xb * kTileBytes;
                        tma_load_3d(dq, &tmQ, bar_qfull, 0, x.g * G, tq);
                        tma_load_3d(dq + kHalfBytes, &tmQ, bar_qfull, 64, x.g * G, tq);
                    }
                }
            }
            // block entry of this lane's segment of key tile kt: the row to load, or -1
            auto entry = [&](int kt) -> int64_t {
                if (lane >= nseg) return -1;
                const int32_t p0 = kt * kTile + lane * seg_rows;
                if (p0 >= x.kend) return -1;
                const int32_t lb = p0 / a.bs;
                if (lb >= a.bt_cols) {
                    if (!is_v && a.err) atomicAdd(a.err, 1);
                    return -1;
                }
                const int64_t e = __ldg(a.bt + (int64_t)x.r * a.bt_stride + lb);
                if (e <= 0) return -1;
                if (e >= a.total_blocks) {
                    if (!is_v && a.err) atomicAdd(a.err, 1);
                    return -1;
                }
                return e * a.bs + (p0 - (int64_t)lb * a.bs);
            };
            int64_t row_cur = entry(0);
            for (int kt = 0; kt < x.nk; ++kt, ++j) {
                const int64_t row_nxt = kt + 1 < x.nk ? entry(kt + 1) : -1;   // in flight meanwhile
                const int s = (int)(j % kStages);
                const uint32_t bar_e = is_v ? bar_vempty(s) : bar_kempty(s);
                const uint32_t bar_f = is_v ? bar_vfull(s) : bar_kfull(s);
                if (!mbar_wait_warp(bar_e, (uint32_t)((j / kStages) & 1) ^ 1u, abort_flag)) break;
                const bool load = row_cur >= 0;
                const uint32_t ballot = __ballot_sync(0xffffffffu, load);
                if (lane == 0) {
                    // the mask word ring is written at most a few tiles ahead of its
                    // readers (two K slots, one S per softmax), well inside its 8 entries
                    if (!is_v) {
                        mask_words[j & 7] = ballot;
                        mbar_arrive(bar_mask((int)(j & 7)));
                    }
                    mbar_arrive_expect_tx(bar_f, (uint32_t)__popc(ballot) * (uint32_t)seg_rows * 128u * 2u);
                }
                __syncwarp();
                if (load) {
                    const uint32_t dst = (is_v ? sm_v : sm_k) + s * kTileBytes + lane * seg_rows * 128;
                    const CUtensorMap *map = is_v ? &tmV : &tmK;
                    tma_load_3d(dst, map, bar_f, 0, x.g, (int)row_cur);
                    tma_load_3d(dst + kHalfBytes, map, bar_f, 64, x.g, (int)row_cur);
                }
                __syncwarp();
                row_cur = row_nxt;
            }
            ++uq;
        }
        if (*abort_flag) {
            const unsigned long long t0 = global_ns();
            while (global_ns() - t0 < 200000ull) {
            }
        }
    } else if (warp == 1) {
        // ================= MMA issuer (one thread) =================
        if (lane == 0) {
            constexpr uint32_t kIdescS = idesc_bf16(128, 128, 0, 0);   // Q (K-major) x K (K-major)
            constexpr uint32_t kIdescO = idesc_bf16(128, 128, 0, 1);   // P (TMEM) x V (MN-major)
            int64_t j = 0;
            int uq = 0;
            int np[2] = {0, 0};   // P tiles of A / B consumed so far
            int nu[2] = {0, 0};   // units of A / B started so far
            bool ok = true;
            // O_X += P_X(tile) V(stage): the unit's first P V (first) overwrites O_X,
            // so it waits until softmax X has read the previous unit's O_X out
            auto issue_pv = [&](int xb, int stage, bool first) -> bool {
                if (!mbar_wait(bar_pfull(xb), (uint32_t)(np[xb] & 1), abort_flag)) return false;
                ++np[xb];
                if (first && nu[xb] > 1 && !mbar_wait(bar_oempty(xb), (uint32_t)((nu[xb] - 2) & 1), abort_flag))
                    return false;
                tc_fence_after();
                const uint32_t v_base = sm_v + stage * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk) {
                    const uint64_t bdesc = sdesc(v_base + kk * 2048, kHalfBytes, 1024);
                    // keys 16 kk .. 16 kk + 15: P of keys 0..63 is packed over S columns 0..31
                    // and that of keys 64..127 over columns 64..95 (each key half's own columns)
                    const uint32_t pcol = (kk < 4 ? 0u : 64u) + 8u * (uint32_t)(kk & 3);
                    mma_bf16_ts(tmem + col_o(xb), tmem + col_s(xb) + pcol, bdesc, kIdescO,
                                (first && kk == 0) ? 0u : 1u);
                }
                return true;
            };
            auto issue_s = [&](int xb, int stage) {
                const uint32_t k_base = sm_k + stage * kTileBytes;
                const uint32_t q_base = sm_q + xb * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint32_t off = (uint32_t)(kk >> 2) * kHalfBytes + (kk & 3) * 32;
                    mma_bf16(tmem + col_s(xb), sdesc(q_base + off, 16, 1024), sdesc(k_base + off, 16, 1024), kIdescS,
                             kk > 0 ? 1u : 0u);
                }
                mma_commit(bar_sfull(xb));
            };
            for (int i = 0; ok && i < n_mine; ++i) {
                const Unit x = unit_i(i);
                if (x.nk == 0) continue;
                const bool has_b = x.ntok[1] > 0;
                ++nu[0];
                if (has_b) ++nu[1];
                if (!mbar_wait(bar_qfull, (uint32_t)(uq & 1), abort_flag)) {
                    ok = false;
                    break;
                }
                for (int kt = 0; ok && kt <= x.nk; ++kt, ++j) {
                    // P V of the previous key tile, then S of this one, tile A then B
                    const int sp = (int)((j - 1) % kStages);
                    if (kt > 0 && !mbar_wait(bar_vfull(sp), (uint32_t)(((j - 1) / kStages) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int s = (int)(j % kStages);
                    if (kt < x.nk && !mbar_wait(bar_kfull(s), (uint32_t)((j / kStages) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int xb = 0; xb < (has_b ? 2 : 1); ++xb) {
                        if (kt > 0 && !issue_pv(xb, sp, kt == 1)) {
                            ok = false;
                            break;
                        }
                        if (kt == x.nk) mma_commit(bar_ofull(xb));
                        if (kt < x.nk) issue_s(xb, s);
                    }
                    if (!ok) break;
                    if (kt > 0) mma_commit(bar_vempty(sp));
                    if (kt < x.nk) {
                        mma_commit(bar_kempty(s));
                        if (kt == x.nk - 1) mma_commit(bar_qempty);
                    }
                }
                --j;   // the loop ran nk + 1 turns for nk key tiles
                ++uq;
            }
        }
        __syncwarp();
    } else if (warp < kWarpV) {
        // ====== softmax (warps 2..9: tile A, 10..17: tile B; per tile one warpgroup per half of the
        // ====== keys, one query row per thread) ======
        const int xb = (warp - 2) >> 3;                  // query tile of this warpgroup
        const int kh = ((warp - 2) >> 2) & 1;            // its half of each key tile: keys [64 kh, 64 kh + 64)
        const int qw = warp & 3;                         // TMEM lane quarter this warp may access
        const int row = 32 * qw + lane;                  // query row of the tile: token row / G, head row % G
        const uint32_t lane_base = (uint32_t)(32 * qw) << 16;
        const int tt = row / G;
        const int hh = row - tt * G;
        const uint32_t s_col = tmem + lane_base + col_s(xb);
        const uint32_t o_col = tmem + lane_base + col_o(xb);
        int64_t j = 0;       // key-tile sequence number in this CTA (the mask ring)
        int ns = 0;          // S tiles of this query tile seen so far
        int no = 0;          // units of this query tile finished so far
        bool ok = true;
        // Bounded exchange point of this warp and the warp that holds the other key half of the
        // same rows (an mbarrier, so that a timed-out wait elsewhere never leaves a warp stuck)
        uint32_t pphase = 0;
        auto pair_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_pair(xb, qw));
            const bool r = mbar_wait_warp(bar_pair(xb, qw), pphase, abort_flag);
            pphase ^= 1u;
            return r;
        };
        float *xmax = reinterpret_cast<float *>(smem + kOffXmax) + xb * (2 * 2 * kTile);   // [half][parity][row]
        float *xsum = reinterpret_cast<float *>(smem + kOffXsum) + xb * (2 * kTile);       // [half][row]
        for (int i = 0; ok && i < n_mine; ++i) {
            const Unit x = unit_i(i);
            const int ntok = x.ntok[xb];
            if (ntok <= 0) {      // no tile B in this unit
                j += x.nk;
                continue;
            }
            const bool valid = row < G * T && tt < ntok;
            const int32_t tok = x.tok0 + xb * T + tt;                    // this row's token (of the request)
            const int32_t pos = x.L - x.ql + tok;                        // and its position
            const int32_t lastv = a.mask_mode == 0 ? pos : x.L - 1;
            const bool warp_valid = __any_sync(0xffffffffu, valid);
            __nv_bfloat16 *out =
                static_cast<__nv_bfloat16 *>(a.out) + ((x.t0 + tok) * a.H_q + (int64_t)x.g * G + hh) * kD;
            if (x.nk == 0) {   // nothing visible: this half's 64 output values are 0
                if (valid)
                    for (int d = 64 * kh; d < 64 * kh + 64; d += 8)
                        *reinterpret_cast<uint4 *>(out + d) = make_uint4(0, 0, 0, 0);
                continue;
            }
            float m = -INFINITY, l = 0.f;
            for (int kt = 0; kt < x.nk; ++kt, ++j) {
                const int s = (int)(j % kStages);
                if (!mbar_wait_warp(bar_sfull(xb), (uint32_t)(ns & 1), abort_flag) ||
                    !mbar_wait_warp(bar_mask((int)(j & 7)), (uint32_t)((j >> 3) & 1), abort_flag)) {
                    ok = false;
                    break;
                }
                ++ns;
                tc_fence_after();
                const uint32_t mword = mask_words[j & 7];
                const int32_t k0 = kt * kTile;
                // This row sees keys k < lim of the tile (cache end and causal bound),
                // and only those of loaded segments; invalid rows see none.
                int32_t lim = min(x.L, lastv + 1) - k0;
                lim = valid ? max(0, min(kTile, lim)) : 0;
                const bool segs = mword == all_seg;   // no null entry in the tile
                // Visible keys [32c, 32c + 32) of the tile as a bit mask: below lim, and in
                // a loaded segment (segments of seg_rows keys, one bit each in mword).
                auto vis32 = [&](int c) -> uint32_t {
                    const int lo = 32 * c;
                    uint32_t v = lim >= lo + 32 ? 0xffffffffu : (lim > lo ? (1u << (lim - lo)) - 1u : 0u);
                    if (!segs) {
                        uint32_t sb;
                        if (seg_rows >= 32) {
                            sb = ((mword >> (lo >> seg_shift)) & 1u) ? 0xffffffffu : 0u;
                        } else {
                            const int per = 32 >> seg_shift;            // segments in the chunk: 2 or 4
                            const uint32_t ones = (1u << seg_rows) - 1u;
                            const uint32_t bits = mword >> (lo >> seg_shift);
                            sb = 0u;
                            for (int i = 0; i < per; ++i)
                                if ((bits >> i) & 1u) sb |= ones << (i * seg_rows);
                        }
                        v &= sb;
                    }
                    return v;
                };
                // Every key of this half visible to every row of this warp (the common
                // case inside a long prefix): no per-key tests.
                const bool full = __all_sync(0xffffffffu, lim >= 64 * kh + 64) && segs;
                // A warp with no valid row does no softmax work: its P rows feed O rows
                // that are never stored, and the MMA keeps rows apart.
                // V rows loaded past the cache end (the last segment's tail) must be zero
                // for P V; softmax A clears them (every warp its 32 rows of the tile)
                // once the V tile has landed; P V of tile B is issued after that of A.
                auto zero_v_rows = [&]() -> bool {
                    if (xb != 0 || kh != 0) return true;
                    const bool zero_row = ((mword >> (row >> seg_shift)) & 1u) && k0 + row >= x.L;
                    if (!__any_sync(0xffffffffu, zero_row)) return true;
                    if (!mbar_wait_warp(bar_vfull(s), (uint32_t)((j / kStages) & 1), abort_flag)) return false;
                    if (zero_row) {
                        uint4 *v0 = reinterpret_cast<uint4 *>(smem + kOffV + s * kTileBytes + row * 128);
                        uint4 *v1 = reinterpret_cast<uint4 *>(smem + kOffV + s * kTileBytes + kHalfBytes + row * 128);
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            v0[c] = make_uint4(0, 0, 0, 0);
                            v1[c] = make_uint4(0, 0, 0, 0);
                        }
                    }
                    fence_proxy_async();
                    return true;
                };
                if (!warp_valid) {
                    if (!zero_v_rows()) {
                        ok = false;
                        break;
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_pfull(xb));
                    continue;
                }
                // pass 1: this half's max of the raw scores (the scale is positive), as a tree,
                // then the tile max of the row from the two halves
                float mraw = -INFINITY;
#pragma unroll 1
                for (int c = 2 * kh; c < 2 * kh + 2; ++c) {
                    float sv[32];
                    tmem_ld32(s_col + 32u * c, sv);
                    if (!full) {
                        const uint32_t vm = vis32(c);
#pragma unroll
                        for (int k = 0; k < 32; ++k) sv[k] = (vm & (1u << k)) ? sv[k] : -INFINITY;
                    }
                    mraw = fmaxf(mraw, tree_max32(sv));
                }
                float *xm = xmax + (int)(j & 1) * kTile;     // this tile's exchange slots, parity j
                xm[kh * 2 * kTile + row] = mraw;
                if (!pair_sync()) {
                    ok = false;
                    break;
                }
                mraw = fmaxf(mraw, xm[(1 - kh) * 2 * kTile + row]);
                const float mt = mraw * a.scale_log2;
                // Lazy rescale: the reference max m moves (and O, l are rescaled) only
                // when the tile max passes it by more than kSlack, so weights stay
                // below 2^kSlack and most tiles leave O alone.  Both halves take the same
                // decision from the same maximum.
                const bool bump = mt > m + kSlack;
                const float mn = bump ? mt : m;
                const float corr = bump ? fast_exp2(m - mn) : 1.f;
                // O_X(kt - 1) completed before S_X(kt) did: rescale this half's 64 columns of it
                if (kt > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll 1
                    for (int c = 2 * kh; c < 2 * kh + 2; ++c) {
                        float ov[32];
                        tmem_ld32(o_col + 32u * c, ov);
#pragma unroll
                        for (int k = 0; k < 32; ++k) ov[k] *= corr;
                        tmem_st32(o_col + 32u * c, ov);
                    }
                }
                // pass 2: weights 2^(s * scale - mn) (0 where masked), their sum, and P (bf16)
                // packed over the first 32 of this half's 64 S columns: chunk c's 8 packed
                // columns lie at or below the 16 columns of the chunk just read
                float psum = 0.f;
                {
                    const float nb = -mn;
                    uint32_t vm = 0;
#pragma unroll 1
                    for (int c = 4 * kh; c < 4 * kh + 4; ++c) {
                        float sv[16];
                        tmem_ld16(s_col + 16u * c, sv);
                        if (full) {
#pragma unroll
                            for (int k = 0; k < 16; ++k) sv[k] = fast_exp2(fmaf(sv[k], a.scale_log2, nb));
                        } else {
                            if ((c & 1) == 0) vm = vis32(c >> 1);
                            const uint32_t vh = (c & 1) ? (vm >> 16) : vm;
#pragma unroll
                            for (int k = 0; k < 16; ++k) {
                                // computed for every key, then selected: no branch per key
                                const float e = fast_exp2(fmaf(sv[k], a.scale_log2, nb));
                                sv[k] = (vh & (1u << k)) ? e : 0.f;
                            }
                        }
                        uint32_t pk[8];
#pragma unroll
                        for (int k = 0; k < 16; k += 2) {
                            const __nv_bfloat162 pb = __floats2bfloat162_rn(sv[k], sv[k + 1]);
                            pk[k >> 1] = *reinterpret_cast<const uint32_t *>(&pb);
                            psum += sv[k] + sv[k + 1];
                        }
                        tmem_st8(s_col + 64u * kh + 8u * (c & 3), pk);
                    }
                    tmem_st_wait();
                }
                l = fmaf(l, corr, psum);
                m = mn;
                if (!zero_v_rows()) {
                    ok = false;
                    break;
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_pfull(xb));
            }
            if (!ok) break;
            // the unit's last P V, then this row's output; O_X is free again after
            if (!mbar_wait_warp(bar_ofull(xb), (uint32_t)(no & 1), abort_flag)) {
                ok = false;
                break;
            }
            ++no;
            tc_fence_after();
            // the row's weight sum from the two halves (both warps of a pair have the same rows,
            // so they take this exchange together or skip it together)
            if (warp_valid) {
                xsum[kh * kTile + row] = l;
                if (!pair_sync()) {
                    ok = false;
                    break;
                }
                l += xsum[(1 - kh) * kTile + row];
            }
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int c = 2 * kh; c < 2 * kh + 2; ++c) {
                float ov[32];
                tmem_ld32(o_col + 32u * c, ov);
                if (valid) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const __nv_bfloat162 h2 =
                                __floats2bfloat162_rn(ov[8 * q4 + 2 * e] * inv, ov[8 * q4 + 2 * e + 1] * inv);
                            w[e] = *reinterpret_cast<const uint32_t *>(&h2);
                        }
                        *reinterpret_cast<uint4 *>(out + 32 * c + 8 * q4) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_oempty(xb));
        }
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0 && a.err) atomicAdd(a.err, kTimeoutErr);
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

static bool encode_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1_bytes,
                      uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {s1_bytes, s2_bytes};
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace rtc

bool prepare_ragged_tc(const RaggedArgs &a, RaggedTc *t) {
    using namespace rtc;
    if (a.dtype != BKV_BF16 || a.D != kD || a.G < 1 || a.G > 128) return false;
    if (a.bs < 8 || !((kTile % a.bs == 0) || (a.bs % kTile == 0))) return false;
    if (a.num_reqs > kMaxReqs || a.num_tokens >= ((int64_t)1 << 31) || a.H_kv > 65535) return false;
    if ((int64_t)a.total_blocks * a.bs >= ((int64_t)1 << 31) || a.total_blocks <= 0) return false;
    // the unit prefix stays within int32 (a request has at most max_q query tiles per KV head)
    if ((int64_t)a.num_reqs * a.H_kv * a.max_q >= ((int64_t)1 << 31)) return false;
    if (!aligned(a.k, 16) || !aligned(a.v, 16) || !aligned(a.q, 16) || !aligned(a.out, 16)) return false;
    if (!encode_fn()) return false;
    t->seg_rows = a.bs < kTile ? a.bs : kTile;
    t->tok_per_tile = kTile / a.G;
    const uint64_t rows = (uint64_t)a.total_blocks * (uint64_t)a.bs;
    const uint64_t row_stride = (uint64_t)a.H_kv * kD * 2;
    return encode_3d(&t->mk, a.k, kD, a.H_kv, rows, kD * 2, row_stride, 64, 1, t->seg_rows) &&
           encode_3d(&t->mv, a.v, kD, a.H_kv, rows, kD * 2, row_stride, 64, 1, t->seg_rows) &&
           encode_3d(&t->mq, a.q, kD, a.H_q, (uint64_t)a.num_tokens, kD * 2, (uint64_t)a.H_q * kD * 2, 64, a.G,
                     t->tok_per_tile);
}

int launch_ragged_tc(const RaggedArgs &a, const RaggedTc &t, cudaStream_t st) {
    using namespace rtc;
    auto kern = ragged_tc_kernel<0>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
            return launch_status();
        attr_set[dev] = true;
    }
    const cudaError_t e = launch_pdl(kern, dim3((unsigned)current_sm_count()), dim3(kThreads), kSmemBytes, st, t.mk,
                                     t.mv, t.mq, a, t.seg_rows, t.tok_per_tile);
    if (e != cudaSuccess) set_cuda_error(e);
    return launch_status();
}

}  // namespace bkv
