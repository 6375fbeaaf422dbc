// bkv_ragged_tc.cu -- tensor-core (tcgen05 + TMA) prefill kernel of the
// mixed-step attention: bf16, head_dim 128, query tiles of 128 rows.
//
// Operation ("Padding and Batching with Block KV", Batching with Block KV
// and Cache Masking; see bkv_ragged.cu): each query token of a request
// attends, at its own position, over the request's paged keys.
//
// Design (sm_103a):
// * Work unit = (request r, KV head g, query tile qt): the T = 128 / G query
//   tokens qt T, ... of r for the G query heads of g, 128 rows ordered
//   (token, head) -- exactly the box a 3-D TMA load of q (head_dim, H_q,
//   tokens) delivers.  Persistent CTAs (one per SM) take units round robin.
// * Warp roles: warp 0 loads Q (per unit) and gathers K tiles, the last warp
//   gathers V tiles (2-slot rings of 128 keys, 32 KB), warp 1 issues
//   tcgen05.mma from one thread, warps 2..5 run the softmax, one query row
//   (TMEM lane) per thread.
// * S = Q K^T (M = 128 query rows, N = 128 keys, K = head_dim; both operands
//   K-major from the TMA tiles) into one of two TMEM buffers; the softmax
//   reads its row in 32-column chunks (max pass, then exponentials), keeps
//   the running max and sum, and writes P (bf16, K-major, 128-byte swizzle).
//   The running max is a lazy reference: it moves only when a tile's max
//   passes it by more than 8 (log2 units), so weights stay below 2^8 and O
//   is rescaled only on those tiles; a tile every key of which is visible
//   to all rows of a warp skips the per-key mask tests.
// * O += P V (N = head_dim, V read MN-major straight from the TMA tile)
//   accumulates in TMEM across the unit's key tiles; when a row's reference
//   max moves the softmax rescales its O row in TMEM (only warps with such a
//   row do).
// * Keys are gathered through the block table with one TMA load per block
//   segment and head_dim half; null and out-of-range entries are not loaded,
//   positions past the causal bound of the tile's last token are not loaded,
//   and V rows loaded past the cache end are zeroed before P V.
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
constexpr int kThreads = 224;                // K producer, MMA, 4 softmax warps, V producer
constexpr int kWarpV = kThreads / 32 - 1;
constexpr int kTmemCols = 512;               // S x2 (128 columns each) + O (128)
constexpr uint32_t kColO = 256;
constexpr int kTimeoutErr = 1 << 24;
constexpr int kMaxReqs = 2048;

constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffQ = kOffV + kStages * kTileBytes;
constexpr int kOffP = kOffQ + kTileBytes;
constexpr int kOffMask = kOffP + kTileBytes;             // 8 words: loaded segments per tile (ring)
constexpr int kOffBar = kOffMask + 64;
constexpr int kNumBars = 4 * kStages + 2 + 2 + 1 + 1 + 8;
constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
constexpr int kOffPre = (kOffAbort + 4 + 15) / 16 * 16;  // [kMaxReqs + 1] units before request r
constexpr int kSmemUsed = kOffPre + (kMaxReqs + 1) * 4;
constexpr int kSmemBytes = kSmemUsed + 1024;             // slack for 1024 alignment
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA exceeds the sm_103a limit");

// One unit of work and the facts every role derives from it.
struct Unit {
    int r, g;
    int64_t t0;          // first packed token of the request
    int32_t ql, L;       // query tokens and cache length of the request
    int32_t tok0, ntok;  // the tile's tokens: [tok0, tok0 + ntok) of the request
    int32_t kend;        // keys [0, kend) may be visible to some row of the tile
    int32_t nk;          // key tiles
};

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
    const int qtiles = ceil_div_i(q.ql, T);
    const int64_t v = u - pre[lo];
    x.g = (int)(v / qtiles);
    const int qt = (int)(v - (int64_t)x.g * qtiles);
    x.tok0 = qt * T;
    x.ntok = min(T, q.ql - x.tok0);
    const int32_t plast = q.L - q.ql + x.tok0 + x.ntok - 1;   // position of the tile's last token
    int32_t kend = a.mask_mode == 0 ? min(q.L, plast + 1) : q.L;
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
    auto bar_sfull = [&](int b) { return bar0 + 8u * (4 * kStages + 2 + b); };
    const uint32_t bar_pfull = bar0 + 8u * (4 * kStages + 4);
    const uint32_t bar_ofull = bar0 + 8u * (4 * kStages + 5);
    auto bar_mask = [&](int m) { return bar0 + 8u * (4 * kStages + 6 + m); };
    const uint32_t sm_k = sbase + kOffK;
    const uint32_t sm_v = sbase + kOffV;
    const uint32_t sm_q = sbase + kOffQ;
    const uint32_t sm_p = sbase + kOffP;

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
        mbar_init(bar_sfull(0), 1);
        mbar_init(bar_sfull(1), 1);
        mbar_init(bar_pfull, 4);
        mbar_init(bar_ofull, 1);
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
        // V ring, Q and P start at zero: a row no TMA load or softmax writes must
        // never hold uninitialised bits (NaN) that an MMA could read
        const uint4 z = make_uint4(0, 0, 0, 0);
        uint4 *v = reinterpret_cast<uint4 *>(smem + kOffV);
        for (int i = threadIdx.x; i < (kStages + 2) * kTileBytes / 16; i += kThreads) v[i] = z;
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
    // units per request (H_kv * query tiles), then their exclusive prefix sum
    for (int r = threadIdx.x; r < a.num_reqs; r += kThreads) {
        const RaggedReq q = ragged_req(a, r);
        pre[r] = q.ql > 0 ? a.H_kv * ceil_div_i(q.ql, T) : 0;
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

    if (warp == 0 || warp == kWarpV) {
        // ================= TMA producers (warp 0: Q and K, last warp: V) =================
        const bool is_v = warp == kWarpV;
        int64_t j = 0;   // key-tile sequence number in this CTA
        int uq = 0;      // units with key tiles
        for (int64_t u = blockIdx.x; u < U && !*abort_flag; u += gridDim.x) {
            const Unit x = unit_at(a, pre, u, T);
            if (x.nk == 0) continue;
            if (!is_v) {
                if (!mbar_wait_warp(bar_qempty, (uint32_t)(uq & 1) ^ 1u, abort_flag)) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar_qfull, 2u * 128u * (uint32_t)(G * T));
                    const int tq = (int)(x.t0 + x.tok0);
                    tma_load_3d(sm_q, &tmQ, bar_qfull, 0, x.g * G, tq);
                    tma_load_3d(sm_q + kHalfBytes, &tmQ, bar_qfull, 64, x.g * G, tq);
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
                    // the mask word ring is written at most a few tiles ahead of its reader
                    // (two K slots, two S buffers), well inside its 8 entries
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
            constexpr uint32_t kIdescO = idesc_bf16(128, 128, 0, 1);   // P (K-major) x V (MN-major)
            int64_t j = 0;
            int uq = 0;
            int64_t pend = -1;   // key tile whose P.V is still to be issued
            bool pend_first = false;
            bool ok = true;
            auto issue_pv = [&](int64_t jp, bool first) -> bool {
                const int s = (int)(jp % kStages);
                if (!mbar_wait(bar_pfull, (uint32_t)(jp & 1), abort_flag) ||
                    !mbar_wait(bar_vfull(s), (uint32_t)((jp / kStages) & 1), abort_flag))
                    return false;
                tc_fence_after();
                const uint32_t v_base = sm_v + s * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kTile / 16; ++kk) {
                    const uint64_t adesc = sdesc(sm_p + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
                    const uint64_t bdesc = sdesc(v_base + kk * 2048, kHalfBytes, 1024);
                    mma_bf16(tmem + kColO, adesc, bdesc, kIdescO, (first && kk == 0) ? 0u : 1u);
                }
                mma_commit(bar_ofull);
                mma_commit(bar_vempty(s));
                return true;
            };
            for (int64_t u = blockIdx.x; ok && u < U; u += gridDim.x) {
                const Unit x = unit_at(a, pre, u, T);
                if (x.nk == 0) continue;
                if (!mbar_wait(bar_qfull, (uint32_t)(uq & 1), abort_flag)) {
                    ok = false;
                    break;
                }
                for (int kt = 0; kt < x.nk; ++kt, ++j) {
                    const int s = (int)(j % kStages);
                    const int b = (int)(j & 1);
                    if (!mbar_wait(bar_kfull(s), (uint32_t)((j / kStages) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t k_base = sm_k + s * kTileBytes;
#pragma unroll
                    for (int kk = 0; kk < kD / 16; ++kk) {
                        const uint32_t off = (uint32_t)(kk >> 2) * kHalfBytes + (kk & 3) * 32;
                        mma_bf16(tmem + 128u * b, sdesc(sm_q + off, 16, 1024), sdesc(k_base + off, 16, 1024), kIdescS,
                                 kk > 0 ? 1u : 0u);
                    }
                    mma_commit(bar_sfull(b));
                    mma_commit(bar_kempty(s));
                    if (kt == x.nk - 1) mma_commit(bar_qempty);
                    if (pend >= 0 && !issue_pv(pend, pend_first)) {
                        ok = false;
                        break;
                    }
                    pend = j;
                    pend_first = kt == 0;
                }
                ++uq;
            }
            if (ok && pend >= 0) issue_pv(pend, pend_first);
        }
        __syncwarp();
    } else {
        // ================= softmax (warps 2..5: one query row per thread) =================
        const int qw = warp & 3;                         // TMEM lane quarter this warp may access
        const int row = 32 * qw + lane;                  // query row of the tile: token row / G, head row % G
        const uint32_t lane_base = (uint32_t)(32 * qw) << 16;
        const int tt = row / G;
        const int hh = row - tt * G;
        // this thread's bytes in P (K-major, 128-byte swizzle): row `row`, 16-byte chunk c of key half h
        auto p_addr = [&](int h, int c) -> uint8_t * {
            return smem + kOffP + h * kHalfBytes + (row >> 3) * 1024 + (row & 7) * 128 + ((c ^ (row & 7)) << 4);
        };
        int64_t j = 0;
        bool ok = true;
        for (int64_t u = blockIdx.x; ok && u < U; u += gridDim.x) {
            const Unit x = unit_at(a, pre, u, T);
            const bool valid = row < G * T && tt < x.ntok;
            const int32_t pos = x.L - x.ql + x.tok0 + tt;           // this row's token position
            const int32_t lastv = a.mask_mode == 0 ? pos : x.L - 1;
            const bool warp_valid = __any_sync(0xffffffffu, valid);
            __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out) +
                                 ((x.t0 + x.tok0 + tt) * a.H_q + (int64_t)x.g * G + hh) * kD;
            if (x.nk == 0) {
                if (valid)
                    for (int d = 0; d < kD; d += 8) *reinterpret_cast<uint4 *>(out + d) = make_uint4(0, 0, 0, 0);
                continue;
            }
            float m = -INFINITY, l = 0.f;
            for (int kt = 0; kt < x.nk; ++kt, ++j) {
                const int b = (int)(j & 1);
                const int s = (int)(j % kStages);
                if (!mbar_wait_warp(bar_sfull(b), (uint32_t)((j >> 1) & 1), abort_flag) ||
                    !mbar_wait_warp(bar_mask((int)(j & 7)), (uint32_t)((j >> 3) & 1), abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t mword = mask_words[j & 7];
                const int32_t k0 = kt * kTile;
                // This row sees keys k < lim of the tile (cache end and causal bound),
                // and only those of loaded segments; invalid rows see none.
                int32_t lim = min(x.L, lastv + 1) - k0;
                lim = valid ? max(0, min(kTile, lim)) : 0;
                const bool segs = mword == all_seg;   // no null entry in the tile
                auto seen = [&](int k) { return k < lim && (segs || ((mword >> (k >> seg_shift)) & 1u)); };
                // Every key of the tile visible to every row of this warp (the common
                // case inside a long prefix): no per-key tests.
                const bool full = __all_sync(0xffffffffu, lim == kTile) && segs;
                // pass 1: the tile max of the raw scores (the scale is positive), as a tree
                float mraw = -INFINITY;
                if (warp_valid) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float sv[32];
                        tmem_ld32(tmem + lane_base + 128u * b + 32u * c, sv);
                        if (!full) {
#pragma unroll
                            for (int k = 0; k < 32; ++k) sv[k] = seen(32 * c + k) ? sv[k] : -INFINITY;
                        }
                        mraw = fmaxf(mraw, tree_max32(sv));
                    }
                }
                const float mt = mraw * a.scale_log2;
                // Lazy rescale: the reference max m moves (and O, l are rescaled) only
                // when the tile max passes it by more than kSlack, so weights stay
                // below 2^kSlack and most tiles leave O alone.
                const bool bump = mt > m + kSlack;
                const float mn = bump ? mt : m;
                const float corr = bump ? fast_exp2(m - mn) : 1.f;
                // the previous tile's P.V must be done before P and O are touched
                if (kt > 0) {
                    if (!mbar_wait_warp(bar_ofull, (uint32_t)((j - 1) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (warp_valid && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            float ov[32];
                            tmem_ld32(tmem + lane_base + kColO + 32u * c, ov);
#pragma unroll
                            for (int k = 0; k < 32; ++k) ov[k] *= corr;
                            tmem_st32(tmem + lane_base + kColO + 32u * c, ov);
                        }
                    }
                }
                if (warp_valid) {
                    // pass 2: weights 2^(s * scale - mn) (0 where masked), their sum, P in bf16
                    const float nb = -mn;
                    float psum = 0.f;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float sv[32];
                        tmem_ld32(tmem + lane_base + 128u * b + 32u * c, sv);
                        if (full) {
#pragma unroll
                            for (int k = 0; k < 32; ++k) sv[k] = fast_exp2(fmaf(sv[k], a.scale_log2, nb));
                        } else {
#pragma unroll
                            for (int k = 0; k < 32; ++k) {
                                // computed for every key, then selected: no branch per key
                                const float e = fast_exp2(fmaf(sv[k], a.scale_log2, nb));
                                sv[k] = seen(32 * c + k) ? e : 0.f;
                            }
                        }
                        uint32_t pk[16];
#pragma unroll
                        for (int k = 0; k < 32; k += 2) {
                            const __nv_bfloat162 pb = __floats2bfloat162_rn(sv[k], sv[k + 1]);
                            pk[k >> 1] = *reinterpret_cast<const uint32_t *>(&pb);
                        }
                        psum += tree_sum32(sv);
                        // keys 32c .. 32c + 31: half c / 2, 16-byte chunks 4 (c % 2) .. + 3
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
                            *reinterpret_cast<uint4 *>(p_addr(c >> 1, 4 * (c & 1) + q4)) =
                                make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
                    }
                    l = fmaf(l, corr, psum);
                    m = mn;
                }
                // V rows loaded past the cache end (the last segment's tail) must be zero
                // for P.V; any thread may clear any row once the V tile has landed
                const bool zero_row = ((mword >> (row >> seg_shift)) & 1u) && k0 + row >= x.L;
                if (__any_sync(0xffffffffu, zero_row)) {
                    if (!mbar_wait_warp(bar_vfull(s), (uint32_t)((j / kStages) & 1), abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (zero_row) {
                        uint4 *v0 = reinterpret_cast<uint4 *>(smem + kOffV + s * kTileBytes + row * 128);
                        uint4 *v1 = reinterpret_cast<uint4 *>(smem + kOffV + s * kTileBytes + kHalfBytes + row * 128);
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            v0[c] = make_uint4(0, 0, 0, 0);
                            v1[c] = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_pfull);
            }
            if (!ok) break;
            // the unit's last P.V, then this row's output
            if (!mbar_wait_warp(bar_ofull, (uint32_t)((j - 1) & 1), abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float ov[32];
                tmem_ld32(tmem + lane_base + kColO + 32u * c, ov);
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
