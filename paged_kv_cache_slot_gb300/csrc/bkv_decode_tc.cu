// bkv_decode_tc.cu -- tensor-core (tcgen05 + TMA) partition kernel of the
// paged decode, bf16 queries, bf16 or FP8 (E4M3) caches, head_dim 128, up to
// 16 query rows per KV head.
//
// Operation ("Padding and Batching with Block KV", Cache Masking; Special
// Block and Slot Values): for a run of consecutive 128-position tiles of one
// stream (request r, KV head g), compute for every query row n = t * G + hh
// of the GQA group the online-softmax partial (o, m, l) over the visible
// positions of those tiles.  The merge kernel in bkv_decode.cu combines the
// partials of each stream.
//
// Design (sm_103a):
// * Head-grouped stream-K schedule.  The persistent grid (one CTA per SM)
//   is P groups of H_kv CTAs.  The requests' position tiles (ceil(len / 128)
//   per request, requests in order) are laid end to end and group q takes
//   [q * TP / P, (q + 1) * TP / P) of them, CTA g of the group for KV head
//   g, so every SM gets the same number of tiles to within one whatever the
//   mix of lengths, and the H_kv CTAs of a group read the same positions of
//   all heads at the same time: whole cache rows (a row holds every head of
//   one position), where a CTA alone would take a 128- or 256-byte piece
//   of each row.  Each overlap of a CTA range with a stream (request,
//   head) is a unit; it writes two partial slots (one per softmax
//   warpgroup), and a stream's slots are the contiguous range the merge
//   recomputes from the context lengths.
// * Warp roles: warp 0 gathers K tiles (and Q), warp 10 gathers V tiles,
//   warp 1 issues the S MMAs from one thread and owns the TMEM allocation,
//   warp 11 issues the P.V MMAs from one thread, and two warpgroups (warps
//   2..5 and 6..9) run the softmax and the output update on alternate
//   tiles.  K and V have separate rings (bf16: 3 slots of 32 KB each): a K
//   slot is released as soon as the S MMA that reads it completes, an S
//   tile as soon as its softmax warpgroup has read it, so the next S MMA
//   into that tile need not wait for the P.V MMA.
// * A tile's K (or V) rows of KV head g are gathered through the block
//   table with 3-D TMA loads (cp.async.bulk.tensor; map over (head_dim,
//   H_kv, total_blocks * block_size), box = 64 x 1 x min(block_size, 128)
//   rows, 128-byte swizzle), one load per block segment and head_dim half.
//   Null (<= 0) and out-of-range entries are not loaded at all and blocks
//   past the request's end are never touched, so the traffic is the
//   ceil(len / block_size) blocks actually needed.  Table entries are loaded
//   a window ahead into registers and parked in shared memory.
// * S^T[128 x 16] = K_tile . Q^T (M = positions, N = query rows padded to
//   16, K = head_dim), fp32 in TMEM.  Each softmax thread owns one position
//   (TMEM lane): masks by select, reduces the tile max per query row across
//   its warpgroup, exponentiates in base 2, keeps its partial row sums, and
//   writes P (bf16) to shared memory in the K-major swizzled layout.
// * O^T[128 x 16] = V_tile^T . P^T (M = head_dim, V read MN-major straight
//   from the TMA tile, K = positions); each softmax thread owns one head_dim
//   row of O^T and accumulates o = o * 2^(m_old - m_new) + O_tile.
// * V rows that were loaded but lie past the request's end are zeroed in
//   shared memory before the P.V MMA, so unwritten cache memory (which may
//   hold NaN) never reaches the output; K rows there are masked by select.
// * Every wait is bounded: after ~2 s a wait gives up, the CTA records an
//   error in *err_count (+ 1 << 24), lets copies in flight land, frees its
//   TMEM and exits.
// * FP8 caches (the reading of the cache format is stated in bkv.h): tiles
//   are 128 rows x 128 E4M3 codes (16 KB, one box per block segment).  S^T =
//   K . Q^T runs as kind::f8f6f4 on the codes straight from TMA, with q split
//   beforehand (q_split_e4m3_kernel) into two E4M3 parts whose sum is the
//   query row divided by a power of two, so the products are exact; the
//   softmax multiplies each column back.  O^T = V^T . P^T runs as
//   kind::f8f6f4 too, with V^T read MN-major straight from the E4M3 TMA
//   tile (one 128-code span per row) and P^T as two E4M3 parts, P 2^8 =
//   hi + lo, accumulated in one TMEM tile: the softmax never touches V.
//   (Widening V to f16 in the softmax warpgroups, the earlier design, made
//   the per-tile chain longer than the halved load time.)
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "bkv_decode.cuh"
#include "bkv_tc_ptx.cuh"

namespace bkv {
namespace tc {

constexpr int kTile = kDecodeTile;    // positions per tile
constexpr int kD = 128;               // head_dim handled
constexpr int kN = 16;                // query rows per MMA (padded)
// K and V tiles have separate rings of 32 KB slots
#ifndef BKV_K_STAGES
#define BKV_K_STAGES 3
#endif
#ifndef BKV_V_STAGES
#define BKV_V_STAGES 3
#endif
// tiles whose loaded-segment words are kept (a ring indexed by tile number)
constexpr int kMaskRing = 16;
static_assert(BKV_K_STAGES >= 2 && BKV_K_STAGES <= 3, "K slots of the bf16 ring");
// FP8 caches: slots of the E4M3 K and V rings (16 KB each, read by the MMAs as loaded)
#ifndef BKV_F8_K_STAGES
#define BKV_F8_K_STAGES 4
#endif
#ifndef BKV_F8_V_STAGES
#define BKV_F8_V_STAGES 4
#endif
static_assert(BKV_F8_K_STAGES >= 2 && BKV_F8_K_STAGES + 2 < kMaskRing, "the mask ring needs more than K slots + 2 words");
// FP8 caches: the weights enter the P.V MMA as p 2^kF8PExp (p <= 1, so at most
// 256 < 448, the largest finite E4M3 value); the partial output takes it back
constexpr int kF8PExp = 8;
constexpr int kHalfBytes = kTile * 128;          // 128 rows x 64 bf16 (128 B): one head_dim half
constexpr int kTileBytes = 2 * kHalfBytes;       // K or V tile: 32 KB
constexpr int kT8Bytes = kTile * 128;            // an FP8 K or V tile as loaded: 128 rows x 128 codes, 16 KB
constexpr int kQBytes = 2 * kN * 128;            // 16 rows x 128 B x 2 halves (FP8: 2 parts): 4 KB
constexpr int kPBytes = 2 * kN * 128;            // 16 rows x 128 positions, 2 x 64 bf16 or 2 E4M3 parts: 4 KB
constexpr int kWarpV = 10;                       // the V producer's warp
constexpr int kWarpPV = 11;                      // the P.V MMA issuer's warp
// TMEM: S tile b at columns 32 b, O tile b at 64 + 32 b (FP8: the hi and lo
// parts' products side by side, 16 columns each; bf16: the first 16)
constexpr int kTmemCols = 128;
constexpr int kTimeoutErr = 1 << 24;
constexpr int kMaxReqs = 2048;                   // requests the in-kernel tile prefix handles
constexpr int kWinBlocks = 128;                  // table entries a producer caches per window

// Shared-memory layout and role counts (offsets from a 1024-aligned base).
// kF8: FP8 caches.  Both MMAs run on E4M3 operands (kind::f8f6f4): K and V
// tiles straight from TMA, q as two E4M3 parts prepared by
// q_split_e4m3_kernel, P as two E4M3 parts written by the softmax.
template <bool kF8>
struct Cfg {
    // K producer, S MMA issuer, two softmax warpgroups, V producer, P.V MMA issuer
    static constexpr int kThreads = 384;
    static constexpr int kKStages = kF8 ? BKV_F8_K_STAGES : BKV_K_STAGES;
    static constexpr int kVStages = kF8 ? BKV_F8_V_STAGES : BKV_V_STAGES;
    static constexpr int kKSlot = kF8 ? kT8Bytes : kTileBytes;
    static constexpr int kVSlot = kKSlot;
    static constexpr int kOffK = 0;                                  // kKStages K slots
    static constexpr int kOffV = kOffK + kKStages * kKSlot;          // kVStages V slots
    static constexpr int kOffQ = kOffV + kVStages * kVSlot;
    static constexpr int kOffP = kOffQ + 2 * kQBytes;
    static constexpr int kOffMask = kOffP + 2 * kPBytes;             // kMaskRing words: loaded segments per tile
    static constexpr int kOffRedMax = kOffMask + 4 * kMaskRing;      // [warpgroup][2][16 rows][4 warps] floats
    static constexpr int kOffRedSum = kOffRedMax + 4 * kN * 4 * 4;   // [warpgroup][16 rows][4 warps] floats
    static constexpr int kOffBar = kOffRedSum + 2 * kN * 4 * 4;      // barriers (8 B each)
    static constexpr int kNumBars = 2 * kKStages + 2 * kVStages + 2 * 5 + 2 + kMaskRing + 2;
    static constexpr int kOffTmemSlot = kOffBar + kNumBars * 8;
    static constexpr int kOffAbort = kOffTmemSlot + 4;
    static constexpr int kOffPre = kOffAbort + 4;                    // [kMaxReqs + 1] tile prefix per request
    static constexpr int kOffEnt = (kOffPre + (kMaxReqs + 1) * 4 + 15) / 16 * 16;   // [producer][2][kWinBlocks]
    // [kMaxReqs] last-tile fill of each request minus one: with the tile count it
    // gives the clamped length without a global read, len = (tiles - 1) * 128 + fill
    static constexpr int kOffLrem = kOffEnt + 4 * kWinBlocks * 4;
    static constexpr int kSmemUsed = kOffLrem + kMaxReqs;
    static constexpr int kSmemBytes = kSmemUsed + 1024;              // slack for 1024 alignment
    static constexpr int kLensPerThread = (kMaxReqs + kThreads - 1) / kThreads;
    static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA exceeds the sm_103a limit");
    static_assert(kOffEnt % 16 == 0, "entry buffers must stay aligned");
    static_assert(kOffV % 1024 == 0 && kOffQ % 1024 == 0 && kOffP % 1024 == 0, "swizzled tiles need 1 KB alignment");
    static_assert(kWarpPV == kThreads / 32 - 1 && kWarpV == kWarpPV - 1, "warp roles");
};

// The first NQ accumulator columns of this thread's TMEM lane.
template <int NQ>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[NQ]) {
    if constexpr (NQ == 16) tmem_ld16(taddr, v);
    else if constexpr (NQ == 8) tmem_ld8(taddr, v);
    else tmem_ld4(taddr, v);
}

// FP8 caches: an S or O tile holds the products with the hi part in columns
// [0, 16) and with the lo part in [16, 32); the sum of the first NQ of each.
template <int NQ>
__device__ __forceinline__ void tmem_ld_sum2(uint32_t taddr, float (&v)[NQ]) {
    uint32_t h[NQ], l[NQ];
    if constexpr (NQ == 16) {
        tmem_ld16_nw(taddr, h);
        tmem_ld16_nw(taddr + 16u, l);
    } else if constexpr (NQ == 8) {
        tmem_ld8_nw(taddr, h);
        tmem_ld8_nw(taddr + 16u, l);
    } else {
        tmem_ld4_nw(taddr, h);
        tmem_ld4_nw(taddr + 16u, l);
    }
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < NQ; ++i) v[i] = __uint_as_float(h[i]) + __uint_as_float(l[i]);
}

// A ring slot and its phase parity, advanced one tile at a time (no division
// by the ring size on the per-tile path).
struct Ring {
    int slot = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void advance(int n) {
        if (++slot == n) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// ---------------------------------------------------------------------------
// Stream-K schedule
// ---------------------------------------------------------------------------
// The schedule's global reads, issued together right after the grid
// dependency wait: every thread loads its share of context_lens (one round
// trip for up to kMaxReqs requests) and prefetches a slice of the block table
// into L2, so that the producers' first table reads hit L2; the V ring is
// zeroed while those loads are in flight (a V row that no TMA load writes
// must hold zeros, never uninitialised bits, for the P.V MMA).  Leaves the
// tile count of request r in pre[r] and its last tile's fill in lrem[r]; a
// length above the host bound is clamped to it and counted once (CTA 0).
// The caller orders the V-ring stores before the TMA writes (proxy fence +
// barrier).
template <bool kF8>
__device__ void schedule_loads(const DecodeArgs &a, int32_t *pre, uint8_t *lrem, uint8_t *smem) {
    using C = Cfg<kF8>;
    constexpr int kThreads = C::kThreads;
    constexpr int kLensPerThread = C::kLensPerThread;
    const int n = a.num_reqs;
    int32_t lens[kLensPerThread];
#pragma unroll
    for (int i = 0; i < kLensPerThread; ++i) {
        const int r = threadIdx.x + i * kThreads;
        lens[i] = r < n ? __ldg(a.ctx + r) : 0;
    }
    {
        // 128-byte lines of the table rows, at most two per thread of the grid
        const int64_t lines_per_row = ((int64_t)a.bt_cols + 31) / 32;
        const int64_t lines = lines_per_row * n;
        const int64_t nthr = (int64_t)gridDim.x * kThreads;
        int64_t l = (int64_t)blockIdx.x * kThreads + threadIdx.x;
        for (int k = 0; k < 2 && l < lines; ++k, l += nthr) {
            const int64_t r = l / lines_per_row;
            prefetch_l2(a.bt + r * a.bt_stride + (l - r * lines_per_row) * 32);
        }
    }
    const uint4 z = make_uint4(0, 0, 0, 0);
    uint4 *v = reinterpret_cast<uint4 *>(smem + C::kOffV);
    for (int i = threadIdx.x; i < C::kVStages * C::kVSlot / 16; i += kThreads) v[i] = z;
#pragma unroll
    for (int i = 0; i < kLensPerThread; ++i) {
        const int r = threadIdx.x + i * kThreads;
        if (r < n) {
            if (lens[i] > a.max_ctx && blockIdx.x == 0 && a.err) atomicAdd(a.err, 1);
            const int32_t Lg = lens[i] > a.max_ctx ? a.max_ctx : (lens[i] < 0 ? 0 : lens[i]);
            // the keys this rank holds (all of them without context parallelism); a
            // sliding window (never combined with it) drops the tiles wholly before
            // its first visible key
            const int32_t L = cp_local_len(a, Lg);
            pre[r] = sk_tiles(a, lens[i]);
            lrem[r] = (uint8_t)((L - 1) & (kTile - 1));
        }
    }
}

// Exclusive prefix sum of the tile counts in place, pre[n] = total, over all
// threads of the CTA (tot: one int per warp plus one of scratch).  Starts and
// ends with a __syncthreads.
template <int kThreads>
__device__ void scan_prefix(const DecodeArgs &a, int32_t *pre, int32_t *tot) {
    constexpr int kWarps = kThreads / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = a.num_reqs;
    __syncthreads();
    const int per = (n + kThreads - 1) / kThreads;
    const int lo = min(n, (int)threadIdx.x * per), hi = min(n, lo + per);
    int32_t sum = 0;
    for (int r = lo; r < hi; ++r) sum += pre[r];
    int32_t inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t x = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += x;
    }
    if (lane == 31) tot[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int32_t w = lane < kWarps ? tot[lane] : 0;
        int32_t wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t x = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += x;
        }
        __syncwarp();
        if (lane < kWarps) tot[lane] = wi - w;
        if (lane == kWarps - 1) tot[kWarps] = wi;
    }
    __syncthreads();
    int32_t run = tot[warp] + inc - sum;
    for (int r = lo; r < hi; ++r) {
        const int32_t t = pre[r];
        pre[r] = run;
        run += t;
    }
    if (threadIdx.x == 0) pre[n] = tot[kWarps];
    __syncthreads();
}

// One unit: tiles [lo, hi) of stream s = r * H_kv + g, counted from the
// stream's first tile f (0, or the tile holding the sliding window's first
// visible key): positions [start, cend) with start = (f + lo) * 128, cend =
// min((f + hi) * 128, L).  Its partials go to slots slot2 and slot2 + 1.
struct Unit {
    int r, g;
    int64_t s, slot2;
    int32_t L, start, cend, ntiles;
};

// Walks this CTA's units in order.  The grid is P groups of H_kv CTAs; the
// requests' position tiles (pre[r] .. pre[r + 1] for request r) are laid end
// to end and group q takes [q TP / Peff, (q + 1) TP / Peff) of them (TP
// tiles in all, Peff = min(P, TP)), CTA g of the group for KV head g.  The
// H_kv CTAs of a group thus read the same positions of all heads at the
// same time, i.e. whole cache rows (one row holds every head of a
// position).  Unit (group q, request r, head g) writes slots
// 2 (g (P + R) + q + r) + {0, 1}: q + r grows by at least one from one unit
// of a head to the next, so the slots are distinct, and a stream's slots
// are the contiguous range the merge recomputes from the context lengths.
struct StreamK {
    const int32_t *pre;
    const uint8_t *lrem;
    int n, H, q, g;
    int64_t t, t1;   // next position tile, end of this CTA's range
    int64_t hbase;   // g (P + R): this head's slot block
    int r;
    __device__ void init(const DecodeArgs &a, const int32_t *pre_, const uint8_t *lrem_) {
        pre = pre_;
        lrem = lrem_;
        n = a.num_reqs;
        H = a.H_kv;
        const int P = (int)gridDim.x / H;
        q = (int)blockIdx.x / H;
        g = (int)blockIdx.x - q * H;
        hbase = (int64_t)g * (P + n);
        // split over min(P, TP) groups so every participating CTA has at
        // least one tile (the merge recomputes the slots with the same rule);
        // floor(TP q / peff) in 32-bit operations: TP = A peff + B gives
        // A q + floor(B q / peff), and B q < peff^2 is small
        const int32_t TP = pre[n];
        const int32_t peff = TP < P ? TP : P;
        if (q < peff) {
            const int32_t A = TP / peff, B = TP - A * peff;
            t = (int64_t)A * q + (B * q) / peff;
            t1 = (int64_t)A * (q + 1) + (B * (q + 1)) / peff;
        } else {
            t = t1 = TP;
        }
        // first request whose tiles end after t
        int lo = 0, hi = n;   // invariant: answer in [lo, hi]
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if ((int64_t)pre[mid + 1] > t) hi = mid;
            else lo = mid + 1;
        }
        r = lo;
    }
    __device__ bool next(const DecodeArgs &a, Unit &x) {
        if (t >= t1) return false;
        while (r < n && (int64_t)pre[r + 1] <= t) ++r;
        const int64_t S = pre[r];
        const int64_t Tr = pre[r + 1] - S;
        const int64_t lo = t - S;
        const int64_t hi = (t1 - S) < Tr ? (t1 - S) : Tr;
        x.r = r;
        x.g = g;
        x.s = (int64_t)r * H + g;
        x.slot2 = 2 * (hbase + q + r);
        int64_t f = 0;
        if (a.window > 0) {
            // the tile count no longer gives the length: read it (clamped) again
            const int32_t Lg = __ldg(a.ctx + r);
            x.L = Lg > a.max_ctx ? a.max_ctx : Lg;
            f = window_lo(a, x.L) / kTile;
        } else {
            x.L = (int32_t)(Tr - 1) * kTile + lrem[r] + 1;   // Tr > 0: the stream has this tile
        }
        x.start = (int32_t)((f + lo) * kTile);
        x.cend = (int32_t)((f + hi) * kTile < (int64_t)x.L ? (f + hi) * kTile : (int64_t)x.L);
        x.ntiles = (int32_t)(hi - lo);
        t = S + hi;
        return true;
    }
};

// Transposed butterfly over a warp: NQ values per lane in, one value out.
// Each halving step exchanges half of the remaining values with the partner
// lane, so after log2(NQ) steps lane l holds query row (l >> (5 - log2 NQ)) &
// (NQ - 1), reduced over the lanes that differ in the high bits; the last
// steps reduce over the low lane bits.  NQ + 5 - log2(NQ) - ... shuffles in
// all (16 for NQ = 16, 6 for NQ = 4).
template <bool kMax, int NQ>
__device__ __forceinline__ float warp_reduce_rows(const float (&v)[NQ], int lane) {
    auto op = [](float x, float y) { return kMax ? fmaxf(x, y) : x + y; };
    float cur[NQ];
#pragma unroll
    for (int i = 0; i < NQ; ++i) cur[i] = v[i];
    int width = NQ;
    int shift = 16;
#pragma unroll
    for (int step = 0; step < 4; ++step) {
        if (width > 1) {
            const bool hi = lane & shift;
            const int h = width / 2;
#pragma unroll
            for (int i = 0; i < NQ / 2; ++i) {
                if (i < h) {
                    const float send = hi ? cur[i] : cur[i + h];
                    const float keep = hi ? cur[i + h] : cur[i];
                    cur[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, shift));
                }
            }
            width = h;
            shift >>= 1;
        }
    }
    float x = cur[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        if (o <= shift) x = op(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

template <int NQ>
__device__ __forceinline__ int reduced_row(int lane) {
    constexpr int k = NQ == 16 ? 4 : (NQ == 8 ? 3 : 2);
    return (lane >> (5 - k)) & (NQ - 1);
}

template <int NQ>
__device__ __forceinline__ bool reduced_writer(int lane) {
    constexpr int k = NQ == 16 ? 4 : (NQ == 8 ? 3 : 2);
    return (lane & ((1 << (5 - k)) - 1)) == 0;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int NQ, bool kCP, bool kF8>
__global__ void __launch_bounds__(Cfg<kF8>::kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ CUtensorMap tmQ, const DecodeArgs a, int seg_rows) {
    using C = Cfg<kF8>;
    constexpr int kThreads = C::kThreads;
    constexpr int kKStages = C::kKStages;
    constexpr int kVStages = C::kVStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint32_t *mask_words = reinterpret_cast<uint32_t *>(smem + C::kOffMask);
    float *red_max = reinterpret_cast<float *>(smem + C::kOffRedMax);
    float *red_sum = reinterpret_cast<float *>(smem + C::kOffRedSum);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::kOffTmemSlot);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::kOffAbort);
    int32_t *pre = reinterpret_cast<int32_t *>(smem + C::kOffPre);
    const uint32_t bar0 = sbase + C::kOffBar;
    // K and V tiles have separate rings (same slot numbering): a K slot is
    // released as soon as the S MMA that reads it completes.
    constexpr int kB = 2 * kKStages + 2 * kVStages;   // first barrier after the rings
    auto bar_kfull = [&](int s) { return bar0 + 8u * s; };
    auto bar_kempty = [&](int s) { return bar0 + 8u * (kKStages + s); };
    auto bar_vfull = [&](int s) { return bar0 + 8u * (2 * kKStages + s); };
    auto bar_vempty = [&](int s) { return bar0 + 8u * (2 * kKStages + kVStages + s); };
    auto bar_qfull = [&](int b) { return bar0 + 8u * (kB + b); };
    auto bar_qempty = [&](int b) { return bar0 + 8u * (kB + 2 + b); };
    auto bar_sfull = [&](int b) { return bar0 + 8u * (kB + 4 + b); };
    auto bar_pfull = [&](int b) { return bar0 + 8u * (kB + 6 + b); };
    auto bar_ofull = [&](int b) { return bar0 + 8u * (kB + 8 + b); };
    auto bar_group = [&](int k) { return bar0 + 8u * (kB + 10 + k); };   // four warps of warpgroup k
    // "loaded segments" word of tile j: mask_words[j % kMaskRing], published with bar_mask(j % kMaskRing)
    auto bar_mask = [&](int m) { return bar0 + 8u * (kB + 12 + m); };
    // S tile b read into registers (four softmax warps): the S issuer may overwrite it
    auto bar_sfree = [&](int b) { return bar0 + 8u * (kB + 12 + kMaskRing + b); };
    const uint32_t sm_k = sbase + C::kOffK;
    const uint32_t sm_v = sbase + C::kOffV;
    const uint32_t sm_q = sbase + C::kOffQ;
    const uint32_t sm_p = sbase + C::kOffP;

    // ---- set-up (no global memory): barriers, zeroed Q / P buffers, TMEM ----
    if (threadIdx.x == 0) {
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(bar_kfull(s), 1);
            mbar_init(bar_kempty(s), 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(bar_vfull(s), 1);
            mbar_init(bar_vempty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_qfull(b), 1);
            mbar_init(bar_qempty(b), 1);
            mbar_init(bar_sfull(b), 1);
            mbar_init(bar_pfull(b), 4);
            mbar_init(bar_ofull(b), 1);
        }
        mbar_init(bar_group(0), 4);
        mbar_init(bar_group(1), 4);
        mbar_init(bar_sfree(0), 4);
        mbar_init(bar_sfree(1), 4);
        for (int m = 0; m < kMaskRing; ++m) mbar_init(bar_mask(m), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmQ);
    }
    {
        // Q rows past the group and P start at zero
        const uint4 z = make_uint4(0, 0, 0, 0);
        uint4 *qp = reinterpret_cast<uint4 *>(smem + C::kOffQ);
        for (int i = threadIdx.x; i < (2 * kQBytes + 2 * kPBytes) / 16; i += kThreads) qp[i] = z;
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
    // Global memory is read from here on.  bf16: the preceding kernel may be
    // the caller's and may have written anything read below, so wait for it.
    // E4M3: the preceding kernel is this call's query split
    // (q_split_e4m3_kernel), which waited for its own predecessors before
    // letting this grid start, so only its outputs (the split queries and
    // their scales) wait: the K producer before the first Q load, the softmax
    // before the first scale read; the schedule, the table and the first K and
    // V loads overlap the split.
    if constexpr (!kF8) pdl_wait();
    pdl_trigger();
    uint8_t *lrem = smem + C::kOffLrem;
    schedule_loads<kF8>(a, pre, lrem, smem);
    fence_proxy_async();       // the zeroed V ring before any TMA write to it
    // red_max is free until the softmax starts: scratch for the scan
    scan_prefix<kThreads>(a, pre, reinterpret_cast<int32_t *>(red_max));
    const uint32_t tmem = *tmem_slot;

    const int G = a.G;
    const int nq = a.nq;
    const int nseg = kTile / seg_rows;              // block segments per tile (1..16)
    const int seg_shift = 31 - __clz(seg_rows);     // seg_rows is a power of two

    if (warp == 0 || warp == kWarpV) {
        // ================= TMA producers (warp 0: K and Q, last warp: V) =================
        // Units are walked in windows of at most kWinBlocks table entries; a
        // window's entries are loaded into registers while the previous
        // window's tiles are issued, then parked in shared memory, so no
        // table lookup sits between a slot becoming free and its refill.  An
        // entry past the table width is parked as INT32_MIN.
        const bool is_v = warp == kWarpV;
        int32_t *ent_buf = reinterpret_cast<int32_t *>(smem + C::kOffEnt) + (is_v ? 2 * kWinBlocks : 0);
        const int win_tiles = max(1, ((kWinBlocks - 1) * a.bs) / kTile);
        struct Win {
            Unit u;
            int32_t t0, t1;   // tiles of the unit
        };
        StreamK sk;
        sk.init(a, pre, lrem);
        Unit cu = {};
        bool have_u = false;
        int32_t wt = 0;
        auto next_win = [&](Win &w) -> bool {
            if (!have_u || wt >= cu.ntiles) {
                if (!sk.next(a, cu)) return false;
                have_u = true;
                wt = 0;
            }
            w.u = cu;
            w.t0 = wt;
            w.t1 = min(cu.ntiles, wt + win_tiles);
            wt = w.t1;
            return true;
        };
        auto win_first_block = [&](const Win &w) { return (w.u.start + w.t0 * kTile) / a.bs; };
        auto win_blocks = [&](const Win &w) {
            const int32_t p1 = min(w.u.start + w.t1 * kTile, w.u.cend);
            return (p1 - 1) / a.bs - win_first_block(w) + 1;
        };
        constexpr int kEntRegs = kWinBlocks / 32;
        int32_t ent_reg[kEntRegs];
        auto fetch_entries = [&](const Win &w) {
            const int32_t lb0 = win_first_block(w);
            const int32_t nblk = win_blocks(w);
#pragma unroll
            for (int kk = 0; kk < kEntRegs; ++kk) {
                const int32_t lbl = kk * 32 + lane;
                if (lbl < nblk) {
                    const int32_t lb = lb0 + lbl;
                    ent_reg[kk] = lb < a.bt_cols ? __ldg(a.bt + (int64_t)w.u.r * a.bt_stride + lb) : INT32_MIN;
                }
            }
        };
        auto park_entries = [&](const Win &w, int buf) {
            const int32_t nblk = win_blocks(w);
#pragma unroll
            for (int kk = 0; kk < kEntRegs; ++kk) {
                const int32_t lbl = kk * 32 + lane;
                if (lbl < nblk) ent_buf[buf * kWinBlocks + lbl] = ent_reg[kk];
            }
            __syncwarp();
        };
        int64_t j = 0;   // tile sequence number in this CTA
        int us = 0;      // unit sequence number in this CTA
        int ws = 0;      // window sequence number
        const int nst = is_v ? kVStages : kKStages;
        Ring ring;       // slot of tile j in this producer's ring
        Win cur, nxt;
        bool have = next_win(cur);
        if (have) {
            fetch_entries(cur);
            park_entries(cur, 0);
        }
        while (have && !*abort_flag) {
            const bool have_n = next_win(nxt);
            if (have_n) fetch_entries(nxt);   // in flight while this window's tiles are issued
            const int32_t *ents = ent_buf + (ws & 1) * kWinBlocks;
            const int32_t lb_first = win_first_block(cur);
            const Unit &x = cur.u;
            const int32_t wlo = window_lo(a, x.L);   // segments ending at or before it are not needed
            // the unit's Q (K producer), once its buffer is free; the first unit's E4M3
            // queries go after its first K tile, behind the wait for the query split
            auto issue_q = [&]() {
                const int qb = us & 1;
                if (lane == 0) {
                    if (kF8 && us == 0) pdl_wait();   // the split queries are the query split's output
                    mbar_arrive_expect_tx(bar_qfull(qb), 2u * 128u * (uint32_t)nq);
                    const uint32_t dq = sm_q + qb * kQBytes;
                    if constexpr (kF8) {
                        // the two E4M3 parts of the rows, 128 codes each: part p of token row
                        // t is row p * num_reqs * q_len + t of the split map
                        const int rows = a.num_reqs * a.q_len;
                        tma_load_3d(dq, &tmQ, bar_qfull(qb), 0, x.g * G, x.r * a.q_len);
                        tma_load_3d(dq + kN * 128, &tmQ, bar_qfull(qb), 0, x.g * G, rows + x.r * a.q_len);
                    } else {
                        tma_load_3d(dq, &tmQ, bar_qfull(qb), 0, x.g * G, x.r * a.q_len);
                        tma_load_3d(dq + kN * 128, &tmQ, bar_qfull(qb), 64, x.g * G, x.r * a.q_len);
                    }
                }
                __syncwarp();
            };
            bool q_after_first = false;
            if (cur.t0 == 0 && !is_v) {
                if (!mbar_wait_warp(bar_qempty(us & 1), ((us >> 1) & 1) ^ 1, abort_flag)) break;
                if (kF8 && us == 0) q_after_first = true;
                else issue_q();
            }
            for (int jt = cur.t0; jt < cur.t1; ++jt, ++j, ring.advance(nst)) {
                const int s = ring.slot;
                const uint32_t bar_e = is_v ? bar_vempty(s) : bar_kempty(s);
                const uint32_t bar_f = is_v ? bar_vfull(s) : bar_kfull(s);
                if (!mbar_wait_warp(bar_e, ring.phase ^ 1u, abort_flag)) break;
                const int32_t ts = x.start + jt * kTile;
                // lane i handles block segment i of the tile
                bool load = false;
                int64_t row0 = 0;
                if (lane < nseg) {
                    const int32_t p0 = ts + lane * seg_rows;
                    if (p0 < x.cend && p0 + seg_rows > wlo) {
                        const int32_t lb = p0 / a.bs;
                        const int64_t e = ents[lb - lb_first];
                        if (e == INT32_MIN || e >= a.total_blocks) {
                            // a bad entry counts once per stream, at the first segment of
                            // its block that is read: the block's first segment, or the
                            // one holding the window's first key
                            if (!is_v && a.err && (p0 - lb * a.bs < seg_rows || p0 <= wlo)) atomicAdd(a.err, 1);
                        } else if (e > 0) {
                            load = true;
                            row0 = e * a.bs + (p0 - (int64_t)lb * a.bs);
                        }
                    }
                }
                const uint32_t ballot = __ballot_sync(0xffffffffu, load);
                if (lane == 0) {
                    // bit i: segment i was loaded.  A ring of kMaskRing words by tile number
                    // with its own barriers: the K producer writes tile j's word only after
                    // the S MMA of tile j - kKStages completed, which is issued only after
                    // the softmax read S (and, before that, the word) of tile
                    // j - kKStages - 2, so the writer is at most kKStages + 2 < kMaskRing
                    // tiles ahead of the reader and neither words nor barrier phases alias.
                    if (!is_v) {
                        mask_words[j & (kMaskRing - 1)] = ballot;
                        mbar_arrive(bar_mask((int)(j & (kMaskRing - 1))));
                    }
                    const uint32_t bytes = (uint32_t)__popc(ballot) * (uint32_t)seg_rows * 128u * (kF8 ? 1u : 2u);
                    mbar_arrive_expect_tx(bar_f, bytes);
                }
                __syncwarp();
                if (load) {
                    const CUtensorMap *map = is_v ? &tmV : &tmK;
                    const int z = (int)row0;
                    if constexpr (kF8) {
                        // one box of seg_rows rows x 128 codes (the whole head_dim)
                        const uint32_t dst = (is_v ? sm_v : sm_k) + s * kT8Bytes + lane * seg_rows * 128;
                        tma_load_3d(dst, map, bar_f, 0, x.g, z);
                    } else {
                        const uint32_t dst = (is_v ? sm_v : sm_k) + s * kTileBytes + lane * seg_rows * 128;
                        tma_load_3d(dst, map, bar_f, 0, x.g, z);
                        tma_load_3d(dst + kHalfBytes, map, bar_f, 64, x.g, z);
                    }
                }
                __syncwarp();
                if (q_after_first) {
                    issue_q();
                    q_after_first = false;
                }
            }
            if (q_after_first) issue_q();   // (a window without tiles: never, kept for safety)
            if (have_n) park_entries(nxt, (ws + 1) & 1);
            if (cur.t1 == x.ntiles) ++us;
            ++ws;
            cur = nxt;
            have = have_n;
        }
        if (*abort_flag) {
            // let copies already issued land before the CTA retires
            const unsigned long long t0 = global_ns();
            while (global_ns() - t0 < 200000ull) {
            }
        }
    } else if (warp == 1 || warp == kWarpPV) {
        // ================= MMA issuers (one thread each) =================
        // Warp 1 issues the S MMAs, warp kWarpPV the P.V MMAs, so neither waits on
        // the other's operands.  K (K-major) x Q (K-major); V^T (MN-major) x P
        // (K-major).  FP8 caches: both on E4M3 operands (the descriptor's E4M3
        // type codes are 0, as f16's), with the hi and lo parts of Q (resp. P)
        // stacked as 32 B rows, so one MMA of N = 32 multiplies both.
        constexpr int kNM = kF8 ? 2 * kN : kN;
        bool ok = true;
        StreamK sk;
        sk.init(a, pre, lrem);
        if (lane == 0 && warp == 1) {
            constexpr uint32_t kIdescS = kF8 ? idesc_f16(128, kNM, 0, 0) : idesc_bf16(128, kNM, 0, 0);
            int64_t j = 0;
            int us = 0;
            Ring kr;
            Unit x;
            while (ok && sk.next(a, x)) {
                const int qb = us & 1;
                if (!mbar_wait(bar_qfull(qb), (uint32_t)((us >> 1) & 1), abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t q_base = sm_q + qb * kQBytes;
                for (int jt = 0; jt < x.ntiles; ++jt, ++j, kr.advance(kKStages)) {
                    const int b = (int)(j & 1);
                    // K landed, and the softmax has read S tile b of tile j - 2
                    if (!mbar_wait(bar_kfull(kr.slot), kr.phase, abort_flag) ||
                        (j >= 2 && !mbar_wait(bar_sfree(b), (uint32_t)((j >> 1) & 1) ^ 1u, abort_flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + 32u * (uint32_t)b;
                    if constexpr (kF8) {
                        // S^T[:, 0:16] = K . Q_hi^T, S^T[:, 16:32] = K . Q_lo^T (E4M3, 128-code
                        // rows): four 32-code steps
                        const uint32_t k_base = sm_k + kr.slot * kT8Bytes;
#pragma unroll
                        for (int kk = 0; kk < kD / 32; ++kk) {
                            const uint64_t adesc = sdesc(k_base + kk * 32, 16, 1024);
                            const uint64_t bdesc = sdesc(q_base + kk * 32, 16, 1024);
                            mma_f8(d_tmem, adesc, bdesc, kIdescS, kk > 0);
                        }
                    } else {
                        const uint32_t k_base = sm_k + kr.slot * kTileBytes;
#pragma unroll
                        for (int kk = 0; kk < kD / 16; ++kk) {
                            const uint32_t half = (uint32_t)(kk >> 2) * kHalfBytes;
                            const uint64_t adesc = sdesc(k_base + half + (kk & 3) * 32, 16, 1024);
                            const uint64_t bdesc = sdesc(q_base + (kk >> 2) * (kN * 128) + (kk & 3) * 32, 16, 1024);
                            mma_bf16(d_tmem, adesc, bdesc, kIdescS, kk > 0);
                        }
                    }
                    mma_commit(bar_sfull(b));
                    mma_commit(bar_kempty(kr.slot));
                    if (jt == x.ntiles - 1) mma_commit(bar_qempty(qb));
                }
                ++us;
            }
        } else if (lane == 0) {
            constexpr uint32_t kIdescO = kF8 ? idesc_f16(128, kNM, 1, 0) : idesc_bf16(128, kNM, 1, 0);
            // the P.V MMAs do not depend on unit boundaries: this CTA's tiles in order
            const int64_t ntot = sk.t1 - sk.t;
            Ring vr;
            for (int64_t j = 0; j < ntot; ++j, vr.advance(kVStages)) {
                const int b = (int)(j & 1);
                if (!mbar_wait(bar_vfull(vr.slot), vr.phase, abort_flag) ||
                    !mbar_wait(bar_pfull(b), (uint32_t)((j >> 1) & 1), abort_flag))
                    break;
                tc_fence_after();
                const uint32_t p_base = sm_p + b * kPBytes;
                const uint32_t d_tmem = tmem + 64u + 32u * (uint32_t)b;
                if constexpr (kF8) {
                    // O^T[:, 0:16] = V^T . P_hi^T, O^T[:, 16:32] = V^T . P_lo^T; V^T as E4M3
                    // codes MN-major (a row's 128 codes are one 128-byte span, 8-row groups
                    // 1024 bytes apart), 32 positions per step
                    const uint32_t v_base = sm_v + vr.slot * kT8Bytes;
#pragma unroll
                    for (int kk = 0; kk < kTile / 32; ++kk) {
                        const uint64_t adesc = sdesc(v_base + kk * 4096, 16, 1024);
                        const uint64_t bdesc = sdesc(p_base + kk * 32, 16, 1024);
                        mma_f8(d_tmem, adesc, bdesc, kIdescO, kk > 0);
                    }
                } else {
                    const uint32_t v_base = sm_v + vr.slot * kTileBytes;
#pragma unroll
                    for (int kk = 0; kk < kTile / 16; ++kk) {
                        const uint64_t adesc = sdesc(v_base + kk * 2048, kHalfBytes, 1024);
                        const uint64_t bdesc = sdesc(p_base + (kk >> 2) * (kN * 128) + (kk & 3) * 32, 16, 1024);
                        mma_bf16(d_tmem, adesc, bdesc, kIdescO, kk > 0);
                    }
                }
                mma_commit(bar_ofull(b));
                mma_commit(bar_vempty(vr.slot));
            }
        }
        __syncwarp();
    } else if (warp < kWarpV) {
        // ================= softmax + output (two warpgroups of 128 threads) =================
        // Warpgroup k takes the tiles with (tile sequence number & 1) == k,
        // i.e. the S / P / O buffers of parity k, and writes partial slot
        // slot2 + k of every unit.
        const int wg = (warp - 2) >> 2;
        // FP8 caches: query row i entered the S MMA divided by qexp[i] (a power of two),
        // taken back per column below; the weights enter the P.V MMA and the row sums
        // as p 2^kF8PExp, taken back at the partial output
        const float s_scale = a.scale_log2;
        constexpr float kOutScale = kF8 ? 1.f / (float)(1 << kF8PExp) : 1.f;
        const int row = 32 * (warp & 3) + lane;          // TMEM lane: position in tile / head_dim row
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const int wq = warp & 3;
        float o[NQ], lsum[NQ], mrun[NQ];
        int64_t j = 0;
        Ring vring;      // V slot of tile j (rows past the end are zeroed there)
        bool ok = true;
        uint32_t gphase = 0;
        // Bounded barrier of the warpgroup's four warps (an mbarrier, so that a
        // timed-out wait elsewhere can never leave a warp stuck here).
        auto group_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_group(wg));
            const bool r = mbar_wait_warp(bar_group(wg), gphase, abort_flag);
            gphase ^= 1u;
            return r;
        };
        // This thread's byte offset in the P^T operand (K-major, 128-byte
        // swizzle): position `row`, query row n adds n * 128 and swizzles the
        // 16-byte chunk index with n & 7.  bf16: positions 64 h .. 64 h + 63
        // form block h of 16 rows x 128 bytes; E4M3: one block of 128
        // positions per part (hi, then lo).
        const int p_row_off = kF8 ? (row & 15) : (row >> 6) * (kN * 128) + (row & 7) * 2;
        const int p_chunk = kF8 ? (row >> 4) : (row & 63) >> 3;
        const int red_row = reduced_row<NQ>(lane);
        const bool red_writer = reduced_writer<NQ>(lane);
        float *my_red_sum = red_sum + wg * (kN * 4);
        StreamK sk;
        sk.init(a, pre, lrem);
        if constexpr (kF8) pdl_wait();   // the query scales are the query split's output
        Unit x;
        while (ok && sk.next(a, x)) {
            // masks are in global positions: with context parallelism x.L counts
            // only this rank's keys, so the request's length is read again
            int32_t Lg = x.L;
            if (kCP) {
                const int32_t c = __ldg(a.ctx + x.r);
                Lg = c > a.max_ctx ? a.max_ctx : c;
            }
            int32_t lastv[NQ], firstv[NQ];
            float cs[NQ];   // score scale of each query column
#pragma unroll
            for (int n = 0; n < NQ; ++n) {
                o[n] = 0.f;
                lsum[n] = 0.f;
                mrun[n] = -INFINITY;
                const int t = n / G;
                cs[n] = s_scale;
                if (kF8 && n < nq)
                    cs[n] = s_scale * __ldg(a.qexp + ((int64_t)x.r * a.q_len + t) * a.H_q + x.g * G + (n - t * G));
                lastv[n] = (n < nq) ? (a.mask_mode == 0 ? Lg - a.q_len + t : Lg - 1) : -1;
                firstv[n] = a.window > 0 ? Lg - a.q_len + t - a.window + 1 : INT32_MIN;
            }
            for (int jt = 0; jt < x.ntiles; ++jt, ++j, vring.advance(kVStages)) {
                if ((int)(j & 1) != wg) continue;
                const int sv_slot = vring.slot;
                const int b = wg;
                const uint32_t par = (uint32_t)((j >> 1) & 1);
                if (!mbar_wait_warp(bar_sfull(b), par, abort_flag) ||
                    !mbar_wait_warp(bar_mask((int)(j & (kMaskRing - 1))), (uint32_t)((j / kMaskRing) & 1), abort_flag)) {
                    ok = false;
                    break;
                }
                // the loaded-segment word is read before S tile b is released: the K
                // producer can rewrite this word (for tile j + kMaskRing) only after the
                // S MMA of tile j + 2 completed, which waits for that release
                const bool loaded = (mask_words[j & (kMaskRing - 1)] >> (row >> seg_shift)) & 1u;
                tc_fence_after();
                float sv[NQ];
                if constexpr (kF8) tmem_ld_sum2<NQ>(tmem + lane_base + 32u * b, sv);
                else tmem_ld_cols<NQ>(tmem + lane_base + 32u * b, sv);
                // S tile b may now be overwritten (by the S MMA of tile j + 2)
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_sfree(b));
                const int32_t pos = x.start + jt * kTile + row;
                const bool inrange = loaded && pos < x.cend;
                const int32_t gpos = kCP ? cp_global32(a, pos) : pos;
#pragma unroll
                for (int n = 0; n < NQ; ++n)
                    sv[n] = (inrange && gpos <= lastv[n] && gpos >= firstv[n]) ? sv[n] * cs[n] : -INFINITY;
                // tile max per query row across the warpgroup's 128 threads
                const float wmax = warp_reduce_rows<true, NQ>(sv, lane);
                float *rm = red_max + (wg * 2 + (int)par) * (kN * 4);
                if (red_writer) rm[red_row * 4 + wq] = wmax;
                if (!group_sync()) {
                    ok = false;
                    break;
                }
                float corr[NQ];
                uint8_t *pgen = smem + C::kOffP + b * kPBytes + p_row_off;
                // new running max, rescale factor and weight of each query row, then
                // P as the MMA's operand type; the row sums take the rounded weights
                auto weight = [&](int n) -> float {
                    const float4 t4 = *reinterpret_cast<const float4 *>(rm + n * 4);
                    const float mt = fmaxf(fmaxf(t4.x, t4.y), fmaxf(t4.z, t4.w));
                    const float mn = fmaxf(mrun[n], mt);
                    corr[n] = (mn == -INFINITY) ? 1.f : fast_exp2(mrun[n] - mn);
                    mrun[n] = mn;
                    return (sv[n] == -INFINITY) ? 0.f : fast_exp2(sv[n] - mn);
                };
                if constexpr (kF8) {
                    // p 2^8 = hi + lo, two E4M3 codes per weight, two query rows per
                    // conversion: hi is p 2^8 to 4 significant bits, lo the remainder to
                    // 4 more (absolute error at most 2^-10 in p 2^8)
#pragma unroll
                    for (int n = 0; n < NQ; n += 2) {
                        const float p0 = weight(n), p1 = weight(n + 1);
                        const float2 x2 = make_float2(p0 * (float)(1 << kF8PExp), p1 * (float)(1 << kF8PExp));
                        const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(x2, __NV_SATFINITE, __NV_E4M3);
                        const float2 hf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(hi, __NV_E4M3)));
                        const __nv_fp8x2_storage_t lo =
                            __nv_cvt_float2_to_fp8x2(make_float2(x2.x - hf.x, x2.y - hf.y), __NV_SATFINITE, __NV_E4M3);
                        const float2 lf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(lo, __NV_E4M3)));
                        lsum[n] = fmaf(lsum[n], corr[n], hf.x + lf.x);
                        lsum[n + 1] = fmaf(lsum[n + 1], corr[n + 1], hf.y + lf.y);
                        uint8_t *d0 = pgen + n * 128 + ((p_chunk ^ (n & 7)) << 4);
                        uint8_t *d1 = pgen + (n + 1) * 128 + ((p_chunk ^ ((n + 1) & 7)) << 4);
                        d0[0] = (uint8_t)(hi & 0xFF);
                        d1[0] = (uint8_t)(hi >> 8);
                        d0[kN * 128] = (uint8_t)(lo & 0xFF);
                        d1[kN * 128] = (uint8_t)(lo >> 8);
                    }
                } else {
#pragma unroll
                    for (int n = 0; n < NQ; ++n) {
                        const __nv_bfloat16 pbv = __float2bfloat16_rn(weight(n));
                        lsum[n] = fmaf(lsum[n], corr[n], __bfloat162float(pbv));
                        *reinterpret_cast<__nv_bfloat16 *>(pgen + n * 128 + ((p_chunk ^ (n & 7)) << 4)) = pbv;
                    }
                }
                // V rows that were loaded but lie past the end must be zero for P.V
                // (after the V tile has landed)
                const bool zero_row = loaded && pos >= x.cend;
                if (__any_sync(0xffffffffu, zero_row) && !mbar_wait_warp(bar_vfull(sv_slot), vring.phase, abort_flag)) {
                    ok = false;
                    break;
                }
                if (zero_row) {
                    uint4 *vrow = reinterpret_cast<uint4 *>(smem + C::kOffV + sv_slot * C::kVSlot + row * 128);
#pragma unroll
                    for (int c = 0; c < 8; ++c) vrow[c] = make_uint4(0, 0, 0, 0);
                    if constexpr (!kF8) {
                        vrow = reinterpret_cast<uint4 *>(smem + C::kOffV + sv_slot * kTileBytes + kHalfBytes + row * 128);
#pragma unroll
                        for (int c = 0; c < 8; ++c) vrow[c] = make_uint4(0, 0, 0, 0);
                    }
                }
                fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_pfull(b));
                // this tile's P.V (the other warpgroup works meanwhile)
                if (!mbar_wait_warp(bar_ofull(b), par, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float ot[NQ];
                if constexpr (kF8) tmem_ld_sum2<NQ>(tmem + lane_base + 64u + 32u * b, ot);
                else tmem_ld_cols<NQ>(tmem + lane_base + 64u + 32u * b, ot);
#pragma unroll
                for (int n = 0; n < NQ; ++n) o[n] = fmaf(o[n], corr[n], ot[n]);
            }
            if (!ok) break;
            // row sums across the warpgroup, then this warpgroup's partial (o, m, l)
            {
                const float wsum = warp_reduce_rows<false, NQ>(lsum, lane);
                if (red_writer) my_red_sum[red_row * 4 + wq] = wsum;
                if (!group_sync()) {
                    ok = false;
                    break;
                }
                const int64_t prow0 = (x.slot2 + wg) * nq;
#pragma unroll
                for (int n = 0; n < NQ; ++n)
                    if (n < nq) a.ws_o[(prow0 + n) * kD + row] = o[n] * kOutScale;
                if (row < nq) {
                    const float4 t4 = *reinterpret_cast<const float4 *>(my_red_sum + row * 4);
                    float m_row = -INFINITY;
#pragma unroll
                    for (int n = 0; n < NQ; ++n)
                        if (n == row) m_row = mrun[n];
                    a.ws_ml[(prow0 + row) * 2 + 0] = m_row;
                    a.ws_ml[(prow0 + row) * 2 + 1] = ((t4.x + t4.y) + (t4.z + t4.w)) * kOutScale;
                }
                if (!group_sync()) {   // the row-sum buffer is reused by the next unit
                    ok = false;
                    break;
                }
            }
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
// FP8 caches: the queries as two E4M3 parts for the S MMA
// ---------------------------------------------------------------------------
// Row i of q (one query token and head, 128 bf16 values) with absolute maximum
// m is scaled by 2^-e, e = floor(log2 m) - 7, so that its largest element
// lies in [128, 256); each scaled element x is written as hi = E4M3(x) (round
// to nearest) and lo = E4M3(x - hi).  x has at most 8 significant bits, so
// x - hi is a multiple of ulp(x) / 128 of at most 8 of them: hi + lo = x
// exactly when |x| >= 2^-2 (the step of E4M3 subnormals is 2^-9), and
// otherwise within 2^-10, i.e. 2^-17 of the row's largest element.
// qexp[i] = 2^e restores the scale of the row's scores.  One warp per row.
__global__ void __launch_bounds__(256) q_split_e4m3_kernel(const __nv_bfloat16 *__restrict__ q, int64_t rows,
                                                           uint8_t *__restrict__ q8, float *__restrict__ qexp) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const uint2 raw = *reinterpret_cast<const uint2 *>(q + row * kD + 4 * lane);
    const float2 x01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.x));
    const float2 x23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.y));
    const float x[4] = {x01.x, x01.y, x23.x, x23.y};
    float m = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int e = (m > 0.f && m <= 3.402823466e38f) ? ilogbf(m) - 7 : 0;
    uint32_t hi = 0, lo = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float xs = ldexpf(x[i], -e);
        const __nv_fp8_storage_t h = __nv_cvt_float_to_fp8(xs, __NV_SATFINITE, __NV_E4M3);
        const float hf = __half2float(__half(__nv_cvt_fp8_to_halfraw(h, __NV_E4M3)));
        const __nv_fp8_storage_t l = __nv_cvt_float_to_fp8(xs - hf, __NV_SATFINITE, __NV_E4M3);
        hi |= (uint32_t)h << (8 * i);
        lo |= (uint32_t)l << (8 * i);
    }
    *reinterpret_cast<uint32_t *>(q8 + row * kD + 4 * lane) = hi;
    *reinterpret_cast<uint32_t *>(q8 + (rows + row) * kD + 4 * lane) = lo;
    if (lane == 0) qexp[row] = ldexpf(1.f, e);
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
                      uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2,
                      CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {s1_bytes, s2_bytes};
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, type, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tc

bool prepare_decode_tc(const DecodeArgs &a, TcLaunch *t) {
    if (a.kv_fp8 && a.cp_world > 1) return false;   // FP8 caches are decoded without context parallelism
    if (a.dtype != BKV_BF16 || a.D != tc::kD || a.nq > tc::kN || a.nq <= 0) return false;
    if (a.bs < 8 || !((tc::kTile % a.bs == 0) || (a.bs % tc::kTile == 0))) return false;
    if (a.G > 256 || a.q_len > 256 || a.H_kv > 65535 || a.num_reqs > tc::kMaxReqs || !a.stream_k) return false;
    if ((int64_t)a.total_blocks * a.bs >= ((int64_t)1 << 31) || a.total_blocks <= 0) return false;
    if ((int64_t)a.num_reqs * a.q_len >= ((int64_t)1 << 31)) return false;
    // the tile prefix sums and the global tile numbers stay within int32
    if ((int64_t)a.num_reqs * ((a.max_ctx + tc::kTile - 1) / tc::kTile) * a.H_kv >= ((int64_t)1 << 31)) return false;
    if (!aligned(a.k, 16) || !aligned(a.v, 16) || !aligned(a.q, 16) || !aligned(a.out, 16)) return false;
    if (!tc::encode_fn()) return false;
    using namespace tc;
    t->seg_rows = a.bs < kTile ? a.bs : kTile;
    const uint64_t rows = (uint64_t)a.total_blocks * (uint64_t)a.bs;
    if (a.kv_fp8) {
        // E4M3 codes: one box of 128 codes (the whole head_dim, 128 bytes) per row;
        // the split queries (two parts stacked along the token rows) likewise
        if (!a.q8 || !aligned(a.q8, 16)) return false;
        const uint64_t row_stride = (uint64_t)a.H_kv * kD;
        const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
        if (!encode_3d(&t->mk, a.k, kD, a.H_kv, rows, kD, row_stride, 128, 1, t->seg_rows, u8) ||
            !encode_3d(&t->mv, a.v, kD, a.H_kv, rows, kD, row_stride, 128, 1, t->seg_rows, u8))
            return false;
        return encode_3d(&t->mq, a.q8, kD, a.H_q, 2 * (uint64_t)a.num_reqs * a.q_len, kD, (uint64_t)a.H_q * kD, 128,
                         a.G, a.q_len, u8);
    }
    const uint64_t row_stride = (uint64_t)a.H_kv * kD * 2;
    return encode_3d(&t->mk, a.k, kD, a.H_kv, rows, kD * 2, row_stride, 64, 1, t->seg_rows) &&
           encode_3d(&t->mv, a.v, kD, a.H_kv, rows, kD * 2, row_stride, 64, 1, t->seg_rows) &&
           encode_3d(&t->mq, a.q, kD, a.H_q, (uint64_t)a.num_reqs * a.q_len, kD * 2, (uint64_t)a.H_q * kD * 2, 64,
                     a.G, a.q_len);
}

template <bool kF8>
static int launch_variant(const DecodeArgs &a, const TcLaunch &t, cudaStream_t st) {
    using namespace tc;
    using C = Cfg<kF8>;
    // the grid is the stream-K CTA count the workspace was laid out for
    const int64_t grid = a.sk_grid;
    // the softmax handles only the query rows that exist (4, 8 or 16 columns);
    // context parallelism (global-position masks) has its own instances
    const bool cp = !kF8 && a.cp_world > 1;
    auto plain = a.nq <= 4 ? decode_tc_kernel<4, false, kF8>
                           : (a.nq <= 8 ? decode_tc_kernel<8, false, kF8> : decode_tc_kernel<16, false, kF8>);
    auto kern = plain;
    if constexpr (!kF8) {
        if (cp)
            kern = a.nq <= 4 ? decode_tc_kernel<4, true, false>
                             : (a.nq <= 8 ? decode_tc_kernel<8, true, false> : decode_tc_kernel<16, true, false>);
    }
    const int slot = (a.nq <= 4 ? 0 : (a.nq <= 8 ? 1 : 2)) + (cp ? 3 : 0) + (kF8 ? 6 : 0);
    static bool attr_set[64][9] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev][slot]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
            return launch_status();
        attr_set[dev][slot] = true;
    }
    const cudaError_t e = launch_pdl(kern, dim3((unsigned)grid), dim3(C::kThreads), C::kSmemBytes, st, t.mk, t.mv,
                                     t.mq, a, t.seg_rows);
    if (e != cudaSuccess) set_cuda_error(e);
    return launch_status();
}

int launch_q_split_e4m3(const DecodeArgs &a, cudaStream_t st) {
    const int64_t rows = (int64_t)a.num_reqs * a.q_len * a.H_q;
    const int64_t blocks = (rows + 7) / 8;
    if (blocks <= 0) return BKV_OK;
    if (blocks > 0x7fffffff) return BKV_ERR_INVALID_ARG;
    const cudaError_t e = launch_pdl(tc::q_split_e4m3_kernel, dim3((unsigned)blocks), dim3(256), 0, st,
                                     static_cast<const __nv_bfloat16 *>(a.q), rows, a.q8, a.qexp);
    if (e != cudaSuccess) set_cuda_error(e);
    return launch_status();
}

int launch_decode_tc(const DecodeArgs &a, const TcLaunch &t, cudaStream_t st) {
    return a.kv_fp8 ? launch_variant<true>(a, t, st) : launch_variant<false>(a, t, st);
}

}  // namespace bkv
