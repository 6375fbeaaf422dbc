// bkv_decode.cu -- GQA paged decode attention: planner, the generic
// CUDA-core partition kernel, the split-KV merge kernel and the ABI entry
// points.
//
// "Padding and Batching with Block KV", Cache Masking: a query of request r
// sees cached positions [0, cache_len) (mask_cache) and, among this step's
// tokens, those the mask_active reading allows (causal by default, all-ones
// on request).  Special Block and Slot Values: a null (0) or sentinel (-1)
// table entry contributes nothing.  "Decode Context-Length Bucketing",
// Problem: read only the ceil(cache_len / block_size) blocks a request needs.
//
// Work decomposition: a unit is (request, KV head, partition of `chunk`
// logical positions).  Every query row of the KV head's GQA group (q_len *
// G rows) is handled in the unit, so each K/V byte is read once.  A unit
// writes an unnormalised partial (o, running max m, weight sum l) to the
// workspace; the merge kernel combines a request's partitions with
// log-sum-exp weights.  Partition boundaries depend only on logical
// positions, so the result is independent of where blocks sit in memory.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "bkv_decode.cuh"

namespace bkv {

static constexpr float kLog2e = 1.4426950408889634f;
static constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(float x) { return x; }
// an E4M3 cache code as its (unscaled) value, exactly
__device__ __forceinline__ float to_f(__nv_fp8_e4m3 x) { return static_cast<float>(x); }
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }
__device__ __forceinline__ void store_out(float *p, float x) { *p = x; }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Cache length of request r, clamped to the host bound (an excess is an error).
__device__ __forceinline__ int32_t clamped_len(const DecodeArgs &a, int r, bool count) {
    int32_t L = __ldg(a.ctx + r);
    if (L > a.max_ctx) {
        if (count && a.err) atomicAdd(a.err, 1);
        L = a.max_ctx;
    }
    return L > 0 ? L : 0;
}

// ---------------------------------------------------------------------------
// Generic partition kernel: any dtype, head_dim <= 256, any block size.
// CTA = (unit = (request * H_kv + KV head) * n_chunks + partition, group of
// up to QR query rows); four
// warps stride over the partition's positions, lanes split head_dim, dot
// products reduce with warp shuffles, each warp keeps its own online softmax
// and the four are combined through shared memory at the end.
// ---------------------------------------------------------------------------
template <typename T, typename KV, int DPL, int QR>
__global__ void __launch_bounds__(128) decode_generic_kernel(const DecodeArgs a) {
    constexpr int NW = 4;
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int rg = blockIdx.x / a.n_chunks;
    const int c = blockIdx.x - rg * a.n_chunks;
    const int r = rg / a.H_kv;
    const int g = rg - r * a.H_kv;
    const int i0 = blockIdx.y * QR;

    // L: global cache length (masks); Lk: the keys this rank holds (loop)
    const int32_t L = clamped_len(a, r, c == 0 && g == 0 && blockIdx.y == 0 && threadIdx.x == 0);
    const int32_t Lk = cp_local_len(a, L);
    const int32_t start = c * a.chunk;
    if (start >= Lk) return;
    const int32_t end = min(start + a.chunk, Lk);
    const int nrows = min(QR, a.nq - i0);

    const T *Q = static_cast<const T *>(a.q);
    const KV *K = static_cast<const KV *>(a.k);
    const KV *V = static_cast<const KV *>(a.v);

    float q[QR][DPL];
    int32_t lastv[QR], firstv[QR];
    int32_t jmax = -1;
    const int32_t jmin = window_lo(a, L);   // no query sees a key before this one
#pragma unroll
    for (int i = 0; i < QR; ++i) {
        if (i < nrows) {
            const int row = i0 + i;
            const int t = row / a.G;
            const int h = g * a.G + (row - t * a.G);
            const int64_t qb = (((int64_t)r * a.q_len + t) * a.H_q + h) * a.D;
            lastv[i] = a.mask_mode == 0 ? L - a.q_len + t : L - 1;
            firstv[i] = a.window > 0 ? L - a.q_len + t - a.window + 1 : INT32_MIN;
            jmax = max(jmax, lastv[i]);
#pragma unroll
            for (int e = 0; e < DPL; ++e) {
                const int d = e * 32 + lane;
                q[i][e] = d < a.D ? to_f(Q[qb + d]) * a.scale_log2 : 0.f;
            }
        } else {
            lastv[i] = -1;
            firstv[i] = 0;
#pragma unroll
            for (int e = 0; e < DPL; ++e) q[i][e] = 0.f;
        }
    }

    float m[QR], l[QR], o[QR][DPL];
#pragma unroll
    for (int i = 0; i < QR; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[i][e] = 0.f;
    }

    const int32_t j0 = max(start, jmin);   // a window implies cp_world == 1: local = global
    // Bad entries among the blocks this partition needs (past the table width,
    // or an id past the cache): counted once per (request, KV head) by the
    // first query-row group.  Partitions hold whole blocks, so no block is
    // counted twice; every needed block counts, whichever query sees it.
    if (a.err && blockIdx.y == 0 && j0 < end) {
        for (int32_t lb = j0 / a.bs + threadIdx.x; lb <= (end - 1) / a.bs; lb += blockDim.x) {
            const bool bad = lb >= a.bt_cols || __ldg(a.bt + (int64_t)r * a.bt_stride + lb) >= a.total_blocks;
            if (bad) atomicAdd(a.err, 1);
        }
    }
    for (int32_t j = j0 + warp; j < end && cp_global(a, j) <= jmax; j += NW) {
        const int64_t gj = cp_global(a, j);
        const int32_t lb = j / a.bs;
        const int32_t off = j - lb * a.bs;
        if (lb >= a.bt_cols) continue;
        const int64_t b = __ldg(a.bt + (int64_t)r * a.bt_stride + lb);
        if (b <= 0 || b >= a.total_blocks) continue;  // null, sentinel or bad: masked, never read
        const int64_t rowoff = ((b * a.bs + off) * a.H_kv + g) * a.D;
        float kv[DPL];
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
            const int d = e * 32 + lane;
            kv[e] = d < a.D ? to_f(K[rowoff + d]) : 0.f;
        }
        float s[QR];
#pragma unroll
        for (int i = 0; i < QR; ++i) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc = fmaf(q[i][e], kv[e], acc);
            s[i] = warp_sum(acc);
        }
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
            const int d = e * 32 + lane;
            kv[e] = d < a.D ? to_f(V[rowoff + d]) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < QR; ++i) {
            if (i < nrows && gj <= lastv[i] && gj >= firstv[i]) {
                const float mn = fmaxf(m[i], s[i]);
                const float corr = exp2f(m[i] - mn);
                const float p = exp2f(s[i] - mn);
                l[i] = fmaf(l[i], corr, p);
#pragma unroll
                for (int e = 0; e < DPL; ++e) o[i][e] = fmaf(o[i][e], corr, p * kv[e]);
                m[i] = mn;
            }
        }
    }

    // Combine the four warps' (m, l, o) and write the partition's partial.
    __shared__ float sm_m[NW][QR], sm_l[NW][QR];
    __shared__ float sm_o[NW][QR][32 * DPL];
#pragma unroll
    for (int i = 0; i < QR; ++i) {
        if (lane == 0) {
            sm_m[warp][i] = m[i];
            sm_l[warp][i] = l[i];
        }
#pragma unroll
        for (int e = 0; e < DPL; ++e) sm_o[warp][i][e * 32 + lane] = o[i][e];
    }
    __syncthreads();
    const int64_t unit = (int64_t)rg * a.n_chunks + c;
    for (int idx = threadIdx.x; idx < nrows * a.D; idx += blockDim.x) {
        const int i = idx / a.D;
        const int d = idx - i * a.D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, sm_m[w][i]);
        float acc = 0.f, lsum = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float f = exp2f(sm_m[w][i] - M);
                acc = fmaf(f, sm_o[w][i][d], acc);
                lsum = fmaf(f, sm_l[w][i], lsum);
            }
        }
        const int64_t prow = unit * a.parts * a.nq + i0 + i;
        a.ws_o[prow * a.D + d] = acc;
        if (d == 0) {
            a.ws_ml[prow * 2 + 0] = M;
            a.ws_ml[prow * 2 + 1] = lsum;
        }
    }
}

// ---------------------------------------------------------------------------
// Merge: out = sum_c 2^(m_c - M) o_c / sum_c 2^(m_c - M) l_c over a stream's
// partial slots, M = max_c m_c; 0 when no slot saw a visible key.  One CTA
// per stream (request, KV head); each warp takes query rows warp, warp + 4,
// ...: the lanes read the slots' (m, l) pairs in one round and keep the
// weights (up to 32 slots: lane k slot k; beyond, in the warp's own shared-
// memory strip), and then each lane sums four head_dim elements over the
// slots with 16-byte loads, eight slots (up to 8 slots and head_dim 128:
// all of them) per round of loads.
// The stream's slots follow from the context lengths alone (the stream-K
// split of the tensor-core kernel), which the partition kernel does not
// write: they are read and the slot range computed before the grid-
// dependency wait, so that only the partials' loads follow it.
// ---------------------------------------------------------------------------
template <typename T>
// (six CTAs per SM: on batches of thousands of streams the merge runs in waves)
__global__ void __launch_bounds__(128, 6) decode_merge_kernel(const DecodeArgs a, int max_slots) {
    extern __shared__ float sw[];   // [4 warps][max_slots] weights
    __shared__ int64_t red[2][4];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t rg = blockIdx.x;            // stream: r * H_kv + g
    const int r = (int)(rg / a.H_kv);
    const int g = (int)(rg - (int64_t)r * a.H_kv);
    const int32_t L = cp_local_len(a, clamped_len(a, r, false));   // keys this rank holds
    // a stream's partial slots are contiguous
    int nch = 0;          // slots of this stream
    int64_t unit0 = 0;    // its first slot
    if (a.stream_k) {
        // tiles of all requests and of those before r, over the CTA
        int64_t all = 0, before = 0;
        for (int rr = threadIdx.x; rr < a.num_reqs; rr += blockDim.x) {
            const int64_t t = sk_tiles(a, __ldg(a.ctx + rr));
            all += t;
            if (rr < r) before += t;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            all += __shfl_xor_sync(0xffffffffu, all, o);
            before += __shfl_xor_sync(0xffffffffu, before, o);
        }
        if (lane == 0) {
            red[0][warp] = all;
            red[1][warp] = before;
        }
        __syncthreads();
        all = red[0][0] + red[0][1] + red[0][2] + red[0][3];
        before = red[1][0] + red[1][1] + red[1][2] + red[1][3];
        const int64_t Ts = sk_tiles(a, __ldg(a.ctx + r));   // tiles of the stream
        const int64_t TP = all;
        if (Ts > 0 && L > 0) {
            // request r's Ts position tiles start at tile `before`; of the P = sk_grid /
            // H_kv groups, group q of peff = min(P, TP) covers [q TP / peff, (q + 1) TP /
            // peff), and its CTA for head g writes slots 2 (g (P + R) + q + r) + {0, 1}
            const int64_t P = a.sk_grid / a.H_kv;
            const int64_t peff = TP < P ? TP : P;
            const int64_t q0 = ((before + 1) * peff - 1) / TP;
            const int64_t q1 = ((before + Ts) * peff - 1) / TP;
            nch = (int)(2 * (q1 - q0 + 1));
            unit0 = 2 * ((int64_t)g * (P + a.num_reqs) + q0 + r);
        }
    } else {
        nch = L > 0 ? (int)ceil_div<int32_t>(L, a.chunk) * a.parts : 0;
        unit0 = rg * a.n_chunks * a.parts;
    }
    pdl_wait();
    pdl_trigger();
    if (nch <= 4 && (a.D & 3) == 0 && a.D <= 128) {
        // at most 4 slots and head_dim <= 128 (streams no CTA split, or split once): a warp's rows
        // (warp, warp + 4, ...) two at a time, every (m, l) and partial load of the two issued
        // before either is used, so two rows cost one round of loads (two, not more: the
        // registers stay low enough for six CTAs per SM); lane k keeps slot k's weight, lanes past
        // head_dim / 4 load and store no partials
        const bool act = lane < a.D / 4;
        for (int row0 = warp; row0 < a.nq; row0 += 8) {
            float2 ml[2];
            float4 v[2][4];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int row = row0 + 4 * i;
                const bool rv = row < a.nq;
                ml[i] = (rv && lane < nch) ? *reinterpret_cast<const float2 *>(a.ws_ml + ((unit0 + lane) * a.nq + row) * 2)
                                           : make_float2(-INFINITY, 0.f);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    v[i][k] = (rv && act && k < nch)
                                  ? *reinterpret_cast<const float4 *>(a.ws_o + ((unit0 + k) * a.nq + row) * a.D + 4 * lane)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int row = row0 + 4 * i;
                if (row >= a.nq) break;   // the same for the whole warp
                const int t = row / a.G;
                const int h = g * a.G + (row - t * a.G);
                const int64_t orow = ((int64_t)r * a.q_len + t) * a.H_q + h;
                T *out = static_cast<T *>(a.out) + orow * a.D;
                float M = ml[i].x;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
                const float wl = (M == -INFINITY || lane >= nch) ? 0.f : exp2f(ml[i].x - M);
                const float lsum = warp_sum(wl * ml[i].y);
                const float iv = (M == -INFINITY || !(lsum > 0.f)) ? 0.f : a.v_scale / lsum;
                if (a.lse && lane == 0)
                    a.lse[orow] = (M == -INFINITY || !(lsum > 0.f)) ? -INFINITY : (M + log2f(lsum)) * kLn2;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float wgt = __shfl_sync(0xffffffffu, wl, k);
                    acc.x = fmaf(wgt, v[i][k].x, acc.x);
                    acc.y = fmaf(wgt, v[i][k].y, acc.y);
                    acc.z = fmaf(wgt, v[i][k].z, acc.z);
                    acc.w = fmaf(wgt, v[i][k].w, acc.w);
                }
                if (act) {
                    store_out(out + 4 * lane + 0, acc.x * iv);
                    store_out(out + 4 * lane + 1, acc.y * iv);
                    store_out(out + 4 * lane + 2, acc.z * iv);
                    store_out(out + 4 * lane + 3, acc.w * iv);
                }
            }
        }
        return;
    }
    float *wts = sw + (size_t)warp * max_slots;
    for (int row = warp; row < a.nq; row += 4) {
        const int t = row / a.G;
        const int h = g * a.G + (row - t * a.G);
        const int64_t orow = ((int64_t)r * a.q_len + t) * a.H_q + h;
        T *out = static_cast<T *>(a.out) + orow * a.D;
        // log-sum-exp of the row, back from base 2 to natural log (-inf: no visible key)
        auto put_lse = [&](float M, float lsum) {
            if (a.lse && lane == 0)
                a.lse[orow] = (M == -INFINITY || !(lsum > 0.f)) ? -INFINITY : (M + log2f(lsum)) * kLn2;
        };
        if (nch <= 32 && (a.D & 3) == 0) {
            // up to 32 slots: lane k reads slot k's (m, l) and keeps its weight; the partials
            // are read eight slots at a time, the first eight issued together with the
            // (m, l) loads (they do not depend on the weights), so up to 8 slots and head_dim
            // 128 take one round of loads
            // every lane runs every round (the shuffles need the whole warp); lanes past head_dim / 4
            // load and store nothing
            const float2 ml = lane < nch
                                  ? *reinterpret_cast<const float2 *>(a.ws_ml + ((unit0 + lane) * a.nq + row) * 2)
                                  : make_float2(-INFINITY, 0.f);
            float wl = 0.f, iv = 0.f;
            for (int base = 0; base < a.D / 4; base += 32) {
                const int d4 = base + lane;
                const bool act = d4 < a.D / 4;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int c = 0; c < nch; c += 8) {
                    float4 v[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        if (act && c + k < nch)
                            v[k] = *reinterpret_cast<const float4 *>(a.ws_o + ((unit0 + c + k) * a.nq + row) * a.D +
                                                                     4 * d4);
                    if (base == 0 && c == 0) {
                        float M = ml.x;
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
                        wl = (M == -INFINITY || lane >= nch) ? 0.f : exp2f(ml.x - M);
                        const float lsum = warp_sum(wl * ml.y);
                        iv = (M == -INFINITY || !(lsum > 0.f)) ? 0.f : a.v_scale / lsum;
                        put_lse(M, lsum);
                    }
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float wgt = __shfl_sync(0xffffffffu, wl, (c + k) & 31);
                        if (act && c + k < nch) {
                            acc.x = fmaf(wgt, v[k].x, acc.x);
                            acc.y = fmaf(wgt, v[k].y, acc.y);
                            acc.z = fmaf(wgt, v[k].z, acc.z);
                            acc.w = fmaf(wgt, v[k].w, acc.w);
                        }
                    }
                }
                if (act) {
                    store_out(out + 4 * d4 + 0, acc.x * iv);
                    store_out(out + 4 * d4 + 1, acc.y * iv);
                    store_out(out + 4 * d4 + 2, acc.z * iv);
                    store_out(out + 4 * d4 + 3, acc.w * iv);
                }
            }
            if (nch == 0) put_lse(-INFINITY, 0.f);
            continue;
        }
        float M = -INFINITY;
        for (int c = lane; c < nch; c += 32) M = fmaxf(M, a.ws_ml[((unit0 + c) * a.nq + row) * 2]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float lsum = 0.f;
        for (int c = lane; c < nch; c += 32) {
            const float2 ml = *reinterpret_cast<const float2 *>(a.ws_ml + ((unit0 + c) * a.nq + row) * 2);
            const float wgt = M == -INFINITY ? 0.f : exp2f(ml.x - M);
            wts[c] = wgt;
            lsum = fmaf(wgt, ml.y, lsum);
        }
        lsum = warp_sum(lsum);
        const float iv = (M == -INFINITY || !(lsum > 0.f)) ? 0.f : a.v_scale / lsum;
        put_lse(M, lsum);
        __syncwarp();
        if ((a.D & 3) == 0) {
            for (int d4 = lane; d4 < a.D / 4; d4 += 32) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                int c = 0;
                for (; c + 4 <= nch; c += 4) {
                    float4 v[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        v[k] = *reinterpret_cast<const float4 *>(a.ws_o + ((unit0 + c + k) * a.nq + row) * a.D + 4 * d4);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float wgt = wts[c + k];
                        acc.x = fmaf(wgt, v[k].x, acc.x);
                        acc.y = fmaf(wgt, v[k].y, acc.y);
                        acc.z = fmaf(wgt, v[k].z, acc.z);
                        acc.w = fmaf(wgt, v[k].w, acc.w);
                    }
                }
                for (; c < nch; ++c) {
                    const float4 v = *reinterpret_cast<const float4 *>(a.ws_o + ((unit0 + c) * a.nq + row) * a.D + 4 * d4);
                    const float wgt = wts[c];
                    acc.x = fmaf(wgt, v.x, acc.x);
                    acc.y = fmaf(wgt, v.y, acc.y);
                    acc.z = fmaf(wgt, v.z, acc.z);
                    acc.w = fmaf(wgt, v.w, acc.w);
                }
                store_out(out + 4 * d4 + 0, acc.x * iv);
                store_out(out + 4 * d4 + 1, acc.y * iv);
                store_out(out + 4 * d4 + 2, acc.z * iv);
                store_out(out + 4 * d4 + 3, acc.w * iv);
            }
        } else {
            for (int d = lane; d < a.D; d += 32) {
                float acc = 0.f;
                for (int c = 0; c < nch; ++c) acc = fmaf(wts[c], a.ws_o[((unit0 + c) * a.nq + row) * a.D + d], acc);
                store_out(out + d, acc * iv);
            }
        }
        __syncwarp();   // the weight strip is rewritten for the warp's next row
    }
}

// ---------------------------------------------------------------------------
// Planner
// ---------------------------------------------------------------------------
static int64_t gcd64(int64_t x, int64_t y) {
    while (y) {
        int64_t t = x % y;
        x = y;
        y = t;
    }
    return x;
}

bool make_decode_plan(int32_t num_reqs, int32_t q_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, int32_t max_context_len, DecodePlan *plan) {
    if (num_reqs <= 0 || q_len <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        max_context_len < 0 || num_q_heads % num_kv_heads != 0 || block_size > 65536)
        return false;
    // Partitions are whole 128-position tiles and whole blocks.  512
    // positions keeps the partial outputs near 2% of the K/V bytes while
    // leaving enough units for an even spread over the SMs; large batches of
    // long requests take bigger partitions (up to 2048) to cut partial
    // traffic, small ones smaller partitions to fill the device.
    const int64_t align = (int64_t)block_size / gcd64(block_size, 128) * 128;
    const int64_t units = (int64_t)num_reqs * num_kv_heads;
    const int64_t sms = current_sm_count();
    int64_t chunk = 512;
    const int64_t big = (int64_t)max_context_len * units / (32 * sms);
    if (big > chunk) chunk = big < 2048 ? big : 2048;
    chunk = ceil_div<int64_t>(chunk, align) * align;
    if (units * ceil_div<int64_t>(max_context_len, chunk) < 4 * sms) {
        // Few, short units: split finer so the grid still fills the device.
        const int64_t want = ceil_div<int64_t>((int64_t)max_context_len * units, 4 * sms);
        chunk = ceil_div<int64_t>(want > 0 ? want : 1, align) * align;
    }
    // keep the merge's weight tables (4 warps x partitions, fp32) within 32 KB
    if (ceil_div<int64_t>(max_context_len, chunk) > 2048)
        chunk = ceil_div<int64_t>(ceil_div<int64_t>(max_context_len, 2048), align) * align;
    if (chunk > (int64_t)1 << 30) return false;
    const int64_t n_chunks = max_context_len > 0 ? ceil_div<int64_t>(max_context_len, chunk) : 1;
    const int64_t nq = (int64_t)q_len * (num_q_heads / num_kv_heads);
    if (units * n_chunks >= ((int64_t)1 << 31) || nq > 65535 * 8) return false;
    plan->chunk = (int32_t)chunk;
    plan->n_chunks = (int32_t)n_chunks;
    plan->nq = (int32_t)nq;
    // the tensor-core kernel's grid: whole groups of one CTA per KV head
    plan->sk_grid = (int32_t)(num_kv_heads <= sms ? (sms / num_kv_heads) * num_kv_heads : num_kv_heads);
    plan->header_bytes = 256;
    const int64_t slots_generic = units * n_chunks;
    const int64_t slots_sk = 2 * (plan->sk_grid + units);
    const int64_t slots = slots_generic > slots_sk ? slots_generic : slots_sk;
    const int64_t prows = slots * nq;
    const int64_t o_bytes = ceil_div<int64_t>(prows * head_dim * 4, 256) * 256;
    const int64_t part_bytes = ceil_div<int64_t>(o_bytes + prows * 2 * 4, 256) * 256;
    // the FP8 tensor-core path's split queries: two E4M3 parts and a scale per row
    const int64_t qrows = (int64_t)num_reqs * q_len * num_q_heads;
    const int64_t q8_bytes = head_dim == 128 ? qrows * (2 * 128 + 4) : 0;
    plan->q8_offset = plan->header_bytes + (size_t)part_bytes;
    plan->ws_bytes = plan->q8_offset + (size_t)q8_bytes;
    return true;
}

template <typename T, typename KV, int DPL>
static void launch_generic(const DecodeArgs &a, cudaStream_t st) {
    constexpr int QR = 8;
    dim3 grid(a.n_chunks * a.num_reqs * a.H_kv, ceil_div(a.nq, QR));
    const cudaError_t e = launch_pdl(decode_generic_kernel<T, KV, DPL, QR>, grid, dim3(128), 0, st, a);
    if (e != cudaSuccess) set_cuda_error(e);
}

template <typename T, typename KV>
static void launch_generic_dpl(const DecodeArgs &a, cudaStream_t st) {
    if (a.D <= 32) launch_generic<T, KV, 1>(a, st);
    else if (a.D <= 64) launch_generic<T, KV, 2>(a, st);
    else if (a.D <= 128) launch_generic<T, KV, 4>(a, st);
    else launch_generic<T, KV, 8>(a, st);
}

}  // namespace bkv

extern "C" size_t bkv_paged_decode_workspace_size(int32_t num_reqs, int32_t q_len, int32_t num_q_heads,
                                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                                  int32_t max_context_len) {
    bkv::DecodePlan p;
    if (!bkv::make_decode_plan(num_reqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                               &p))
        return 0;
    return p.ws_bytes;
}

namespace bkv {

// Not part of the ABI (bkv.h does not declare it): a process-wide switch that
// makes every later decode call run the CUDA-core kernel, so that the
// tensor-core kernel can be timed against it on the same shapes.  The library
// itself never sets it.
static volatile int g_force_generic = 0;

}  // namespace bkv

extern "C" void bkv_testing_force_generic_decode(int on) { bkv::g_force_generic = on ? 1 : 0; }

namespace bkv {

// Everything one decode call needs, decided from its arguments alone (so the
// partition and merge entry points, called separately with the same
// arguments, agree on the kernel, the plan and the workspace layout).
struct DecodeCall {
    DecodeArgs a;
    DecodePlan plan;
    bool tc;
    TcLaunch t;
};

static int decode_setup(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                        int64_t bt_stride, int32_t bt_cols, const int32_t *context_lens, int32_t max_context_len,
                        int32_t num_reqs, int32_t q_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                        int32_t block_size, int64_t total_blocks, float softmax_scale, int mask_mode, int dtype,
                        int32_t sliding_window, int32_t cp_world, int32_t cp_rank, int32_t cp_interleave,
                        void *out, float *lse, void *workspace, size_t workspace_bytes, int32_t *err_count,
                        DecodeCall *c, int kv_fp8 = 0, float k_scale = 1.f, float v_scale = 1.f) {
    if (dtype != BKV_BF16 && dtype != BKV_F32) return BKV_ERR_UNSUPPORTED;
    if (kv_fp8 && (!(k_scale > 0.f) || !(v_scale > 0.f) || !isfinite(k_scale) || !isfinite(v_scale)))
        return BKV_ERR_INVALID_ARG;
    if (sliding_window < 0) return BKV_ERR_INVALID_ARG;
    if (cp_world < 1 || cp_rank < 0 || cp_rank >= cp_world || cp_interleave < 1) return BKV_ERR_INVALID_ARG;
    if (cp_world > 1 && sliding_window > 0) return BKV_ERR_UNSUPPORTED;
    if (head_dim > 256 || head_dim % 2 != 0) return BKV_ERR_UNSUPPORTED;
    if (mask_mode != BKV_MASK_CAUSAL && mask_mode != BKV_MASK_ALL) return BKV_ERR_INVALID_ARG;
    if (bt_cols < 0 || bt_stride < bt_cols || total_blocks < 0) return BKV_ERR_INVALID_ARG;
    DecodePlan &plan = c->plan;
    if (!make_decode_plan(num_reqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len, &plan))
        return BKV_ERR_INVALID_ARG;
    if (!q || !out || !context_lens || (bt_cols > 0 && !block_table)) return BKV_ERR_INVALID_ARG;
    if (max_context_len > 0 && (!k_cache || !v_cache)) return BKV_ERR_INVALID_ARG;
    if (workspace_bytes < plan.ws_bytes || !workspace || !aligned(workspace, 16)) return BKV_ERR_INVALID_ARG;
    if (!(softmax_scale > 0.f)) softmax_scale = 1.0f / sqrtf((float)head_dim);

    DecodeArgs &a = c->a;
    a.q = q;
    a.k = k_cache;
    a.v = v_cache;
    a.bt = block_table;
    a.bt_stride = bt_stride;
    a.bt_cols = bt_cols;
    a.ctx = context_lens;
    a.max_ctx = max_context_len;
    a.num_reqs = num_reqs;
    a.q_len = q_len;
    a.H_q = num_q_heads;
    a.H_kv = num_kv_heads;
    a.D = head_dim;
    a.bs = block_size;
    a.total_blocks = total_blocks;
    // an FP8 key is its code's value times k_scale: the factor joins the score scale
    a.scale_log2 = kv_fp8 ? softmax_scale * kLog2e * k_scale : softmax_scale * kLog2e;
    a.kv_fp8 = kv_fp8;
    a.v_scale = kv_fp8 ? v_scale : 1.f;
    a.mask_mode = mask_mode;
    a.window = sliding_window;
    a.cp_world = cp_world;
    a.cp_rank = cp_rank;
    a.cp_inter = cp_interleave;
    a.lse = lse;
    a.dtype = dtype;
    a.chunk = plan.chunk;
    a.n_chunks = plan.n_chunks;
    a.G = num_q_heads / num_kv_heads;
    a.nq = plan.nq;
    a.out = out;
    a.err = err_count;
    // partial-slot layout of the kernel that runs (see DecodePlan)
    auto set_slots = [&](int64_t slots) {
        char *base = static_cast<char *>(workspace) + plan.header_bytes;
        a.ws_o = reinterpret_cast<float *>(base);
        a.ws_ml = reinterpret_cast<float *>(base + ceil_div<int64_t>(slots * plan.nq * head_dim * 4, 256) * 256);
    };
    const int64_t units = (int64_t)num_reqs * num_kv_heads;
    a.q8 = head_dim == 128 ? static_cast<uint8_t *>(workspace) + plan.q8_offset : nullptr;
    a.qexp = head_dim == 128 ? reinterpret_cast<float *>(a.q8 + (size_t)2 * num_reqs * q_len * num_q_heads * 128)
                             : nullptr;
    a.parts = 2;
    a.stream_k = 1;
    a.sk_grid = plan.sk_grid;
    set_slots(2 * (plan.sk_grid + units));
    c->tc = !g_force_generic && prepare_decode_tc(a, &c->t);
    if (!c->tc) {
        a.parts = 1;
        a.stream_k = 0;
        set_slots(units * plan.n_chunks);
    }
    return BKV_OK;
}

static int decode_partition(DecodeCall &c, cudaStream_t st) {
    if (c.tc) {
        if (c.a.kv_fp8) {
            const int rc = launch_q_split_e4m3(c.a, st);
            if (rc != BKV_OK) return rc;
        }
        return launch_decode_tc(c.a, c.t, st);
    }
    if (c.a.kv_fp8) {
        if (c.a.dtype == BKV_BF16) launch_generic_dpl<__nv_bfloat16, __nv_fp8_e4m3>(c.a, st);
        else launch_generic_dpl<float, __nv_fp8_e4m3>(c.a, st);
    } else if (c.a.dtype == BKV_BF16) {
        launch_generic_dpl<__nv_bfloat16, __nv_bfloat16>(c.a, st);
    } else {
        launch_generic_dpl<float, float>(c.a, st);
    }
    return launch_status();
}

static int decode_merge(DecodeCall &c, cudaStream_t st) {
    const DecodeArgs &a = c.a;
    const int max_slots = a.stream_k ? 2 * c.plan.sk_grid : c.plan.n_chunks * a.parts;
    const size_t msmem = 4 * (size_t)max_slots * 4;
    const dim3 mgrid((unsigned)((int64_t)a.num_reqs * a.H_kv));
    const cudaError_t e =
        a.dtype == BKV_BF16
            ? launch_pdl(decode_merge_kernel<__nv_bfloat16>, mgrid, dim3(128), msmem, st, a, max_slots)
            : launch_pdl(decode_merge_kernel<float>, mgrid, dim3(128), msmem, st, a, max_slots);
    if (e != cudaSuccess) set_cuda_error(e);
    return launch_status();
}

}  // namespace bkv

#define BKV_DECODE_PARAMS                                                                                         \
    const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table, int64_t bt_stride,      \
        int32_t bt_cols, const int32_t *context_lens, int32_t max_context_len, int32_t num_reqs, int32_t q_len,  \
        int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int64_t total_blocks,   \
        float softmax_scale, int mask_mode, int32_t sliding_window, int dtype, void *out, void *workspace,       \
        size_t workspace_bytes, int32_t *err_count, bkv_stream_t stream
#define BKV_DECODE_SETUP(c)                                                                                       \
    bkv::decode_setup(q, k_cache, v_cache, block_table, bt_stride, bt_cols, context_lens, max_context_len,       \
                      num_reqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, total_blocks, softmax_scale, \
                      mask_mode, dtype, sliding_window, 1, 0, 1, out, nullptr, workspace, workspace_bytes,      \
                      err_count, &(c))

extern "C" int bkv_paged_decode_swa(BKV_DECODE_PARAMS) {
    bkv::DecodeCall c;
    int rc = BKV_DECODE_SETUP(c);
    if (rc != BKV_OK) return rc;
    rc = bkv::decode_partition(c, (cudaStream_t)stream);
    if (rc != BKV_OK) return rc;
    return bkv::decode_merge(c, (cudaStream_t)stream);
}

// The full-attention decode: bkv_paged_decode_swa without a window.
extern "C" int bkv_paged_decode(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                                int64_t bt_stride, int32_t bt_cols, const int32_t *context_lens,
                                int32_t max_context_len, int32_t num_reqs, int32_t q_len, int32_t num_q_heads,
                                int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int64_t total_blocks,
                                float softmax_scale, int mask_mode, int dtype, void *out, void *workspace,
                                size_t workspace_bytes, int32_t *err_count, bkv_stream_t stream) {
    return bkv_paged_decode_swa(q, k_cache, v_cache, block_table, bt_stride, bt_cols, context_lens, max_context_len,
                                num_reqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, total_blocks,
                                softmax_scale, mask_mode, 0, dtype, out, workspace, workspace_bytes, err_count,
                                stream);
}

extern "C" int bkv_paged_decode_partition(BKV_DECODE_PARAMS) {
    bkv::DecodeCall c;
    const int rc = BKV_DECODE_SETUP(c);
    if (rc != BKV_OK) return rc;
    return bkv::decode_partition(c, (cudaStream_t)stream);
}

extern "C" int bkv_paged_decode_merge(BKV_DECODE_PARAMS) {
    bkv::DecodeCall c;
    const int rc = BKV_DECODE_SETUP(c);
    if (rc != BKV_OK) return rc;
    return bkv::decode_merge(c, (cudaStream_t)stream);
}

#define BKV_DECODE_FP8_PARAMS                                                                                     \
    const void *q, const uint8_t *k_cache, const uint8_t *v_cache, const int32_t *block_table, int64_t bt_stride, \
        int32_t bt_cols, const int32_t *context_lens, int32_t max_context_len, int32_t num_reqs, int32_t q_len,  \
        int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int64_t total_blocks,   \
        float softmax_scale, float k_scale, float v_scale, int mask_mode, int32_t sliding_window, int dtype,     \
        void *out, void *workspace, size_t workspace_bytes, int32_t *err_count, bkv_stream_t stream
#define BKV_DECODE_FP8_SETUP(c)                                                                                   \
    bkv::decode_setup(q, k_cache, v_cache, block_table, bt_stride, bt_cols, context_lens, max_context_len,       \
                      num_reqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, total_blocks, softmax_scale, \
                      mask_mode, dtype, sliding_window, 1, 0, 1, out, nullptr, workspace, workspace_bytes,      \
                      err_count, &(c), 1, k_scale, v_scale)

extern "C" int bkv_paged_decode_fp8(BKV_DECODE_FP8_PARAMS) {
    bkv::DecodeCall c;
    int rc = BKV_DECODE_FP8_SETUP(c);
    if (rc != BKV_OK) return rc;
    rc = bkv::decode_partition(c, (cudaStream_t)stream);
    if (rc != BKV_OK) return rc;
    return bkv::decode_merge(c, (cudaStream_t)stream);
}

extern "C" int bkv_paged_decode_fp8_partition(BKV_DECODE_FP8_PARAMS) {
    bkv::DecodeCall c;
    const int rc = BKV_DECODE_FP8_SETUP(c);
    if (rc != BKV_OK) return rc;
    return bkv::decode_partition(c, (cudaStream_t)stream);
}

extern "C" int bkv_paged_decode_fp8_merge(BKV_DECODE_FP8_PARAMS) {
    bkv::DecodeCall c;
    const int rc = BKV_DECODE_FP8_SETUP(c);
    if (rc != BKV_OK) return rc;
    return bkv::decode_merge(c, (cudaStream_t)stream);
}

extern "C" int bkv_paged_decode_cp(const void *q, const void *k_cache, const void *v_cache,
                                   const int32_t *block_table, int64_t bt_stride, int32_t bt_cols,
                                   const int32_t *context_lens, int32_t max_context_len, int32_t num_reqs,
                                   int32_t q_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, int64_t total_blocks, float softmax_scale, int mask_mode,
                                   int32_t cp_world, int32_t cp_rank, int32_t cp_interleave, int dtype, void *out,
                                   float *lse, void *workspace, size_t workspace_bytes, int32_t *err_count,
                                   bkv_stream_t stream) {
    bkv::DecodeCall c;
    int rc = bkv::decode_setup(q, k_cache, v_cache, block_table, bt_stride, bt_cols, context_lens, max_context_len,
                               num_reqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, total_blocks,
                               softmax_scale, mask_mode, dtype, 0, cp_world, cp_rank, cp_interleave, out, lse,
                               workspace, workspace_bytes, err_count, &c);
    if (rc != BKV_OK) return rc;
    rc = bkv::decode_partition(c, (cudaStream_t)stream);
    if (rc != BKV_OK) return rc;
    return bkv::decode_merge(c, (cudaStream_t)stream);
}

// ---------------------------------------------------------------------------
// Merge of attention states: rows of `parts` normalised partial outputs
// (outs [parts][rows][D]) with their natural-log sums of exponentials
// (lses [parts][rows]) into out = sum_k e^(lse_k - M) out_k / sum_k
// e^(lse_k - M) and lse_out = M + log sum_k e^(lse_k - M), M = max_k lse_k;
// all -inf gives 0 and -inf.  The combination step after the ranks of a
// context-parallel decode exchange their results.  One warp per row; for up
// to 32 parts lane k keeps part k's weight and the others take it by shuffle;
// with head_dim 128 and up to 8 parts every load of a row is issued at once.
// ---------------------------------------------------------------------------
namespace bkv {

// Four consecutive elements of a row as fp32 (one 8- or 16-byte load).
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162 *>(&u.x);
    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162 *>(&u.y);
    return make_float4(__low2float(lo), __high2float(lo), __low2float(hi), __high2float(hi));
}
__device__ __forceinline__ float4 load4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

template <typename T>
__global__ void __launch_bounds__(128) merge_states_kernel(const T *__restrict__ outs, const float *__restrict__ lses,
                                                           int parts, int64_t rows, int D, T *__restrict__ out,
                                                           float *__restrict__ lse_out) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (row >= rows) return;
    T *o = out + row * D;
    if (D == 128 && parts <= 8) {
        // every load of the row at once: lane k < parts its part's lse, each lane
        // its four elements of every part
        const float ll = lane < parts ? lses[(int64_t)lane * rows + row] : -INFINITY;
        float4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (k < parts) v[k] = load4(outs + ((int64_t)k * rows + row) * D + 4 * lane);
        float M = ll;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        const float wl = (M == -INFINITY || lane >= parts) ? 0.f : expf(ll - M);
        const float wsum = warp_sum(wl);
        const float iv = wsum > 0.f ? 1.f / wsum : 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float w = __shfl_sync(0xffffffffu, wl, k);
            if (k < parts) {
                acc.x = fmaf(w, v[k].x, acc.x);
                acc.y = fmaf(w, v[k].y, acc.y);
                acc.z = fmaf(w, v[k].z, acc.z);
                acc.w = fmaf(w, v[k].w, acc.w);
            }
        }
        store_out(o + 4 * lane + 0, acc.x * iv);
        store_out(o + 4 * lane + 1, acc.y * iv);
        store_out(o + 4 * lane + 2, acc.z * iv);
        store_out(o + 4 * lane + 3, acc.w * iv);
        if (lse_out && lane == 0) lse_out[row] = (M == -INFINITY || !(wsum > 0.f)) ? -INFINITY : M + logf(wsum);
        return;
    }
    float M = -INFINITY;
    for (int k = lane; k < parts; k += 32) M = fmaxf(M, lses[(int64_t)k * rows + row]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    auto weight = [&](int k) { return M == -INFINITY ? 0.f : expf(lses[(int64_t)k * rows + row] - M); };
    float wsum = 0.f;
    for (int k = lane; k < parts; k += 32) wsum += weight(k);
    wsum = warp_sum(wsum);
    const float iv = wsum > 0.f ? 1.f / wsum : 0.f;
    const float wl = (parts <= 32 && lane < parts) ? weight(lane) : 0.f;
    for (int d = lane; d < D; d += 32) {
        float acc = 0.f;
        for (int k = 0; k < parts; ++k) {
            const float w = parts <= 32 ? __shfl_sync(0xffffffffu, wl, k & 31) : weight(k);
            acc = fmaf(w, to_f(outs[((int64_t)k * rows + row) * D + d]), acc);
        }
        store_out(o + d, acc * iv);
    }
    if (lse_out && lane == 0) lse_out[row] = (M == -INFINITY || !(wsum > 0.f)) ? -INFINITY : M + logf(wsum);
}

}  // namespace bkv

extern "C" int bkv_merge_attn_states(const void *outs, const float *lses, int32_t parts, int64_t rows,
                                     int32_t head_dim, int dtype, void *out, float *lse_out, bkv_stream_t stream) {
    if (dtype != BKV_BF16 && dtype != BKV_F32) return BKV_ERR_UNSUPPORTED;
    if (parts < 1 || rows < 0 || head_dim < 1) return BKV_ERR_INVALID_ARG;
    if (rows == 0) return BKV_OK;
    if (!outs || !lses || !out) return BKV_ERR_INVALID_ARG;
    if (head_dim == 128 && (!bkv::aligned(outs, 16) || !bkv::aligned(out, 16))) return BKV_ERR_INVALID_ARG;
    const int64_t blocks = (rows + 3) / 4;
    if (blocks > 0x7fffffff) return BKV_ERR_INVALID_ARG;
    const cudaError_t e =
        dtype == BKV_BF16
            ? bkv::launch_pdl(bkv::merge_states_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(128), 0,
                              (cudaStream_t)stream, static_cast<const __nv_bfloat16 *>(outs), lses, (int)parts, rows,
                              (int)head_dim, static_cast<__nv_bfloat16 *>(out), lse_out)
            : bkv::launch_pdl(bkv::merge_states_kernel<float>, dim3((unsigned)blocks), dim3(128), 0,
                              (cudaStream_t)stream, static_cast<const float *>(outs), lses, (int)parts, rows,
                              (int)head_dim, static_cast<float *>(out), lse_out);
    if (e != cudaSuccess) bkv::set_cuda_error(e);
    return bkv::launch_status();
}
