// bkv_ragged.cu -- paged attention over a mixed (ragged) step: requests with
// any number of query tokens (decode tokens, speculative drafts, prefill
// chunks) in one packed batch ("Padding and Batching with Block KV",
// Batching with Block KV: a request's new tokens are consecutive positions
// ending at its cache length; Cache Masking for the causal mask_active).
//
// bf16 with head_dim 128 runs the tensor-core prefill kernel
// (bkv_ragged_tc.cu); every other case this CUDA-core kernel: one CTA per
// (request, KV head, group of QR query rows), four warps striding over the
// request's visible keys with their own online softmax, combined at the end
// and written normalised (no workspace).
#include <cuda_bf16.h>
#include <math.h>

#include "bkv_ragged.cuh"

namespace bkv {

static constexpr float kLog2eR = 1.4426950408889634f;

__device__ __forceinline__ float rto_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float rto_f(float x) { return x; }
__device__ __forceinline__ void rstore(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }
__device__ __forceinline__ void rstore(float *p, float x) { *p = x; }

__device__ __forceinline__ float rwarp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <typename T, int DPL, int QR>
__global__ void __launch_bounds__(128) ragged_generic_kernel(const RaggedArgs a) {
    constexpr int NW = 4;
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int rg = blockIdx.x;
    const int r = rg / a.H_kv;
    const int g = rg - r * a.H_kv;
    const RaggedReq x = ragged_req(a, r);
    if (x.bad && g == 0 && blockIdx.y == 0 && threadIdx.x == 0 && a.err) atomicAdd(a.err, 1);
    const int i0 = blockIdx.y * QR;                 // first query row: row = token * G + (h % G)
    if (i0 >= x.ql * a.G) return;
    const int nrows = min(QR, x.ql * a.G - i0);
    const T *Q = static_cast<const T *>(a.q);
    const T *K = static_cast<const T *>(a.k);
    const T *V = static_cast<const T *>(a.v);

    float q[QR][DPL];
    int32_t lastv[QR];
    int32_t jmax = -1;
    int64_t orow[QR];
#pragma unroll
    for (int i = 0; i < QR; ++i) {
        if (i < nrows) {
            const int row = i0 + i;
            const int t = row / a.G;
            const int h = g * a.G + (row - t * a.G);
            orow[i] = (x.t0 + t) * a.H_q + h;
            lastv[i] = a.mask_mode == 0 ? x.L - x.ql + t : x.L - 1;
            jmax = max(jmax, lastv[i]);
#pragma unroll
            for (int e = 0; e < DPL; ++e) {
                const int d = e * 32 + lane;
                q[i][e] = d < a.D ? rto_f(Q[orow[i] * a.D + d]) * a.scale_log2 : 0.f;
            }
        } else {
            orow[i] = 0;
            lastv[i] = -1;
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
    for (int32_t j = warp; j < x.L && j <= jmax; j += NW) {
        const int32_t lb = j / a.bs;
        const int32_t off = j - lb * a.bs;
        const bool first = off == 0 || j < NW;
        if (lb >= a.bt_cols) {
            if (first && lane == 0 && blockIdx.y == 0 && a.err) atomicAdd(a.err, 1);
            continue;
        }
        const int64_t b = __ldg(a.bt + (int64_t)r * a.bt_stride + lb);
        if (b <= 0) continue;   // null block or sentinel: masked, never read
        if (b >= a.total_blocks) {
            if (first && lane == 0 && blockIdx.y == 0 && a.err) atomicAdd(a.err, 1);
            continue;
        }
        const int64_t rowoff = ((b * a.bs + off) * a.H_kv + g) * a.D;
        float kv[DPL];
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
            const int d = e * 32 + lane;
            kv[e] = d < a.D ? rto_f(K[rowoff + d]) : 0.f;
        }
        float s[QR];
#pragma unroll
        for (int i = 0; i < QR; ++i) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc = fmaf(q[i][e], kv[e], acc);
            s[i] = rwarp_sum(acc);
        }
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
            const int d = e * 32 + lane;
            kv[e] = d < a.D ? rto_f(V[rowoff + d]) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < QR; ++i) {
            if (i < nrows && j <= lastv[i]) {
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
    // combine the four warps and write the normalised rows
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
    T *out = static_cast<T *>(a.out);
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
        // rows are reloaded by index: orow[] lives in registers of every thread
        const int row = i0 + i;
        const int t = row / a.G;
        const int h = g * a.G + (row - t * a.G);
        rstore(out + ((x.t0 + t) * a.H_q + h) * a.D + d, lsum > 0.f ? acc / lsum : 0.f);
    }
}

template <typename T, int DPL>
static cudaError_t launch_ragged_generic(const RaggedArgs &a, cudaStream_t st) {
    constexpr int QR = 8;
    const int64_t rows = (int64_t)a.max_q * a.G;
    const dim3 grid((unsigned)((int64_t)a.num_reqs * a.H_kv), (unsigned)ceil_div<int64_t>(rows, QR));
    return launch_pdl(ragged_generic_kernel<T, DPL, QR>, grid, dim3(128), 0, st, a);
}

template <typename T>
static cudaError_t launch_ragged_generic_dpl(const RaggedArgs &a, cudaStream_t st) {
    if (a.D <= 32) return launch_ragged_generic<T, 1>(a, st);
    if (a.D <= 64) return launch_ragged_generic<T, 2>(a, st);
    if (a.D <= 128) return launch_ragged_generic<T, 4>(a, st);
    return launch_ragged_generic<T, 8>(a, st);
}

}  // namespace bkv

extern "C" int bkv_paged_attention_ragged(const void *q, const int32_t *query_start_loc, const void *k_cache,
                                          const void *v_cache, const int32_t *block_table, int64_t bt_stride,
                                          int32_t bt_cols, const int32_t *context_lens, int32_t max_context_len,
                                          int32_t max_query_len, int32_t num_reqs, int64_t num_tokens,
                                          int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                          int32_t block_size, int64_t total_blocks, float softmax_scale,
                                          int mask_mode, int dtype, void *out, int32_t *err_count,
                                          bkv_stream_t stream) {
    using namespace bkv;
    if (dtype != BKV_BF16 && dtype != BKV_F32) return BKV_ERR_UNSUPPORTED;
    if (head_dim > 256 || head_dim % 2 != 0) return BKV_ERR_UNSUPPORTED;
    if (mask_mode != BKV_MASK_CAUSAL && mask_mode != BKV_MASK_ALL) return BKV_ERR_INVALID_ARG;
    if (num_reqs < 0 || num_tokens < 0 || max_query_len < 0 || max_context_len < 0 || num_q_heads <= 0 ||
        num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0 ||
        bt_cols < 0 || bt_stride < bt_cols || total_blocks < 0)
        return BKV_ERR_INVALID_ARG;
    if ((int64_t)num_reqs * num_kv_heads >= ((int64_t)1 << 31)) return BKV_ERR_INVALID_ARG;
    const int64_t G = num_q_heads / num_kv_heads;
    if (ceil_div<int64_t>((int64_t)max_query_len * G, 8) > 65535) return BKV_ERR_INVALID_ARG;
    if (num_reqs == 0 || num_tokens == 0 || max_query_len == 0) return BKV_OK;
    if (!q || !out || !query_start_loc || !context_lens || (bt_cols > 0 && !block_table))
        return BKV_ERR_INVALID_ARG;
    if (max_context_len > 0 && (!k_cache || !v_cache)) return BKV_ERR_INVALID_ARG;
    if (!(softmax_scale > 0.f)) softmax_scale = 1.0f / sqrtf((float)head_dim);
    RaggedArgs a;
    a.q = q;
    a.qsl = query_start_loc;
    a.k = k_cache;
    a.v = v_cache;
    a.bt = block_table;
    a.bt_stride = bt_stride;
    a.bt_cols = bt_cols;
    a.ctx = context_lens;
    a.max_ctx = max_context_len;
    a.max_q = max_query_len;
    a.num_reqs = num_reqs;
    a.num_tokens = num_tokens;
    a.H_q = num_q_heads;
    a.H_kv = num_kv_heads;
    a.D = head_dim;
    a.bs = block_size;
    a.G = (int32_t)G;
    a.total_blocks = total_blocks;
    a.scale_log2 = softmax_scale * kLog2eR;
    a.mask_mode = mask_mode;
    a.dtype = dtype;
    a.out = out;
    a.err = err_count;
    RaggedTc t;
    if (prepare_ragged_tc(a, &t)) return launch_ragged_tc(a, t, (cudaStream_t)stream);
    const cudaError_t e = dtype == BKV_BF16 ? launch_ragged_generic_dpl<__nv_bfloat16>(a, (cudaStream_t)stream)
                                            : launch_ragged_generic_dpl<float>(a, (cudaStream_t)stream);
    if (e != cudaSuccess) set_cuda_error(e);
    return launch_status();
}
