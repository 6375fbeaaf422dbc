// bkv_cache_write.cu -- scatter of new K/V rows into the paged caches.
//
// "Padding and Batching with Block KV", Block Structure and Slot ID -1:
// Padding Tokens.  Row i (num_kv_heads * head_dim elements) lands at flat
// row s = slot_mapping[i] of the (total_blocks * block_size, H_kv * D) view
// of each cache; s < 0 writes nothing.
//
// One warp per token: a token's row is contiguous in both the source and the
// cache (2 KiB at H_kv = 8, D = 128, bf16), so each lane moves 16-byte
// vectors, all loads of a round issued before its stores.  HBM-bound: the
// algorithmic traffic is 2 * row bytes read + 2 * row bytes written + 8 bytes
// of slot id per token.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "bkv_internal.cuh"
#include "bkv_slot.cuh"

namespace bkv {

constexpr int kCwWarps = 8;     // warps per block
constexpr int kCwUnroll = 4;    // 16-byte vectors in flight per lane per tensor

// 16-byte path: row_bytes, the source stride and every base are multiples of 16.
__global__ void __launch_bounds__(kCwWarps * 32) cache_write_vec16_kernel(
    const char *__restrict__ k_new, const char *__restrict__ v_new, int64_t num_tokens, int64_t src_stride_bytes,
    const int64_t *__restrict__ slot_mapping, char *__restrict__ k_cache, char *__restrict__ v_cache,
    int64_t capacity, int64_t row_bytes, int32_t *err_count) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (int64_t)blockIdx.x * kCwWarps + (threadIdx.x >> 5);
    const int64_t wstep = (int64_t)gridDim.x * kCwWarps;
    for (int64_t i = warp0; i < num_tokens; i += wstep) {
        const int64_t s = __ldg(slot_mapping + i);
        if (s < 0) continue;
        if (s >= capacity) {
            if (lane == 0 && err_count) atomicAdd(err_count, 1);
            continue;
        }
        const char *ks = k_new + i * src_stride_bytes;
        const char *vs = v_new + i * src_stride_bytes;
        char *kd = k_cache + s * row_bytes;
        char *vd = v_cache + s * row_bytes;
        for (int64_t base = (int64_t)lane * 16; base < row_bytes; base += 32 * 16 * kCwUnroll) {
            uint4 kr[kCwUnroll], vr[kCwUnroll];
#pragma unroll
            for (int u = 0; u < kCwUnroll; ++u) {
                const int64_t off = base + (int64_t)u * 32 * 16;
                if (off < row_bytes) {
                    kr[u] = __ldg(reinterpret_cast<const uint4 *>(ks + off));
                    vr[u] = __ldg(reinterpret_cast<const uint4 *>(vs + off));
                }
            }
#pragma unroll
            for (int u = 0; u < kCwUnroll; ++u) {
                const int64_t off = base + (int64_t)u * 32 * 16;
                if (off < row_bytes) {
                    *reinterpret_cast<uint4 *>(kd + off) = kr[u];
                    *reinterpret_cast<uint4 *>(vd + off) = vr[u];
                }
            }
        }
    }
}

// Element path for rows or strides that are not 16-byte multiples.
template <typename E>
__global__ void __launch_bounds__(kCwWarps * 32) cache_write_elem_kernel(
    const E *__restrict__ k_new, const E *__restrict__ v_new, int64_t num_tokens, int64_t src_stride,
    const int64_t *__restrict__ slot_mapping, E *__restrict__ k_cache, E *__restrict__ v_cache, int64_t capacity,
    int64_t row, int32_t *err_count) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (int64_t)blockIdx.x * kCwWarps + (threadIdx.x >> 5);
    const int64_t wstep = (int64_t)gridDim.x * kCwWarps;
    for (int64_t i = warp0; i < num_tokens; i += wstep) {
        const int64_t s = __ldg(slot_mapping + i);
        if (s < 0) continue;
        if (s >= capacity) {
            if (lane == 0 && err_count) atomicAdd(err_count, 1);
            continue;
        }
        for (int64_t e = lane; e < row; e += 32) {
            k_cache[s * row + e] = k_new[i * src_stride + e];
            v_cache[s * row + e] = v_new[i * src_stride + e];
        }
    }
}

// ---------------------------------------------------------------------------
// Slot mapping and cache write in one pass (the composition of
// slot_mapping_kernel and the cache-write kernels above, with the same
// results: the same slot_mapping array, cache bytes and error counts).  One
// warp per token i < max_num_tokens: the lanes read the token's request and
// position, and a real token's source rows are loaded while its table entry
// is (they do not depend on the slot), so a step's slot computation and copy
// cost one chain of memory round trips instead of two dependent launches.
// Lane 0 writes slot_mapping[i] (-1 for the padded tail and padded requests).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kCwWarps * 32) slot_write_vec16_kernel(
    const int32_t *__restrict__ block_table, int32_t num_reqs, int64_t bt_stride, int32_t bt_cols,
    const int32_t *__restrict__ req_indices, const int64_t *__restrict__ positions, int64_t num_tokens,
    int64_t max_num_tokens, int32_t block_size, int64_t *__restrict__ slot_mapping, const char *__restrict__ k_new,
    const char *__restrict__ v_new, int64_t src_stride_bytes, char *__restrict__ k_cache, char *__restrict__ v_cache,
    int64_t capacity, int64_t row_bytes, int32_t *err_count) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (int64_t)blockIdx.x * kCwWarps + (threadIdx.x >> 5);
    const int64_t wstep = (int64_t)gridDim.x * kCwWarps;
    for (int64_t i = warp0; i < max_num_tokens; i += wstep) {
        int32_t r = -1;
        int64_t p = 0;
        if (i < num_tokens) {
            r = __ldg(req_indices + i);
            p = __ldg(positions + i);
        }
        if (r < 0) {   // padded tail or padded request
            if (lane == 0) slot_mapping[i] = -1;
            continue;
        }
        const char *ks = k_new + i * src_stride_bytes;
        const char *vs = v_new + i * src_stride_bytes;
        // the first round of the row (up to 32 x 16 x kCwUnroll bytes) in flight with the table read
        uint4 kr[kCwUnroll], vr[kCwUnroll];
#pragma unroll
        for (int u = 0; u < kCwUnroll; ++u) {
            const int64_t off = (int64_t)lane * 16 + (int64_t)u * 32 * 16;
            if (off < row_bytes) {
                kr[u] = __ldg(reinterpret_cast<const uint4 *>(ks + off));
                vr[u] = __ldg(reinterpret_cast<const uint4 *>(vs + off));
            }
        }
        bool bad;
        const int64_t s = slot_of(block_table, num_reqs, bt_stride, bt_cols, r, p, block_size, 1, 0, 1, &bad);
        if (lane == 0) {
            slot_mapping[i] = s;
            if ((bad || s >= capacity) && err_count) atomicAdd(err_count, 1);
        }
        if (s < 0 || s >= capacity) continue;
        char *kd = k_cache + s * row_bytes;
        char *vd = v_cache + s * row_bytes;
        for (int64_t base = (int64_t)lane * 16;; ) {
#pragma unroll
            for (int u = 0; u < kCwUnroll; ++u) {
                const int64_t off = base + (int64_t)u * 32 * 16;
                if (off < row_bytes) {
                    *reinterpret_cast<uint4 *>(kd + off) = kr[u];
                    *reinterpret_cast<uint4 *>(vd + off) = vr[u];
                }
            }
            base += 32 * 16 * kCwUnroll;
            if (base >= row_bytes) break;
#pragma unroll
            for (int u = 0; u < kCwUnroll; ++u) {
                const int64_t off = base + (int64_t)u * 32 * 16;
                if (off < row_bytes) {
                    kr[u] = __ldg(reinterpret_cast<const uint4 *>(ks + off));
                    vr[u] = __ldg(reinterpret_cast<const uint4 *>(vs + off));
                }
            }
        }
    }
}

// Element path of the fused pass, for rows or strides that are not 16-byte multiples.
template <typename E>
__global__ void __launch_bounds__(kCwWarps * 32) slot_write_elem_kernel(
    const int32_t *__restrict__ block_table, int32_t num_reqs, int64_t bt_stride, int32_t bt_cols,
    const int32_t *__restrict__ req_indices, const int64_t *__restrict__ positions, int64_t num_tokens,
    int64_t max_num_tokens, int32_t block_size, int64_t *__restrict__ slot_mapping, const E *__restrict__ k_new,
    const E *__restrict__ v_new, int64_t src_stride, E *__restrict__ k_cache, E *__restrict__ v_cache,
    int64_t capacity, int64_t row, int32_t *err_count) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (int64_t)blockIdx.x * kCwWarps + (threadIdx.x >> 5);
    const int64_t wstep = (int64_t)gridDim.x * kCwWarps;
    for (int64_t i = warp0; i < max_num_tokens; i += wstep) {
        const int32_t r = i < num_tokens ? __ldg(req_indices + i) : -1;
        if (r < 0) {
            if (lane == 0) slot_mapping[i] = -1;
            continue;
        }
        bool bad;
        const int64_t s = slot_of(block_table, num_reqs, bt_stride, bt_cols, r, __ldg(positions + i), block_size,
                                  1, 0, 1, &bad);
        if (lane == 0) {
            slot_mapping[i] = s;
            if ((bad || s >= capacity) && err_count) atomicAdd(err_count, 1);
        }
        if (s < 0 || s >= capacity) continue;
        for (int64_t e = lane; e < row; e += 32) {
            k_cache[s * row + e] = k_new[i * src_stride + e];
            v_cache[s * row + e] = v_new[i * src_stride + e];
        }
    }
}

// ---------------------------------------------------------------------------
// FP8 (E4M3) cache write.  The pages name a non-FP8 pathway and nothing more
// ("Padding and Batching with Block KV", Block ID 0 vs. Sentinel -1); this
// library's reading: each element x of a new row is stored as the E4M3 code
// of the binary32 quotient x / scale (IEEE division), rounded to nearest even
// with saturation to +-448 and NaN kept NaN, one scale for K and one for V.
// One warp per token as above; each lane turns 16 source elements into one
// 16-byte store.  HBM-bound: row * (2 * src bytes + 2) + 8 bytes per token.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float src_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float src_f(float x) { return x; }

// Two elements to two E4M3 codes (the first in the low byte).
__device__ __forceinline__ uint32_t e4m3x2(float a, float b, float scale) {
    const __nv_fp8x2_storage_t c =
        __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(a, scale), __fdiv_rn(b, scale)), __NV_SATFINITE, __NV_E4M3);
    return (uint32_t)c;
}

// Sixteen consecutive source elements at p (16-byte aligned) as codes.
template <typename E>
__device__ __forceinline__ uint4 quant16(const E *p, float scale) {
    constexpr int kVec = 16 / sizeof(E);   // elements per 16-byte load
    E x[16];
#pragma unroll
    for (int u = 0; u < 16 / kVec; ++u) *reinterpret_cast<uint4 *>(x + u * kVec) = __ldg(reinterpret_cast<const uint4 *>(p) + u);
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        w[q] = e4m3x2(src_f(x[4 * q]), src_f(x[4 * q + 1]), scale) |
               (e4m3x2(src_f(x[4 * q + 2]), src_f(x[4 * q + 3]), scale) << 16);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// One token's K and V rows (`row` source elements each) quantised into their
// cache rows by the 32 lanes of a warp.  kVec16: the row and the source
// stride are multiples of 16 elements and the bases 16-byte aligned, each
// lane turning 16 elements into one 16-byte store; otherwise one element per
// lane and step.
template <typename E, bool kVec16>
__device__ __forceinline__ void quant_rows(const E *ks, const E *vs, uint8_t *kd, uint8_t *vd, int64_t row,
                                           float k_scale, float v_scale, int lane) {
    if constexpr (kVec16) {
        for (int64_t e = (int64_t)lane * 16; e < row; e += 32 * 16) {
            const uint4 kq = quant16(ks + e, k_scale);
            const uint4 vq = quant16(vs + e, v_scale);
            *reinterpret_cast<uint4 *>(kd + e) = kq;
            *reinterpret_cast<uint4 *>(vd + e) = vq;
        }
    } else {
        for (int64_t e = lane; e < row; e += 32) {
            kd[e] = (uint8_t)e4m3x2(src_f(ks[e]), 0.f, k_scale);
            vd[e] = (uint8_t)e4m3x2(src_f(vs[e]), 0.f, v_scale);
        }
    }
}

// The quantising cache write: warps over tokens, slots read from slot_mapping.
template <typename E, bool kVec16>
__global__ void __launch_bounds__(kCwWarps * 32) cache_write_fp8_kernel(
    const E *__restrict__ k_new, const E *__restrict__ v_new, int64_t num_tokens, int64_t src_stride,
    const int64_t *__restrict__ slot_mapping, uint8_t *__restrict__ k_cache, uint8_t *__restrict__ v_cache,
    int64_t capacity, int64_t row, float k_scale, float v_scale, int32_t *err_count) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (int64_t)blockIdx.x * kCwWarps + (threadIdx.x >> 5);
    const int64_t wstep = (int64_t)gridDim.x * kCwWarps;
    for (int64_t i = warp0; i < num_tokens; i += wstep) {
        const int64_t s = __ldg(slot_mapping + i);
        if (s < 0) continue;
        if (s >= capacity) {
            if (lane == 0 && err_count) atomicAdd(err_count, 1);
            continue;
        }
        quant_rows<E, kVec16>(k_new + i * src_stride, v_new + i * src_stride, k_cache + s * row, v_cache + s * row,
                              row, k_scale, v_scale, lane);
    }
}

// Slot mapping and the quantising write in one pass: the composition of
// slot_mapping_kernel and cache_write_fp8_kernel, with the same slots, cache
// bytes and error counts.  One warp per token i < max_num_tokens; lane 0
// writes slot_mapping[i] (-1 for the padded tail and padded requests).
template <typename E, bool kVec16>
__global__ void __launch_bounds__(kCwWarps * 32) slot_write_fp8_kernel(
    const int32_t *__restrict__ block_table, int32_t num_reqs, int64_t bt_stride, int32_t bt_cols,
    const int32_t *__restrict__ req_indices, const int64_t *__restrict__ positions, int64_t num_tokens,
    int64_t max_num_tokens, int32_t block_size, int64_t *__restrict__ slot_mapping, const E *__restrict__ k_new,
    const E *__restrict__ v_new, int64_t src_stride, uint8_t *__restrict__ k_cache, uint8_t *__restrict__ v_cache,
    int64_t capacity, int64_t row, float k_scale, float v_scale, int32_t *err_count) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = (int64_t)blockIdx.x * kCwWarps + (threadIdx.x >> 5);
    const int64_t wstep = (int64_t)gridDim.x * kCwWarps;
    for (int64_t i = warp0; i < max_num_tokens; i += wstep) {
        const int32_t r = i < num_tokens ? __ldg(req_indices + i) : -1;
        if (r < 0) {
            if (lane == 0) slot_mapping[i] = -1;
            continue;
        }
        bool bad;
        const int64_t s = slot_of(block_table, num_reqs, bt_stride, bt_cols, r, __ldg(positions + i), block_size,
                                  1, 0, 1, &bad);
        if (lane == 0) {
            slot_mapping[i] = s;
            if ((bad || s >= capacity) && err_count) atomicAdd(err_count, 1);
        }
        if (s < 0 || s >= capacity) continue;
        quant_rows<E, kVec16>(k_new + i * src_stride, v_new + i * src_stride, k_cache + s * row, v_cache + s * row,
                              row, k_scale, v_scale, lane);
    }
}

}  // namespace bkv

extern "C" int bkv_cache_write_fp8(const void *k_new, const void *v_new, int64_t num_tokens,
                                   int64_t new_token_stride, const int64_t *slot_mapping, uint8_t *k_cache,
                                   uint8_t *v_cache, int64_t total_blocks, int32_t block_size, int32_t num_kv_heads,
                                   int32_t head_dim, int src_dtype, float k_scale, float v_scale,
                                   int32_t *err_count, bkv_stream_t stream) {
    if (src_dtype != BKV_BF16 && src_dtype != BKV_F32) return BKV_ERR_UNSUPPORTED;
    if (num_tokens < 0 || total_blocks < 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return BKV_ERR_INVALID_ARG;
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || !isfinite(k_scale) || !isfinite(v_scale)) return BKV_ERR_INVALID_ARG;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    if (new_token_stride < row) return BKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return BKV_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return BKV_ERR_INVALID_ARG;
    const int64_t capacity = total_blocks * block_size;
    const int threads = bkv::kCwWarps * 32;
    const unsigned grid = bkv::grid_for(num_tokens, bkv::kCwWarps, 16);
    cudaStream_t st = (cudaStream_t)stream;
    const bool vec16 = row % 16 == 0 && new_token_stride % 16 == 0 && bkv::aligned(k_new, 16) &&
                       bkv::aligned(v_new, 16) && bkv::aligned(k_cache, 16) && bkv::aligned(v_cache, 16);
    cudaError_t e;
    if (src_dtype == BKV_BF16) {
        auto kern = vec16 ? bkv::cache_write_fp8_kernel<__nv_bfloat16, true>
                          : bkv::cache_write_fp8_kernel<__nv_bfloat16, false>;
        e = bkv::launch_pdl(kern, grid, threads, 0, st, (const __nv_bfloat16 *)k_new, (const __nv_bfloat16 *)v_new,
                            num_tokens, new_token_stride, slot_mapping, k_cache, v_cache, capacity, row, k_scale,
                            v_scale, err_count);
    } else {
        auto kern = vec16 ? bkv::cache_write_fp8_kernel<float, true> : bkv::cache_write_fp8_kernel<float, false>;
        e = bkv::launch_pdl(kern, grid, threads, 0, st, (const float *)k_new, (const float *)v_new, num_tokens,
                            new_token_stride, slot_mapping, k_cache, v_cache, capacity, row, k_scale, v_scale,
                            err_count);
    }
    if (e != cudaSuccess) bkv::set_cuda_error(e);
    return bkv::launch_status();
}

extern "C" int bkv_cache_write(const void *k_new, const void *v_new, int64_t num_tokens, int64_t new_token_stride,
                               const int64_t *slot_mapping, void *k_cache, void *v_cache, int64_t total_blocks,
                               int32_t block_size, int32_t num_kv_heads, int32_t head_dim, int dtype,
                               int32_t *err_count, bkv_stream_t stream) {
    if (dtype != BKV_BF16 && dtype != BKV_F32) return BKV_ERR_UNSUPPORTED;
    if (num_tokens < 0 || total_blocks < 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return BKV_ERR_INVALID_ARG;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    if (new_token_stride < row) return BKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return BKV_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return BKV_ERR_INVALID_ARG;
    const int64_t eb = dtype == BKV_BF16 ? 2 : 4;
    const int64_t capacity = total_blocks * block_size;
    const int threads = bkv::kCwWarps * 32;
    const unsigned grid = bkv::grid_for(num_tokens, bkv::kCwWarps, 16);
    cudaStream_t st = (cudaStream_t)stream;
    const bool vec16 = (row * eb) % 16 == 0 && (new_token_stride * eb) % 16 == 0 && bkv::aligned(k_new, 16) &&
                       bkv::aligned(v_new, 16) && bkv::aligned(k_cache, 16) && bkv::aligned(v_cache, 16);
    cudaError_t e;
    if (vec16) {
        e = bkv::launch_pdl(bkv::cache_write_vec16_kernel, grid, threads, 0, st, (const char *)k_new,
                            (const char *)v_new, num_tokens, new_token_stride * eb, slot_mapping, (char *)k_cache,
                            (char *)v_cache, capacity, row * eb, err_count);
    } else if (eb == 2) {
        e = bkv::launch_pdl(bkv::cache_write_elem_kernel<uint16_t>, grid, threads, 0, st, (const uint16_t *)k_new,
                            (const uint16_t *)v_new, num_tokens, new_token_stride, slot_mapping, (uint16_t *)k_cache,
                            (uint16_t *)v_cache, capacity, row, err_count);
    } else {
        e = bkv::launch_pdl(bkv::cache_write_elem_kernel<uint32_t>, grid, threads, 0, st, (const uint32_t *)k_new,
                            (const uint32_t *)v_new, num_tokens, new_token_stride, slot_mapping, (uint32_t *)k_cache,
                            (uint32_t *)v_cache, capacity, row, err_count);
    }
    if (e != cudaSuccess) bkv::set_cuda_error(e);
    return bkv::launch_status();
}

extern "C" int bkv_slot_mapping_cache_write(const int32_t *block_table, int32_t num_reqs, int64_t bt_stride,
                                            int32_t bt_cols, const int32_t *req_indices, const int64_t *positions,
                                            int64_t num_tokens, int64_t max_num_tokens, int64_t *slot_mapping,
                                            const void *k_new, const void *v_new, int64_t new_token_stride,
                                            void *k_cache, void *v_cache, int64_t total_blocks, int32_t block_size,
                                            int32_t num_kv_heads, int32_t head_dim, int dtype, int32_t *err_count,
                                            bkv_stream_t stream) {
    if (dtype != BKV_BF16 && dtype != BKV_F32) return BKV_ERR_UNSUPPORTED;
    if (block_size <= 0 || num_tokens < 0 || max_num_tokens < num_tokens || num_reqs < 0 || bt_cols < 0 ||
        bt_stride < bt_cols || total_blocks < 0 || num_kv_heads <= 0 || head_dim <= 0)
        return BKV_ERR_INVALID_ARG;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    if (new_token_stride < row) return BKV_ERR_INVALID_ARG;
    if (max_num_tokens == 0) return BKV_OK;
    if (!slot_mapping) return BKV_ERR_INVALID_ARG;
    if (num_tokens > 0 && (!req_indices || !positions || !k_new || !v_new || !k_cache || !v_cache))
        return BKV_ERR_INVALID_ARG;
    if (num_tokens > 0 && num_reqs > 0 && bt_cols > 0 && !block_table) return BKV_ERR_INVALID_ARG;
    const int64_t eb = dtype == BKV_BF16 ? 2 : 4;
    const int64_t capacity = total_blocks * block_size;
    const int threads = bkv::kCwWarps * 32;
    const unsigned grid = bkv::grid_for(max_num_tokens, bkv::kCwWarps, 16);
    cudaStream_t st = (cudaStream_t)stream;
    const bool vec16 = (row * eb) % 16 == 0 && (new_token_stride * eb) % 16 == 0 && bkv::aligned(k_new, 16) &&
                       bkv::aligned(v_new, 16) && bkv::aligned(k_cache, 16) && bkv::aligned(v_cache, 16);
    cudaError_t e;
    if (vec16) {
        e = bkv::launch_pdl(bkv::slot_write_vec16_kernel, grid, threads, 0, st, block_table, num_reqs, bt_stride,
                            bt_cols, req_indices, positions, num_tokens, max_num_tokens, block_size, slot_mapping,
                            (const char *)k_new, (const char *)v_new, new_token_stride * eb, (char *)k_cache,
                            (char *)v_cache, capacity, row * eb, err_count);
    } else if (eb == 2) {
        e = bkv::launch_pdl(bkv::slot_write_elem_kernel<uint16_t>, grid, threads, 0, st, block_table, num_reqs,
                            bt_stride, bt_cols, req_indices, positions, num_tokens, max_num_tokens, block_size,
                            slot_mapping, (const uint16_t *)k_new, (const uint16_t *)v_new, new_token_stride,
                            (uint16_t *)k_cache, (uint16_t *)v_cache, capacity, row, err_count);
    } else {
        e = bkv::launch_pdl(bkv::slot_write_elem_kernel<uint32_t>, grid, threads, 0, st, block_table, num_reqs,
                            bt_stride, bt_cols, req_indices, positions, num_tokens, max_num_tokens, block_size,
                            slot_mapping, (const uint32_t *)k_new, (const uint32_t *)v_new, new_token_stride,
                            (uint32_t *)k_cache, (uint32_t *)v_cache, capacity, row, err_count);
    }
    if (e != cudaSuccess) bkv::set_cuda_error(e);
    return bkv::launch_status();
}

extern "C" int bkv_slot_mapping_cache_write_fp8(const int32_t *block_table, int32_t num_reqs, int64_t bt_stride,
                                                int32_t bt_cols, const int32_t *req_indices, const int64_t *positions,
                                                int64_t num_tokens, int64_t max_num_tokens, int64_t *slot_mapping,
                                                const void *k_new, const void *v_new, int64_t new_token_stride,
                                                uint8_t *k_cache, uint8_t *v_cache, int64_t total_blocks,
                                                int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                                int src_dtype, float k_scale, float v_scale, int32_t *err_count,
                                                bkv_stream_t stream) {
    if (src_dtype != BKV_BF16 && src_dtype != BKV_F32) return BKV_ERR_UNSUPPORTED;
    if (block_size <= 0 || num_tokens < 0 || max_num_tokens < num_tokens || num_reqs < 0 || bt_cols < 0 ||
        bt_stride < bt_cols || total_blocks < 0 || num_kv_heads <= 0 || head_dim <= 0)
        return BKV_ERR_INVALID_ARG;
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || !isfinite(k_scale) || !isfinite(v_scale)) return BKV_ERR_INVALID_ARG;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    if (new_token_stride < row) return BKV_ERR_INVALID_ARG;
    if (max_num_tokens == 0) return BKV_OK;
    if (!slot_mapping) return BKV_ERR_INVALID_ARG;
    if (num_tokens > 0 && (!req_indices || !positions || !k_new || !v_new || !k_cache || !v_cache))
        return BKV_ERR_INVALID_ARG;
    if (num_tokens > 0 && num_reqs > 0 && bt_cols > 0 && !block_table) return BKV_ERR_INVALID_ARG;
    const int64_t capacity = total_blocks * block_size;
    const int threads = bkv::kCwWarps * 32;
    const unsigned grid = bkv::grid_for(max_num_tokens, bkv::kCwWarps, 16);
    cudaStream_t st = (cudaStream_t)stream;
    const bool vec16 = row % 16 == 0 && new_token_stride % 16 == 0 && bkv::aligned(k_new, 16) &&
                       bkv::aligned(v_new, 16) && bkv::aligned(k_cache, 16) && bkv::aligned(v_cache, 16);
    cudaError_t e;
    if (src_dtype == BKV_BF16) {
        auto kern = vec16 ? bkv::slot_write_fp8_kernel<__nv_bfloat16, true>
                          : bkv::slot_write_fp8_kernel<__nv_bfloat16, false>;
        e = bkv::launch_pdl(kern, grid, threads, 0, st, block_table, num_reqs, bt_stride, bt_cols, req_indices,
                            positions, num_tokens, max_num_tokens, block_size, slot_mapping,
                            (const __nv_bfloat16 *)k_new, (const __nv_bfloat16 *)v_new, new_token_stride, k_cache,
                            v_cache, capacity, row, k_scale, v_scale, err_count);
    } else {
        auto kern = vec16 ? bkv::slot_write_fp8_kernel<float, true> : bkv::slot_write_fp8_kernel<float, false>;
        e = bkv::launch_pdl(kern, grid, threads, 0, st, block_table, num_reqs, bt_stride, bt_cols, req_indices,
                            positions, num_tokens, max_num_tokens, block_size, slot_mapping, (const float *)k_new,
                            (const float *)v_new, new_token_stride, k_cache, v_cache, capacity, row, k_scale, v_scale,
                            err_count);
    }
    if (e != cudaSuccess) bkv::set_cuda_error(e);
    return bkv::launch_status();
}
