// kvcache.cu -- append the K/V of new tokens to a paged KV cache.
//
// The cache stores each sequence's tokens in fixed-size pages reached through a page
// table (inference-kernel-cookbook README, recipe 03 "Paged Attention"); a prefill or a
// decode step appends its new tokens' keys and values before attending (recipe 02 "KV
// Cache"; the "KV-cache append path" on the Kernel-Inference-Engine README's roadmap).
// Token t of sequence b lands at position pos = start_pos[b] + t: page
// page_table[b][pos / 16], slot pos % 16, for every key/value head.  Pure data movement:
// d/8 threads copy one d-element row with 16-byte accesses (d a multiple of 8).
// For an FP8 (E4M3) cache the same scatter converts each element to its e4m3 code under the
// tensor's scale; kv_quantize_fp8 converts a whole bf16 page pool the same way.
#include <cuda_fp8.h>

#include "launch.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kPS = 16;

__global__ void __launch_bounds__(256) kv_append_kernel(const uint4 *__restrict__ k_new,
                                                        const uint4 *__restrict__ v_new, uint4 *k_pages,
                                                        uint4 *v_pages, const int32_t *__restrict__ page_table,
                                                        const int32_t *__restrict__ start_pos, int B, int Hkv,
                                                        int Nnew, int vec_per_row, int max_pages, int num_pages) {
    const long long total = (long long)B * Hkv * Nnew * vec_per_row;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int vec = (int)(e % vec_per_row);
        const long long row = e / vec_per_row;  // (b * Hkv + h) * Nnew + t
        const int t = (int)(row % Nnew);
        const int bh = (int)(row / Nnew);
        const int b = bh / Hkv, h = bh % Hkv;
        const int pos = max(start_pos[b], 0) + t;
        if (pos >= max_pages * kPS) continue;  // past the table's capacity
        const int phys = page_table[(size_t)b * max_pages + pos / kPS];
        if (phys < 0 || phys >= num_pages) continue;
        const size_t dst = (((size_t)phys * Hkv + h) * kPS + (pos % kPS)) * vec_per_row + vec;
        k_pages[dst] = k_new[e];
        v_pages[dst] = v_new[e];
    }
}

// Eight bf16 (one 16-byte vector) -> eight e4m3 codes (8 bytes, element 0 in the low byte):
// code = nearest e4m3 of fp32(x) * inv_scale, ties to even, saturating at +-448.
__device__ __forceinline__ uint2 bf16x8_to_e4m3x8(uint4 v, float inv_scale) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float x0 = __fmul_rn(__uint_as_float(w[i] << 16), inv_scale);
        const float x1 = __fmul_rn(__uint_as_float(w[i] & 0xffff0000u), inv_scale);
        const uint32_t two = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
        out[i >> 1] |= (two & 0xffffu) << (16 * (i & 1));
    }
    return make_uint2(out[0], out[1]);
}

__global__ void __launch_bounds__(256) kv_quantize_fp8_kernel(const uint4 *__restrict__ src, uint2 *__restrict__ dst,
                                                              long long n_vec, float inv_scale) {
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n_vec;
         e += (long long)gridDim.x * blockDim.x)
        dst[e] = bf16x8_to_e4m3x8(src[e], inv_scale);
}

// As kv_append_kernel, for an e4m3 cache: one thread converts 8 elements of a new row.
__global__ void __launch_bounds__(256) kv_append_fp8_kernel(const uint4 *__restrict__ k_new,
                                                            const uint4 *__restrict__ v_new, uint2 *k_pages,
                                                            uint2 *v_pages, float k_inv, float v_inv,
                                                            const int32_t *__restrict__ page_table,
                                                            const int32_t *__restrict__ start_pos, int B, int Hkv,
                                                            int Nnew, int vec_per_row, int max_pages, int num_pages) {
    const long long total = (long long)B * Hkv * Nnew * vec_per_row;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int vec = (int)(e % vec_per_row);
        const long long row = e / vec_per_row;  // (b * Hkv + h) * Nnew + t
        const int t = (int)(row % Nnew);
        const int bh = (int)(row / Nnew);
        const int b = bh / Hkv, h = bh % Hkv;
        const int pos = max(start_pos[b], 0) + t;
        if (pos >= max_pages * kPS) continue;
        const int phys = page_table[(size_t)b * max_pages + pos / kPS];
        if (phys < 0 || phys >= num_pages) continue;
        const size_t dst = (((size_t)phys * Hkv + h) * kPS + (pos % kPS)) * vec_per_row + vec;
        k_pages[dst] = bf16x8_to_e4m3x8(k_new[e], k_inv);
        v_pages[dst] = bf16x8_to_e4m3x8(v_new[e], v_inv);
    }
}

int grid_for(long long work) {
    int sms = 0;
    if (current_sm_count(&sms) != cudaSuccess || sms <= 0) return -1;
    const long long want = (work + 255) / 256;
    return (int)(want < (long long)sms * 16 ? want : (long long)sms * 16);
}

}  // namespace

cudaError_t launch_kv_quantize_fp8(const void *src, void *dst, size_t n, float inv_scale, cudaStream_t stream) {
    const long long n_vec = (long long)(n / 8);
    const int grid = grid_for(n_vec);
    if (grid < 0) return cudaErrorUnknown;
    if (grid == 0) return cudaSuccess;
    kv_quantize_fp8_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4 *>(src), static_cast<uint2 *>(dst), n_vec,
                                                     inv_scale);
    return cudaGetLastError();
}

cudaError_t launch_kv_append_fp8(const void *k_new, const void *v_new, void *k_pages, void *v_pages,
                                 float k_inv_scale, float v_inv_scale, const int32_t *page_table,
                                 const int32_t *start_pos, int B, int Hkv, int Nnew, int d, int max_pages,
                                 int num_pages, cudaStream_t stream) {
    const int vpr = d / 8;
    const int grid = grid_for((long long)B * Hkv * Nnew * vpr);
    if (grid < 0) return cudaErrorUnknown;
    if (grid == 0) return cudaSuccess;
    kv_append_fp8_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new),
                                                   static_cast<uint2 *>(k_pages), static_cast<uint2 *>(v_pages),
                                                   k_inv_scale, v_inv_scale, page_table, start_pos, B, Hkv, Nnew, vpr,
                                                   max_pages, num_pages);
    return cudaGetLastError();
}

cudaError_t launch_kv_append(const void *k_new, const void *v_new, void *k_pages, void *v_pages,
                             const int32_t *page_table, const int32_t *start_pos, int B, int Hkv, int Nnew, int d,
                             int max_pages, int num_pages, cudaStream_t stream) {
    int sms = 0;
    cudaError_t e = current_sm_count(&sms);
    if (e != cudaSuccess) return e;
    const long long total = (long long)B * Hkv * Nnew * (d * 2 / 16);
    const long long want = (total + 255) / 256;
    const int grid = (int)(want < (long long)sms * 16 ? want : (long long)sms * 16);
    if (grid <= 0) return cudaSuccess;
    kv_append_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4 *>(k_new), static_cast<const uint4 *>(v_new),
                                               static_cast<uint4 *>(k_pages), static_cast<uint4 *>(v_pages), page_table,
                                               start_pos, B, Hkv, Nnew, d * 2 / 16, max_pages, num_pages);
    return cudaGetLastError();
}

}  // namespace attn
