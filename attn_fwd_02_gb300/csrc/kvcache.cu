// kvcache.cu -- append the K/V of new tokens to a paged KV cache.
//
// The cache stores each sequence's tokens in fixed-size pages reached through a page
// table (inference-kernel-cookbook README, recipe 03 "Paged Attention"); a prefill or a
// decode step appends its new tokens' keys and values before attending (recipe 02 "KV
// Cache"; the "KV-cache append path" on the Kernel-Inference-Engine README's roadmap).
// Token t of sequence b lands at position pos = start_pos[b] + t: page
// page_table[b][pos / 16], slot pos % 16, for every key/value head.  Pure data movement:
// d/8 threads copy one d-element row with 16-byte accesses (d a multiple of 8).
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

}  // namespace

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
