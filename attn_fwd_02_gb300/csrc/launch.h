// launch.h -- internal interface between the C ABI (abi.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace attn {

struct PrefillArgs {
    const void *q, *k, *v;
    void *o;
    float *lse;              // may be null
    const int32_t *kv_lens;  // may be null
    int *status;             // device status word [2]
    int B, H, Nq, Nkv, d, causal;
    float scale;
    int Hkv;                 // key/value heads (H for multi-head; H % Hkv == 0)
    // paged mode: k, v are [num_pages, Hkv, 16, d] pages through page_table [B, max_pages];
    // ctx_lens[b] cached tokens, the queries being the last Nq of them; Nkv = capacity
    int paged = 0;
    const int32_t *page_table = nullptr, *ctx_lens = nullptr;
    int max_pages = 0, num_pages = 0;
    // paged mode over an e4m3 cache: k, v hold codes; value = e4m3(code) * k_scale / v_scale
    int kv_fp8 = 0;
    float k_scale = 1.f, v_scale = 1.f;
};

struct DecodeArgs {
    const void *q, *k_pages, *v_pages;
    const int32_t *page_table, *ctx_lens;
    void *o;
    float *lse;  // may be null
    void *workspace;
    int *status;
    int B, H, d, page_size, max_pages, num_pages;
    float scale;
    int Hkv;  // key/value heads of the cache (H for multi-head; H % Hkv == 0)
    // e4m3 cache: pages hold FP8 codes, value = e4m3(code) * k_scale (keys) or * v_scale (values)
    int kv_fp8 = 0;
    float k_scale = 1.f, v_scale = 1.f;
};

struct BwdArgs {
    const void *q, *k, *v, *o, *dout;  // q, o, dout [B,Hq,Nq,d]; k, v [B,Hkv,Nkv,d] (bf16)
    const float *lse;                  // [B,Hq,Nq], natural log, from the forward
    void *dq, *dk, *dv;                // bf16 outputs, shaped like q, k, v
    float *dterm;                      // workspace: the row term D [B,Hq,Nq]
    const int32_t *kv_lens;            // may be null
    int *status;
    int B, Hq, Hkv, Nq, Nkv, d, causal;
    float scale;
};

// Per-device facts looked up once (host-side caches shared by the launchers): the SM count
// of the current device, and a kernel's dynamic shared-memory opt-in (set once per
// function and device; cudaFuncSetAttribute is not free on every call).
cudaError_t current_sm_count(int *sms);
cudaError_t ensure_max_dynamic_smem(const void *kernel, int bytes);

// TMA descriptor of a bf16 [BH, N, D] tensor viewed as 3-D (innermost first) with boxes of
// 64 x box_rows x 1 and the 128-byte swizzle; rows past N read as zeros.
bool encode_qkv_map(CUtensorMap *m, const void *ptr, int BH, int N, int D, int box_rows = 128);
// [rows, page_rows, D] one-byte (e4m3) page blocks, one box of page_rows x 128 bytes per block,
// with the 128-byte swizzle or none; the bytes of a box past D are read as zeros.
bool encode_page_map_u8(CUtensorMap *m, const void *ptr, int rows, int page_rows, int D, bool swizzle = true);

// Encodes the TMA descriptors and launches the prefill kernel.
cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t stream);

// Backward: the row term D, then the dK/dV kernel and the dQ kernel.
cudaError_t launch_bwd(const BwdArgs &a, cudaStream_t stream);
size_t bwd_workspace_bytes(int B, int Hq, int Nq);

// Writes new tokens' K/V into their pages (token t of sequence b goes to position
// start_pos[b] + t).  Positions past the table's capacity are skipped.
cudaError_t launch_kv_append(const void *k_new, const void *v_new, void *k_pages, void *v_pages,
                             const int32_t *page_table, const int32_t *start_pos, int B, int Hkv, int Nnew, int d,
                             int max_pages, int num_pages, cudaStream_t stream);

// FP8 (E4M3) cache conversion: codes = e4m3_rn_satfinite(fp32(x) * inv_scale).
//   kv_quantize_fp8: n contiguous bf16 elements -> n codes (n % 8 == 0).
//   kv_append_fp8: as launch_kv_append, converting each new element on the way into the pages.
cudaError_t launch_kv_quantize_fp8(const void *src, void *dst, size_t n, float inv_scale, cudaStream_t stream);
cudaError_t launch_kv_append_fp8(const void *k_new, const void *v_new, void *k_pages, void *v_pages,
                                 float k_inv_scale, float v_inv_scale, const int32_t *page_table,
                                 const int32_t *start_pos, int B, int Hkv, int Nnew, int d, int max_pages,
                                 int num_pages, cudaStream_t stream);

// Launches the split kernel and the combine kernel.
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream);

// Workspace bytes the decode needs for H query heads over Hkv cache heads (0 if the sizes are
// unsupported).
size_t decode_workspace_bytes(int B, int H, int Hkv, int d, int max_pages, int page_size);

// Same kernels with the chunk partials in the library's static scratch array
// (no workspace from the caller); see decode.cu.
cudaError_t launch_decode_noalloc(const DecodeArgs &a, cudaStream_t stream);
size_t decode_noalloc_scratch_bytes();

// One block that waits on an mbarrier nobody arrives on (exercises the bounded waits).
cudaError_t launch_selftest_wait(int *status, cudaStream_t stream);

// Tokens per split of the paged decode.
constexpr int kDecodeChunkTokens = 512;

}  // namespace attn
