// abi.cu -- the C ABI declared in include/attn_gb300.h: host-side argument
// checks, the device status word, and dispatch to the kernel launchers.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "attn_gb300.h"
#include "launch.h"

#define ATTN_API extern "C" __attribute__((visibility("default")))

namespace {

// Device status word (see sm103_ptx.cuh): [0] flags, [1] first failing site, [2..3] the address
// of this device's host-visible flag.
__device__ __align__(8) int g_status[4];

constexpr int kMaxDevices = 64;
int *g_status_ptr[kMaxDevices];
int g_arch_ok[kMaxDevices];  // 0 unknown, 1 sm_103, -1 other
std::mutex g_mu;

// Host-visible timeout flags, one per device (16 ints apart), in one page of the library's own
// static storage that is page-locked and mapped for the GPUs once per process.  A kernel whose
// bounded wait runs out stores 1 into its device's flag (and fences), so the host can see the
// timeout with a plain load, without synchronising any stream.
alignas(4096) volatile int g_host_flags[kMaxDevices * 16];
int g_host_flags_registered = 0;  // 0 not yet, 1 registered, -1 failed

int *host_flag_of(int dev) { return const_cast<int *>(&g_host_flags[dev * 16]); }

// Per-device set-up, done once per device by the first call on it (with the device current):
// architecture check, the status word's device address, registration of the flag page, and a
// copy of the flag's device-side address into the status word.  The copy is synchronous, so the
// first call on each device should come before any stream capture.
int device_setup_locked(int dev) {
    if (g_arch_ok[dev] == 0) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return ATTN_ERR_CUDA;
        g_arch_ok[dev] = (prop.major == 10 && prop.minor == 3) ? 1 : -1;
    }
    if (g_arch_ok[dev] != 1) return ATTN_ERR_UNSUPPORTED;
    if (g_status_ptr[dev]) return ATTN_OK;
    if (g_host_flags_registered == 0) {
        const cudaError_t e = cudaHostRegister(const_cast<int *>(g_host_flags), sizeof(g_host_flags),
                                               cudaHostRegisterMapped | cudaHostRegisterPortable);
        g_host_flags_registered = (e == cudaSuccess) ? 1 : -1;
    }
    if (g_host_flags_registered != 1) return ATTN_ERR_CUDA;
    void *flag_dev = nullptr;
    if (cudaHostGetDevicePointer(&flag_dev, host_flag_of(dev), 0) != cudaSuccess || !flag_dev) return ATTN_ERR_CUDA;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess || !p) return ATTN_ERR_CUDA;
    int init[4] = {0, 0, 0, 0};
    static_assert(sizeof(void *) == 2 * sizeof(int), "64-bit device addresses");
    memcpy(&init[2], &flag_dev, sizeof flag_dev);
    if (cudaMemcpy(p, init, sizeof init, cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
    *host_flag_of(dev) = 0;
    g_status_ptr[dev] = static_cast<int *>(p);
    return ATTN_OK;
}

int current_device(int *dev) {
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) return ATTN_ERR_CUDA;
    return ATTN_OK;
}

// Set-up for a call that launches work: also refuses (ATTN_ERR_DEVICE_TIMEOUT, nothing
// launched) while a timeout recorded by an earlier call on this device is not yet cleared.
int device_setup(int **status_out) {
    int dev = -1;
    if (current_device(&dev) != ATTN_OK) return ATTN_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        const int st = device_setup_locked(dev);
        if (st != ATTN_OK) return st;
    }
    if (*host_flag_of(dev) != 0) return ATTN_ERR_DEVICE_TIMEOUT;
    *status_out = g_status_ptr[dev];
    return ATTN_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Head dims of the prefill kernels (forward, paged prefill, KV append): the set the
// Kernel-Inference-Engine README instantiates its attention kernel for.  Decode and the
// backward take 64 and 128.
bool prefill_head_dim(int d) { return d == 32 || d == 64 || d == 80 || d == 96 || d == 128; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int prefill_checks(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int Hkv,
                   int Nq, int Nkv, int d, int causal, float scale, const int32_t *kv_lens) {
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || Nq <= 0 || Nkv <= 0 || d <= 0) return ATTN_ERR_INVALID_ARG;
    if (Hkv <= 0 || H % Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !(scale < 3.0e38f)) return ATTN_ERR_INVALID_ARG;  // finite, positive
    if (!prefill_head_dim(d)) return ATTN_ERR_UNSUPPORTED;
    // grid = ceil(Nq/128) * B * H CTAs and 32-bit TMA coordinates
    const uint64_t bh = (uint64_t)B * (uint64_t)H;
    const uint64_t ctas = ((uint64_t)Nq + 127) / 128 * bh;
    if (bh > (1ull << 31) - 1 || ctas > (1ull << 31) - 1) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_MISALIGNED;
    if ((lse && !aligned4(lse)) || (kv_lens && !aligned4(kv_lens))) return ATTN_ERR_MISALIGNED;
    return ATTN_OK;
}

}  // namespace

namespace attn {

cudaError_t current_sm_count(int *sms) {
    static int cache[kMaxDevices];  // 0 = unknown
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (cache[dev] == 0) {
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        cache[dev] = n;
    }
    *sms = cache[dev];
    return cudaSuccess;
}

cudaError_t ensure_max_dynamic_smem(const void *kernel, int bytes) {
    struct Entry {
        const void *fn;
        int dev;
        int bytes;
    };
    static Entry done[256];
    static int n_done = 0;
    static std::mutex mu;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < n_done; ++i)
        if (done[i].fn == kernel && done[i].dev == dev && done[i].bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    if (n_done < 256) done[n_done++] = Entry{kernel, dev, bytes};
    return cudaSuccess;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// [BH, N, D] bf16 viewed as a 3-D tensor (innermost first), boxes of 64 x 128 x 1, 128-byte swizzle.
bool encode_qkv_map(CUtensorMap *m, const void *ptr, int BH, int N, int D, int box_rows) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_page_map_u8(CUtensorMap *m, const void *ptr, int rows, int page_rows, int D, bool swizzle) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)page_rows, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D, (cuuint64_t)page_rows * D};
    cuuint32_t box[3] = {128, (cuuint32_t)page_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace attn

ATTN_API int attn_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
                          int Hkv, int Nq, int Nkv, int d, int causal, float scale, const int32_t *kv_lens,
                          attn_stream_t stream) {
    int st = prefill_checks(q, k, v, o, lse, B, Hq, Hkv, Nq, Nkv, d, causal, scale, kv_lens);
    if (st != ATTN_OK) return st;
    int *status = nullptr;
    st = device_setup(&status);
    if (st != ATTN_OK) return st;
    attn::PrefillArgs a{q, k, v, o, lse, kv_lens, status, B, Hq, Nq, Nkv, d, causal, scale, Hkv};
    cudaError_t e = attn::launch_prefill(a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

ATTN_API int attn_fwd_kvlen(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H,
                            int Nq, int Nkv, int d, int causal, float scale, const int32_t *kv_lens,
                            attn_stream_t stream) {
    return attn_fwd_gqa(q, k, v, o, lse, B, H, H, Nq, Nkv, d, causal, scale, kv_lens, stream);
}

ATTN_API int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int Nq,
                      int Nkv, int d, int causal, float scale, attn_stream_t stream) {
    return attn_fwd_kvlen(q, k, v, o, lse, B, H, Nq, Nkv, d, causal, scale, nullptr, stream);
}

ATTN_API size_t attn_bwd_workspace_size(int B, int Hq, int Nq) { return attn::bwd_workspace_bytes(B, Hq, Nq); }

ATTN_API int attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse, const void *dout,
                      void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int Nq, int Nkv, int d, int causal,
                      float scale, const int32_t *kv_lens, void *workspace, size_t workspace_bytes,
                      attn_stream_t stream) {
    if (!o || !lse || !dout || !dk || !dv) return ATTN_ERR_INVALID_ARG;
    // q, k, v, dq and the sizes get the forward's checks (dq in the place of o)
    int st = prefill_checks(q, k, v, dq, nullptr, B, Hq, Hkv, Nq, Nkv, d, causal, scale, kv_lens);
    if (st != ATTN_OK) return st;
    if (d != 32 && d != 64 && d != 80 && d != 96 && d != 128) return ATTN_ERR_UNSUPPORTED;
    const uint64_t kv_ctas = ((uint64_t)Nkv + 127) / 128 * (uint64_t)B * (uint64_t)Hkv;
    if (kv_ctas > (1ull << 31) - 1) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(o) || !aligned16(dout) || !aligned16(dk) || !aligned16(dv) || !aligned4(lse))
        return ATTN_ERR_MISALIGNED;
    const size_t need = attn::bwd_workspace_bytes(B, Hq, Nq);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
    int *status = nullptr;
    st = device_setup(&status);
    if (st != ATTN_OK) return st;
    attn::BwdArgs a{q,  k,  v,      o, dout, lse, dq, dk, dv, static_cast<float *>(workspace), kv_lens, status,
                    B,  Hq, Hkv, Nq, Nkv, d, causal, scale};
    cudaError_t e = attn::launch_bwd(a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

ATTN_API int paged_attn_prefill(const void *q, const void *k_pages, const void *v_pages, const int32_t *page_table,
                                const int32_t *ctx_lens, int page_size, void *o, float *lse, int B, int H, int Hkv,
                                int Nq, int d, int max_pages_per_seq, int num_pages, int causal, float scale,
                                attn_stream_t stream) {
    if (!page_table || !ctx_lens || !k_pages || !v_pages) return ATTN_ERR_INVALID_ARG;
    if (page_size <= 0 || max_pages_per_seq <= 0 || num_pages <= 0) return ATTN_ERR_INVALID_ARG;
    if (page_size != 16) return ATTN_ERR_UNSUPPORTED;
    if ((uint64_t)max_pages_per_seq * 16 > (1ull << 30)) return ATTN_ERR_INVALID_ARG;
    if (Hkv <= 0 || (uint64_t)num_pages * (uint64_t)Hkv > (1ull << 31) - 1) return ATTN_ERR_INVALID_ARG;
    const int cap = max_pages_per_seq * 16;
    int st = prefill_checks(q, k_pages, v_pages, o, lse, B, H, Hkv, Nq, cap, d, causal, scale, nullptr);
    if (st != ATTN_OK) return st;
    if (!aligned4(page_table) || !aligned4(ctx_lens)) return ATTN_ERR_MISALIGNED;
    int *status = nullptr;
    st = device_setup(&status);
    if (st != ATTN_OK) return st;
    attn::PrefillArgs a{q, k_pages, v_pages, o, lse, nullptr, status, B, H, Nq, cap, d, causal, scale, Hkv};
    a.paged = 1;
    a.page_table = page_table;
    a.ctx_lens = ctx_lens;
    a.max_pages = max_pages_per_seq;
    a.num_pages = num_pages;
    cudaError_t e = attn::launch_prefill(a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

ATTN_API int paged_attn_prefill_fp8(const void *q, const void *k_pages, const void *v_pages, float k_scale,
                                    float v_scale, const int32_t *page_table, const int32_t *ctx_lens, int page_size,
                                    void *o, float *lse, int B, int H, int Hkv, int Nq, int d, int max_pages_per_seq,
                                    int num_pages, int causal, float scale, attn_stream_t stream) {
    if (!page_table || !ctx_lens || !k_pages || !v_pages) return ATTN_ERR_INVALID_ARG;
    if (page_size <= 0 || max_pages_per_seq <= 0 || num_pages <= 0) return ATTN_ERR_INVALID_ARG;
    if (!(k_scale > 0.f) || !(k_scale < 3.0e38f) || !(v_scale > 0.f) || !(v_scale < 3.0e38f))
        return ATTN_ERR_INVALID_ARG;
    if (page_size != 16) return ATTN_ERR_UNSUPPORTED;
    if ((uint64_t)max_pages_per_seq * 16 > (1ull << 30)) return ATTN_ERR_INVALID_ARG;
    if (Hkv <= 0 || (uint64_t)num_pages * (uint64_t)Hkv > (1ull << 31) - 1) return ATTN_ERR_INVALID_ARG;
    const int cap = max_pages_per_seq * 16;
    int st = prefill_checks(q, k_pages, v_pages, o, lse, B, H, Hkv, Nq, cap, d, causal, scale, nullptr);
    if (st != ATTN_OK) return st;
    if (!aligned4(page_table) || !aligned4(ctx_lens)) return ATTN_ERR_MISALIGNED;
    int *status = nullptr;
    st = device_setup(&status);
    if (st != ATTN_OK) return st;
    attn::PrefillArgs a{q, k_pages, v_pages, o, lse, nullptr, status, B, H, Nq, cap, d, causal, scale, Hkv};
    a.paged = 1;
    a.page_table = page_table;
    a.ctx_lens = ctx_lens;
    a.max_pages = max_pages_per_seq;
    a.num_pages = num_pages;
    a.kv_fp8 = 1;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    cudaError_t e = attn::launch_prefill(a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

ATTN_API int paged_kv_append(const void *k_new, const void *v_new, void *k_pages, void *v_pages,
                             const int32_t *page_table, const int32_t *start_pos, int page_size, int B, int Hkv,
                             int Nnew, int d, int max_pages_per_seq, int num_pages, attn_stream_t stream) {
    if (!k_new || !v_new || !k_pages || !v_pages || !page_table || !start_pos) return ATTN_ERR_INVALID_ARG;
    if (B <= 0 || Hkv <= 0 || Nnew <= 0 || d <= 0 || page_size <= 0 || max_pages_per_seq <= 0 || num_pages <= 0)
        return ATTN_ERR_INVALID_ARG;
    if (!prefill_head_dim(d)) return ATTN_ERR_UNSUPPORTED;
    if (page_size != 16) return ATTN_ERR_UNSUPPORTED;
    if ((uint64_t)max_pages_per_seq * 16 > (1ull << 30)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pages) || !aligned16(v_pages))
        return ATTN_ERR_MISALIGNED;
    if (!aligned4(page_table) || !aligned4(start_pos)) return ATTN_ERR_MISALIGNED;
    int *status = nullptr;
    int st = device_setup(&status);
    if (st != ATTN_OK) return st;
    cudaError_t e = attn::launch_kv_append(k_new, v_new, k_pages, v_pages, page_table, start_pos, B, Hkv, Nnew, d,
                                           max_pages_per_seq, num_pages, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

ATTN_API size_t paged_attn_decode_workspace_size(int B, int H, int d, int max_pages_per_seq, int page_size) {
    return attn::decode_workspace_bytes(B, H, H, d, max_pages_per_seq, page_size);
}

ATTN_API size_t paged_attn_decode_workspace_size_ctx(int B, int H, int d, int max_ctx_len) {
    if (max_ctx_len <= 0) return 0;
    return attn::decode_workspace_bytes(B, H, H, d, (int)(((int64_t)max_ctx_len + 15) / 16), 16);
}

ATTN_API size_t paged_attn_decode_gqa_workspace_size(int B, int H, int Hkv, int d, int max_pages_per_seq,
                                                     int page_size) {
    return attn::decode_workspace_bytes(B, H, Hkv, d, max_pages_per_seq, page_size);
}

namespace {
bool finite_positive(float x) { return x > 0.f && x < 3.0e38f; }
// Head dims of the decode kernels: the same five as the prefill.
bool decode_head_dim(int d) { return prefill_head_dim(d); }

// Checks shared by every decode entry point: everything but the caller's workspace.
int decode_arg_checks(const void *q, const void *k_pages, const void *v_pages, const int32_t *page_table,
                      const int32_t *ctx_lens, int page_size, void *o, float *lse, int B, int H, int Hkv, int d,
                      int max_pages_per_seq, int num_pages, float scale) {
    if (!q || !k_pages || !v_pages || !page_table || !ctx_lens || !o) return ATTN_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || d <= 0 || page_size <= 0 || max_pages_per_seq <= 0 || num_pages <= 0)
        return ATTN_ERR_INVALID_ARG;
    if (Hkv <= 0 || H % Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if ((uint64_t)num_pages * (uint64_t)Hkv > (1ull << 31) - 1) return ATTN_ERR_INVALID_ARG;  // TMA rows
    if (!finite_positive(scale)) return ATTN_ERR_INVALID_ARG;
    if (!decode_head_dim(d)) return ATTN_ERR_UNSUPPORTED;
    if (page_size != 16) return ATTN_ERR_UNSUPPORTED;
    if (B > 65535 || H > 65535) return ATTN_ERR_INVALID_ARG;  // grid y/z limits
    if ((uint64_t)max_pages_per_seq * (uint64_t)page_size > (1ull << 30)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o)) return ATTN_ERR_MISALIGNED;
    if (!aligned4(page_table) || !aligned4(ctx_lens) || (lse && !aligned4(lse))) return ATTN_ERR_MISALIGNED;
    return ATTN_OK;
}

int decode_checks(const void *q, const void *k_pages, const void *v_pages, const int32_t *page_table,
                  const int32_t *ctx_lens, int page_size, void *o, float *lse, int B, int H, int Hkv, int d,
                  int max_pages_per_seq, int num_pages, float scale, void *workspace, size_t workspace_bytes) {
    const int st = decode_arg_checks(q, k_pages, v_pages, page_table, ctx_lens, page_size, o, lse, B, H, Hkv, d,
                                     max_pages_per_seq, num_pages, scale);
    if (st != ATTN_OK) return st;
    const size_t need = attn::decode_workspace_bytes(B, H, Hkv, d, max_pages_per_seq, page_size);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
    return ATTN_OK;
}
}  // namespace

ATTN_API int paged_attn_decode_fp8(const void *q, const void *k_pages, const void *v_pages, float k_scale,
                                   float v_scale, const int32_t *page_table, const int32_t *ctx_lens, int page_size,
                                   void *o, float *lse, int B, int H, int Hkv, int d, int max_pages_per_seq,
                                   int num_pages, float scale, void *workspace, size_t workspace_bytes,
                                   attn_stream_t stream) {
    int st = decode_checks(q, k_pages, v_pages, page_table, ctx_lens, page_size, o, lse, B, H, Hkv, d,
                           max_pages_per_seq, num_pages, scale, workspace, workspace_bytes);
    if (st != ATTN_OK) return st;
    if (!finite_positive(k_scale) || !finite_positive(v_scale)) return ATTN_ERR_INVALID_ARG;
    int *status = nullptr;
    st = device_setup(&status);
    if (st != ATTN_OK) return st;
    attn::DecodeArgs a{q,  k_pages, v_pages, page_table, ctx_lens, o, lse, workspace, status, B, H, d, page_size,
                       max_pages_per_seq, num_pages, scale, Hkv};
    a.kv_fp8 = 1;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    cudaError_t e = attn::launch_decode(a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

ATTN_API int kv_quantize_fp8(const void *src, void *dst, size_t n, float scale, attn_stream_t stream) {
    if (!src || !dst || n == 0 || n % 8 != 0 || n > (1ull << 40)) return ATTN_ERR_INVALID_ARG;
    if (!finite_positive(scale)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(dst)) return ATTN_ERR_MISALIGNED;
    int *status = nullptr;
    int st = device_setup(&status);
    if (st != ATTN_OK) return st;
    cudaError_t e = attn::launch_kv_quantize_fp8(src, dst, n, 1.0f / scale, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

ATTN_API int paged_kv_append_fp8(const void *k_new, const void *v_new, void *k_pages, void *v_pages, float k_scale,
                                 float v_scale, const int32_t *page_table, const int32_t *start_pos, int page_size,
                                 int B, int Hkv, int Nnew, int d, int max_pages_per_seq, int num_pages,
                                 attn_stream_t stream) {
    if (!k_new || !v_new || !k_pages || !v_pages || !page_table || !start_pos) return ATTN_ERR_INVALID_ARG;
    if (B <= 0 || Hkv <= 0 || Nnew <= 0 || d <= 0 || page_size <= 0 || max_pages_per_seq <= 0 || num_pages <= 0)
        return ATTN_ERR_INVALID_ARG;
    if (!finite_positive(k_scale) || !finite_positive(v_scale)) return ATTN_ERR_INVALID_ARG;
    if (!prefill_head_dim(d)) return ATTN_ERR_UNSUPPORTED;
    if (page_size != 16) return ATTN_ERR_UNSUPPORTED;
    if ((uint64_t)max_pages_per_seq * 16 > (1ull << 30)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pages) || !aligned16(v_pages))
        return ATTN_ERR_MISALIGNED;
    if (!aligned4(page_table) || !aligned4(start_pos)) return ATTN_ERR_MISALIGNED;
    int *status = nullptr;
    int st = device_setup(&status);
    if (st != ATTN_OK) return st;
    cudaError_t e = attn::launch_kv_append_fp8(k_new, v_new, k_pages, v_pages, 1.0f / k_scale, 1.0f / v_scale,
                                               page_table, start_pos, B, Hkv, Nnew, d, max_pages_per_seq, num_pages,
                                               reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

ATTN_API int paged_attn_decode_gqa(const void *q, const void *k_pages, const void *v_pages,
                                   const int32_t *page_table, const int32_t *ctx_lens, int page_size, void *o,
                                   float *lse, int B, int H, int Hkv, int d, int max_pages_per_seq, int num_pages,
                                   float scale, void *workspace, size_t workspace_bytes, attn_stream_t stream) {
    int st = decode_checks(q, k_pages, v_pages, page_table, ctx_lens, page_size, o, lse, B, H, Hkv, d,
                           max_pages_per_seq, num_pages, scale, workspace, workspace_bytes);
    if (st != ATTN_OK) return st;
    int *status = nullptr;
    st = device_setup(&status);
    if (st != ATTN_OK) return st;
    attn::DecodeArgs a{q,  k_pages, v_pages, page_table, ctx_lens, o, lse, workspace, status, B, H, d, page_size,
                       max_pages_per_seq, num_pages, scale, Hkv};
    cudaError_t e = attn::launch_decode(a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

ATTN_API int paged_attn_decode(const void *q, const void *k_pages, const void *v_pages, const int32_t *page_table,
                               const int32_t *ctx_lens, int page_size, void *o, float *lse, int B, int H, int d,
                               int max_pages_per_seq, int num_pages, float scale, void *workspace,
                               size_t workspace_bytes, attn_stream_t stream) {
    return paged_attn_decode_gqa(q, k_pages, v_pages, page_table, ctx_lens, page_size, o, lse, B, H, H, d,
                                 max_pages_per_seq, num_pages, scale, workspace, workspace_bytes, stream);
}

// Decode with the chunk partials in the library's static scratch array (decode.cu);
// for callers that cannot allocate device memory.  Same checks as paged_attn_decode
// minus the workspace, plus the scratch capacity.
ATTN_API int paged_attn_decode_noalloc(const void *q, const void *k_pages, const void *v_pages,
                                       const int32_t *page_table, const int32_t *ctx_lens, int page_size, void *o,
                                       float *lse, int B, int H, int d, int max_pages_per_seq, int num_pages,
                                       float scale, attn_stream_t stream) {
    int st = decode_arg_checks(q, k_pages, v_pages, page_table, ctx_lens, page_size, o, lse, B, H, H, d,
                               max_pages_per_seq, num_pages, scale);
    if (st != ATTN_OK) return st;
    const size_t need = attn::decode_workspace_bytes(B, H, H, d, max_pages_per_seq, page_size);
    if (need == 0 || need > attn::decode_noalloc_scratch_bytes()) return ATTN_ERR_SCRATCH_LIMIT;
    int *status = nullptr;
    st = device_setup(&status);
    if (st != ATTN_OK) return st;
    attn::DecodeArgs a{q,  k_pages, v_pages, page_table, ctx_lens, o, lse, nullptr, status, B, H, d, page_size,
                       max_pages_per_seq, num_pages, scale, H};
    cudaError_t e = attn::launch_decode_noalloc(a, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

ATTN_API int attn_selftest_bounded_wait(attn_stream_t stream) {
    int *status = nullptr;
    int st = device_setup(&status);
    if (st != ATTN_OK) return st;
    return attn::launch_selftest_wait(status, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK
                                                                                                     : ATTN_ERR_CUDA;
}

ATTN_API int attn_check_device_status(attn_stream_t stream) {
    int dev = -1;
    if (current_device(&dev) != ATTN_OK) return ATTN_ERR_CUDA;
    int *status = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        const int st = device_setup_locked(dev);
        if (st != ATTN_OK) return st;
        status = g_status_ptr[dev];
    }
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    int h[2] = {0, 0};
    if (cudaMemcpy(h, status, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
    const bool timed_out = h[0] != 0 || *host_flag_of(dev) != 0;
    if (!timed_out) return ATTN_OK;
    const int zero[2] = {0, 0};  // flags and site; the flag address in [2..3] stays
    if (cudaMemcpy(status, zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
    *host_flag_of(dev) = 0;
    return ATTN_ERR_DEVICE_TIMEOUT;
}

ATTN_API int attn_last_device_status(void) {
    int dev = -1;
    if (current_device(&dev) != ATTN_OK) return ATTN_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        const int st = device_setup_locked(dev);
        if (st != ATTN_OK) return st;
    }
    return *host_flag_of(dev) != 0 ? ATTN_ERR_DEVICE_TIMEOUT : ATTN_OK;
}

ATTN_API const char *attn_status_string(int status) {
    switch (status) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID_ARG: return "invalid argument (null pointer, non-positive or oversized dimension, bad scale)";
        case ATTN_ERR_UNSUPPORTED: return "unsupported (head dim 32, 64, 80, 96 or 128; 64 or 128 for the backward; page size 16; device sm_103)";
        case ATTN_ERR_MISALIGNED: return "misaligned pointer (tensors need 16-byte alignment)";
        case ATTN_ERR_WORKSPACE: return "workspace missing, misaligned or smaller than paged_attn_decode_workspace_size() (decode) or attn_bwd_workspace_size() (backward)";
        case ATTN_ERR_CUDA: return "CUDA runtime error or launch failure";
        case ATTN_ERR_DEVICE_TIMEOUT: return "a bounded in-kernel wait ran out; results of the affected calls are invalid, and calls launch nothing until attn_check_device_status() clears it";
        case ATTN_ERR_SCRATCH_LIMIT: return "sizes need more decode scratch than the 12 MiB static array of paged_attn_decode_noalloc (use paged_attn_decode with a workspace)";
        default: return "unknown status";
    }
}

ATTN_API const char *attn_version(void) { return "0.1.0"; }
