// decode.cu -- paged-KV decode attention for sm_103a.
//
// One query token per sequence attends over its ctx_len cached tokens, which
// live in fixed-size pages reached through a page table (inference-kernel-
// cookbook README, recipe 03 "Paged Attention": scattered physical pages, same
// result as a contiguous cache).  The work is HBM-bound: every cached K/V byte
// is read once and used for two FMAs.
//
// Pass 1 (decode_split_kernel): grid (splits, H, B).  A CTA owns one chunk of
// tokens (512 at d = 128, 1024 at smaller d) of one (sequence, head).  Each of its 4 warps owns
// every 4th page of the chunk and streams those pages through a private ring of
// shared-memory slots with cp.async.bulk (one 1-D bulk copy per page per K/V:
// a page of one head is a contiguous page_size x d block), so each SM keeps
// tens of KB of page data in flight.  A warp keeps an online-softmax state
// (running max m, normaliser l, unnormalised O) in the log2 domain; the four
// warp states merge in shared memory and the CTA writes its partial (m, l, O)
// to the workspace.  Grouped-query heads (and multi-head attention at the head dims where it
// measured faster) run pass 1 on the tensor cores instead (decode_gqa_mma_kernel): the group's
// query heads are the M rows of mma.sync products over each page, whose K/V blocks arrive by TMA in
// swizzled boxes.
//
// Pass 2 (decode_combine_kernel): per (sequence, head), the partials of all
// chunks merge with weights 2^(m_s - M):  L = sum l_s 2^(m_s-M),
// O = sum O_s 2^(m_s-M) / L, LSE = ln2 * (M + log2 L).
//
// The cache holds bf16 values, or FP8 E4M3 codes with one scale per tensor (value =
// e4m3 * scale; the FP8 e4m3 storage on the NanoInfer README's roadmap), which halves the
// bytes a decode step reads.  The key scale folds into the query's score scale and the value
// scale into the partial O, so the inner loops only widen codes (to fp32 in the scalar kernel, to
// f16 in the tensor-core one).

#include <mutex>

#include "launch.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kWarps = 4;

// Programmatic dependent launch: the chunk merge is launched while the split kernel drains.
// Each split CTA signals once its partial is written (launch_dependents); the merge's blocks
// wait for the split grid's completion, with its memory visible, before reading (wait).
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Ring slots per warp: 3 page blocks for a bf16 cache and one query head per CTA (4 KB each at
// d = 128: 96 KB per CTA, 2 CTAs per SM); 2 when the arithmetic per byte is higher -- an e4m3
// cache (half the bytes per token; 2 KB blocks, 32 KB per CTA, 7 CTAs per SM) or several query
// heads per CTA (grouped-query) -- where extra warps help more than bytes in flight per warp.
// Measured: e4m3 2 slots > 1 > 3 > 4 > 6; grouped-query bf16 2 slots 4.50 TB/s, 3 or 1 slots
// 3.94 TB/s.
template <bool FP8, int GP> constexpr int kSlotsFor = (FP8 || GP > 1) ? 2 : 3;
constexpr int kPS = 16;    // page size (tokens)
// Tokens per split of the grouped-query kernel: twice the multi-head chunk, so each CTA's start
// (page-table read, first page loads) is spread over 16 pages per warp.  Measured on 32 sequences
// x 8 key/value heads (4 query heads each), contexts U[512, 8192]: 512 tokens 5.84-5.90 TB/s,
// 1024 5.97, 2048 5.78-5.81 (too few CTAs for an even last wave).
constexpr int kGqaChunkTokens = 2 * kDecodeChunkTokens;
// Tokens per split of the multi-head kernel by head dim: kDecodeChunkTokens at d = 128, 1024 at
// smaller d, so that each CTA streams more bytes and its start (page-table read, first loads) is
// spread over more of them.  Measured on 32 sequences x 32 heads, contexts U[512, 8192] (fraction
// of HBM at 512 / 1024 / 2048 tokens): d = 32 0.754 / 0.749 / 0.704, d = 64 0.941 / 0.948 / 0.926,
// d = 80 0.845 / 0.881 / 0.879, d = 96 0.988 / 0.993 / 0.988.  At most 32 pages per warp (one id
// per lane).
constexpr int mha_chunk_tokens(int d) { return d >= 128 ? kDecodeChunkTokens : 1024; }
static_assert(1024 <= 32 * 4 * 16 && kGqaChunkTokens <= 32 * 4 * 16, "one page id per lane");
// Tokens per split for H query heads over Hkv cache heads: groups of two or more query heads run
// the grouped-query kernel and its 1024-token splits.
constexpr int decode_chunk_tokens(int H, int Hkv, int d) {
    return (H / Hkv) % 2 == 0 ? kGqaChunkTokens : mha_chunk_tokens(d);
}
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// 64-column boxes of a page block in the grouped-query kernel's swizzled layout (the columns past
// D of the last box are read as zeros by TMA and never used by the products).
template <int D> constexpr int kBoxes = (D + 63) / 64;
// Bytes of one ring buffer (one page block of K or V): the scalar kernel's bulk-copied block (kPS
// rows of D elements), or the tensor-core kernel's swizzled TMA boxes: kBoxes boxes of 16 x 64
// bf16, or one box of 16 x 128 e4m3 codes.
template <int D, bool FP8> constexpr int kSlotBytes = kPS * D * (FP8 ? 1 : 2);
template <int D, bool FP8> constexpr int kBoxSlotBytes = FP8 ? kPS * 128 : kBoxes<D> * kPS * 128;

template <int D, int GP, bool FP8>
struct DecodeSmem {
    // [warp][slot][0 = K, 1 = V][one page block]; 16-byte aligned blocks
    alignas(128) uint8_t kv[kWarps][kSlotsFor<FP8, GP>][2][kSlotBytes<D, FP8>];
    uint64_t full[kWarps][kSlotsFor<FP8, GP>];
    float red_o[kWarps][GP][D];
    float red_m[kWarps][GP];
    float red_l[kWarps][GP];
    int abort_flag;
};

template <int D>
__host__ __device__ constexpr int ws_stride() {
    return D + 4;  // floats per partial: O[D], m, l, pad (keeps 16-byte alignment)
}

__device__ __forceinline__ float warp_max_pairs(float x) {
    // lanes 2t and 2t+1 hold the same value; reduce over the 16 distinct values
    x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
    x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
    x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 8));
    x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 16));
    return x;
}
__device__ __forceinline__ float warp_sum_pairs(float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    x += __shfl_xor_sync(0xffffffffu, x, 4);
    x += __shfl_xor_sync(0xffffffffu, x, 8);
    x += __shfl_xor_sync(0xffffffffu, x, 16);
    return x;
}

// How the 32 lanes of a warp share the D dims of a row in the multi-head kernel.
//   D = 32, 64, 128: lane l holds DPL = D / 32 consecutive dims from l * DPL (one 2-, 4- or 8-byte
//                    load of bf16);
//   D = 80, 96:      lane l holds the pair 2l, 2l + 1 and, if 64 + l < D, dim 64 + l (DPL = 3: a
//                    4-byte and a 2-byte load); the single slot of lanes 16-31 at D = 80 holds no
//                    dim and stays zero.
template <int D>
struct LaneDims {
    static constexpr bool kSplit = (D % 32 != 0) || (D / 32 == 3);
    static constexpr int DPL = kSplit ? 3 : D / 32;
    static_assert(kSplit ? (D > 64 && D <= 96) : (D == 32 || D == 64 || D == 128), "head dim");
    __device__ static __forceinline__ int dim(int lane, int i) {
        return kSplit ? (i < 2 ? 2 * lane + i : 64 + lane) : lane * DPL + i;
    }
    __device__ static __forceinline__ bool has(int lane, int i) { return dim(lane, i) < D; }
};

__device__ __forceinline__ float bf16_bits_to_float(uint32_t lo16) { return __uint_as_float(lo16 << 16); }

// Load DPL consecutive bf16 from shared memory as fp32.
template <int DPL>
__device__ __forceinline__ void load_bf16(const __nv_bfloat16 *p, float (&f)[DPL]) {
    if constexpr (DPL == 4) {
        uint2 u = *reinterpret_cast<const uint2 *>(p);
        f[0] = __uint_as_float(u.x << 16);
        f[1] = __uint_as_float(u.x & 0xffff0000u);
        f[2] = __uint_as_float(u.y << 16);
        f[3] = __uint_as_float(u.y & 0xffff0000u);
    } else if constexpr (DPL == 2) {
        uint32_t u = *reinterpret_cast<const uint32_t *>(p);
        f[0] = __uint_as_float(u << 16);
        f[1] = __uint_as_float(u & 0xffff0000u);
    } else {
        f[0] = bf16_bits_to_float(*reinterpret_cast<const uint16_t *>(p));
    }
}

// Two e4m3 codes (the low 16 bits, low byte first) -> two fp32 values (exact: every e4m3 value is
// an fp16 value, and every fp16 value an fp32 value).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two) {
    float2 r;
    asm("{\n\t.reg .b16 l, h, a, b;\n\t.reg .b32 x;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 x, l;\n\t"
        "mov.b32 {a, b}, x;\n\t"
        "cvt.f32.f16 %0, a;\n\t"
        "cvt.f32.f16 %1, b;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "r"(two));
    return r;
}

// Four e4m3 codes (byte 0 lowest) -> four fp32 values (exact).
__device__ __forceinline__ void e4m3x4_to_float4(uint32_t w, float (&f)[4]) {
    uint32_t lo, hi;
    e4m3x4_to_f16x2x2(w, lo, hi);
    asm("{\n\t.reg .b16 a, b, c, d;\n\t"
        "mov.b32 {a, b}, %4;\n\t"
        "mov.b32 {c, d}, %5;\n\t"
        "cvt.f32.f16 %0, a;\n\t"
        "cvt.f32.f16 %1, b;\n\t"
        "cvt.f32.f16 %2, c;\n\t"
        "cvt.f32.f16 %3, d;\n\t}"
        : "=f"(f[0]), "=f"(f[1]), "=f"(f[2]), "=f"(f[3])
        : "r"(lo), "r"(hi));
}

// Load DPL consecutive e4m3 codes from shared memory as fp32 (unscaled).
template <int DPL>
__device__ __forceinline__ void load_e4m3(const uint8_t *p, float (&f)[DPL]) {
    if constexpr (DPL == 4) {
        e4m3x4_to_float4(*reinterpret_cast<const uint32_t *>(p), f);
    } else if constexpr (DPL == 2) {
        const float2 a = e4m3x2_to_float2(*reinterpret_cast<const uint16_t *>(p));
        f[0] = a.x;
        f[1] = a.y;
    } else {
        f[0] = e4m3x2_to_float2(*p).x;
    }
}

// This lane's dims of one cache row (bf16 or e4m3) as fp32, laid out as LaneDims<D>.
template <int D, bool FP8>
__device__ __forceinline__ void load_kv(const uint8_t *row, int lane, float (&f)[LaneDims<D>::DPL]) {
    using LD = LaneDims<D>;
    if constexpr (LD::kSplit) {
        float pr[2], one[1] = {0.f};
        if constexpr (FP8) {
            load_e4m3<2>(row + 2 * lane, pr);
            if (lane < D - 64) load_e4m3<1>(row + 64 + lane, one);
        } else {
            load_bf16<2>(reinterpret_cast<const __nv_bfloat16 *>(row) + 2 * lane, pr);
            if (lane < D - 64) load_bf16<1>(reinterpret_cast<const __nv_bfloat16 *>(row) + 64 + lane, one);
        }
        f[0] = pr[0];
        f[1] = pr[1];
        f[2] = one[0];
    } else {
        if constexpr (FP8) load_e4m3<LD::DPL>(row + lane * LD::DPL, f);
        else load_bf16<LD::DPL>(reinterpret_cast<const __nv_bfloat16 *>(row) + lane * LD::DPL, f);
    }
}

// This lane's dims of the query row (bf16 in global memory) as fp32 scaled by c.
template <int D>
__device__ __forceinline__ void load_q(const __nv_bfloat16 *qrow, int lane, float c, float (&qf)[LaneDims<D>::DPL]) {
    load_kv<D, false>(reinterpret_cast<const uint8_t *>(qrow), lane, qf);
#pragma unroll
    for (int i = 0; i < LaneDims<D>::DPL; ++i) qf[i] *= c;
}

// Sum of part[t] over the 32 lanes for the 16 tokens t, as a reduce-scatter: afterwards lane
// L holds the full sum for token L >> 1 (lanes 2t, 2t+1 hold the same value).  16 shuffles.
__device__ __forceinline__ float reduce_scatter16(const float (&part)[16], int lane) {
    float r8[8];
    {
        const bool up = lane & 16;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float send = up ? part[i] : part[i + 8];
            const float keep = up ? part[i + 8] : part[i];
            r8[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
    }
    float r4[4];
    {
        const bool up = lane & 8;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float send = up ? r8[i] : r8[i + 4];
            const float keep = up ? r8[i + 4] : r8[i];
            r4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
    }
    float r2[2];
    {
        const bool up = lane & 4;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float send = up ? r4[i] : r4[i + 2];
            const float keep = up ? r4[i + 2] : r4[i];
            r2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
    }
    float x;
    {
        const bool up = lane & 2;
        const float send = up ? r2[0] : r2[1];
        const float keep = up ? r2[1] : r2[0];
        x = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    return x + __shfl_xor_sync(0xffffffffu, x, 1);
}

// Multi-head decode at d = 32 and 64 splits the warp into groups of T = d / 8 lanes, each lane
// holding 8 consecutive dims of one token, and the 32 / T groups take different tokens of a page in
// each round.  A score then needs a sum over T lanes only (2 or 3 shuffles instead of a 16-token
// reduce-scatter), and each group keeps its own tokens' probabilities for O += P V (no per-token
// broadcasts); the groups' partial O are summed once per CTA.  At d = 128 a token fills the warp.
// Measured, fraction of HBM with 4 / 8 / 16 dims per lane: bf16 d = 32 0.89 / 0.90 / 0.88; e4m3
// d = 32 0.515 / 0.55 / 0.52, d = 64 0.71 / 0.80 / 0.79.
template <int D> constexpr bool kLaneGroups = (D == 32 || D == 64);
// dims per lane in the lane groups (4 or 8)
template <int D, bool FP8> constexpr int kGroupDims = 8;

// N (4, 8 or 16) consecutive elements of a cache row (bf16, or e4m3 codes) as fp32: one 4-, 8- or
// 16-byte load per 4, 8 or 16 codes, one per 4 or 8 bf16 values.
template <bool FP8, int N>
__device__ __forceinline__ void load_n(const uint8_t *p, float (&f)[N]) {
    static_assert(N == 4 || N == 8 || N == 16, "4, 8 or 16 elements");
    uint32_t w[FP8 ? N / 4 : N / 2];  // the packed elements
    if constexpr ((FP8 ? N : 2 * N) == 8) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        w[0] = u.x;
        w[1] = u.y;
    } else if constexpr ((FP8 ? N : 2 * N) == 4) {
        w[0] = *reinterpret_cast<const uint32_t *>(p);
    } else {
#pragma unroll
        for (int j = 0; j < (FP8 ? N : 2 * N) / 16; ++j) {
            const uint4 u = reinterpret_cast<const uint4 *>(p)[j];
            w[4 * j] = u.x;
            w[4 * j + 1] = u.y;
            w[4 * j + 2] = u.z;
            w[4 * j + 3] = u.w;
        }
    }
    if constexpr (FP8) {
#pragma unroll
        for (int j = 0; j < N / 4; ++j) {
            float a[4];
            e4m3x4_to_float4(w[j], a);
#pragma unroll
            for (int i = 0; i < 4; ++i) f[4 * j + i] = a[i];
        }
    } else {
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
}

// One CTA: one chunk of one sequence's cache for one key/value head, applied to GP query
// heads that share that head (grouped-query attention; GP = 1 for multi-head attention).
// Grid (chunks, Hkv * gsplit, B): blockIdx.y = kv_head * gsplit + group slice.
template <int D, int GP, bool FP8>
__global__ void __launch_bounds__(kWarps * 32) decode_split_kernel(const DecodeArgs a, int max_splits, int Hkv,
                                                                   int gsplit, int chunk) {
    using LD = LaneDims<D>;
    constexpr int DPL = LD::DPL;  // head dims per lane
    constexpr int kElem = FP8 ? 1 : 2;
    constexpr uint32_t kRowBytes = D * kElem;
    constexpr uint32_t kBlockBytes = kPS * kRowBytes;
    static_assert(GP == 1, "grouped-query decode runs in decode_gqa_mma_kernel");
    extern __shared__ __align__(128) uint8_t smem_raw[];
    DecodeSmem<D, GP, FP8> &sm = *reinterpret_cast<DecodeSmem<D, GP, FP8> *>(smem_raw);

    const int split = blockIdx.x, b = blockIdx.z;
    const int kvh = (int)blockIdx.y / gsplit;
    const int qh0 = kvh * (a.H / Hkv) + ((int)blockIdx.y % gsplit) * GP;  // first query head
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cap = a.max_pages * kPS;
    const int ctx = min(max(a.ctx_lens[b], 0), cap);
    const int tok0 = split * chunk;
    if (tok0 >= ctx) return;  // uniform over the CTA: this chunk is empty
    const int tok1 = min(ctx, tok0 + chunk);
    const int page0 = tok0 / kPS;
    const int npages = (tok1 - tok0 + kPS - 1) / kPS;  // <= chunk / kPS <= 128
    const int nk = npages > warp ? (npages - warp + kWarps - 1) / kWarps : 0;  // pages of this warp (<= 32)

    if (threadIdx.x == 0) {
        for (int w = 0; w < kWarps; ++w)
            for (int s = 0; s < kSlotsFor<FP8, GP>; ++s) mbar_init(&sm.full[w][s], 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    WaitCtx wc{&sm.abort_flag, a.status};

    // Page ids of this warp's pages: lane k holds the id of local page k.
    int my_pid = -1;
    if (lane < nk) my_pid = a.page_table[(size_t)b * a.max_pages + page0 + warp + kWarps * lane];
    const bool my_ok = (my_pid >= 0 && my_pid < a.num_pages);

    const uint8_t *kbase = reinterpret_cast<const uint8_t *>(a.k_pages);
    const uint8_t *vbase = reinterpret_cast<const uint8_t *>(a.v_pages);
    auto issue = [&](int k) {
        const int pid = __shfl_sync(0xffffffffu, my_pid, k);
        const bool ok = __shfl_sync(0xffffffffu, my_ok ? 1 : 0, k) != 0;
        if (lane == 0) {
            uint64_t *bar = &sm.full[warp][k % kSlotsFor<FP8, GP>];
            if (ok) {
                const size_t off = ((size_t)pid * Hkv + kvh) * (size_t)kBlockBytes;
                mbar_arrive_expect_tx(bar, 2 * kBlockBytes);
                bulk_load(sm.kv[warp][k % kSlotsFor<FP8, GP>][0], kbase + off, kBlockBytes, bar);
                bulk_load(sm.kv[warp][k % kSlotsFor<FP8, GP>][1], vbase + off, kBlockBytes, bar);
            } else {
                mbar_arrive(bar);  // nothing to load: complete the phase so the consumer stays in step
            }
        }
    };
    const int first = nk < kSlotsFor<FP8, GP> ? nk : kSlotsFor<FP8, GP>;
    for (int k = 0; k < first; ++k) issue(k);

    // Queries, pre-scaled into the log2 domain: x = (scale * log2 e) * q.k (times the key scale
    // of an e4m3 cache, whose codes are then used as they are)
    const float c = a.scale * kLog2e * (FP8 ? a.k_scale : 1.f);
    float qf[GP][DPL];
#pragma unroll
    for (int g = 0; g < GP; ++g)
        load_q<D>(reinterpret_cast<const __nv_bfloat16 *>(a.q) + ((size_t)b * a.H + qh0 + g) * D, lane, c, qf[g]);

    float m_run[GP], l_run[GP], o[GP][DPL];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        m_run[g] = -INFINITY;
        l_run[g] = 0.f;
#pragma unroll
        for (int i = 0; i < DPL; ++i) o[g][i] = 0.f;
    }
    // lane groups (d = 32, 64): this lane's token group and its dims 4 cq .. 4 cq + 3
    constexpr int kGD = kGroupDims<D, FP8>;          // dims per lane
    constexpr int kT = kLaneGroups<D> ? D / kGD : 32;  // lanes per token
    constexpr int kG = 32 / kT;                        // tokens per round
    constexpr int kR = kPS / kG;                       // rounds per page
    const int gq = lane / kT, cq = lane % kT;
    float q4[kGD], o4[kGD];
#pragma unroll
    for (int i = 0; i < kGD; ++i) q4[i] = o4[i] = 0.f;
    if constexpr (kLaneGroups<D>) {
        load_n<false, kGD>(reinterpret_cast<const uint8_t *>(a.q) + (((size_t)b * a.H + qh0) * D + kGD * cq) * 2, q4);
#pragma unroll
        for (int i = 0; i < kGD; ++i) q4[i] *= c;
    }

    int issued = first;
    bool failed = false;
    for (int k = 0; k < nk; ++k) {
        const int slot = k % kSlotsFor<FP8, GP>;
        if (!mbar_wait(&sm.full[warp][slot], (uint32_t)((k / kSlotsFor<FP8, GP>) & 1), wc, 100 + warp)) {
            failed = true;
            break;
        }
        const bool ok = __shfl_sync(0xffffffffu, my_ok ? 1 : 0, k) != 0;
        const int page_tok0 = tok0 + (warp + kWarps * k) * kPS;
        const int ntok = min(kPS, tok1 - page_tok0);
        if (ok && kLaneGroups<D>) {
            const uint8_t *Ks = sm.kv[warp][slot][0];
            const uint8_t *Vs = sm.kv[warp][slot][1];
            // round r: token r * kG + gq of the page, scored by its group of kT lanes
            float x[kR];
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                float k4[kGD];
                load_n<FP8, kGD>(Ks + (r * kG + gq) * kRowBytes + kGD * cq * kElem, k4);
                float acc = q4[0] * k4[0];
#pragma unroll
                for (int i = 1; i < kGD; ++i) acc = fmaf(q4[i], k4[i], acc);
#pragma unroll
                for (int off = 1; off < kT; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                x[r] = acc;
            }
            if (ntok < kPS) {  // slots past the context end (a sequence's last page)
#pragma unroll
                for (int r = 0; r < kR; ++r)
                    if (r * kG + gq >= ntok) x[r] = -INFINITY;
            }
            float mx = x[0];
#pragma unroll
            for (int r = 1; r < kR; ++r) mx = fmaxf(mx, x[r]);
#pragma unroll
            for (int off = kT; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_new = fmaxf(m_run[0], mx);  // finite: ntok >= 1
            const float alpha = ex2_approx(m_run[0] - m_new);
            float pr[kR], ps = 0.f;
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                pr[r] = ex2_approx(x[r] - m_new);
                ps += pr[r];
            }
            // each group's lanes hold the same values: sum over the groups only
#pragma unroll
            for (int off = kT; off < 32; off <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
            l_run[0] = l_run[0] * alpha + ps;
            m_run[0] = m_new;
#pragma unroll
            for (int i = 0; i < kGD; ++i) o4[i] *= alpha;
            auto pv_round = [&](int r) {
                float v4[kGD];
                load_n<FP8, kGD>(Vs + (r * kG + gq) * kRowBytes + kGD * cq * kElem, v4);
#pragma unroll
                for (int i = 0; i < kGD; ++i) o4[i] = fmaf(pr[r], v4[i], o4[i]);
            };
            // V rows past the context end are never read (they may hold anything)
            if (ntok == kPS) {
#pragma unroll
                for (int r = 0; r < kR; ++r) pv_round(r);
            } else {
#pragma unroll
                for (int r = 0; r < kR; ++r)
                    if (r * kG + gq < ntok) pv_round(r);
            }
        } else if (ok) {
            const uint8_t *Ks = sm.kv[warp][slot][0];
            const uint8_t *Vs = sm.kv[warp][slot][1];
            // this lane's DPL dims of the 16 keys, read once and used for every query head
            float kf[16][DPL];
#pragma unroll
            for (int t = 0; t < 16; ++t) load_kv<D, FP8>(Ks + t * kRowBytes, lane, kf[t]);
            float p[GP];  // lane L: probability of token L >> 1, per query head
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                float part[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    float acc = 0.f;
#pragma unroll
                    for (int i = 0; i < DPL; ++i) acc = fmaf(qf[g][i], kf[t][i], acc);
                    part[t] = acc;
                }
                float x = reduce_scatter16(part, lane);
                if ((lane >> 1) >= ntok) x = -INFINITY;  // slots past the context end
                const float m_new = fmaxf(m_run[g], warp_max_pairs(x));  // finite: ntok >= 1
                const float alpha = ex2_approx(m_run[g] - m_new);
                p[g] = ex2_approx(x - m_new);
                l_run[g] = l_run[g] * alpha + warp_sum_pairs(p[g]);
                m_run[g] = m_new;
#pragma unroll
                for (int i = 0; i < DPL; ++i) o[g][i] *= alpha;
            }
            auto pv_token = [&](int t) {
                float vf[DPL];
                load_kv<D, FP8>(Vs + t * kRowBytes, lane, vf);
#pragma unroll
                for (int g = 0; g < GP; ++g) {
                    const float pt = __shfl_sync(0xffffffffu, p[g], 2 * t);
#pragma unroll
                    for (int i = 0; i < DPL; ++i) o[g][i] = fmaf(pt, vf[i], o[g][i]);
                }
            };
            // V rows past the context end are never read (they may hold anything); every page but a
            // sequence's last is full and takes the unrolled form
            if (ntok == kPS) {
#pragma unroll
                for (int t = 0; t < kPS; ++t) pv_token(t);
            } else {
                for (int t = 0; t < ntok; ++t) pv_token(t);
            }
        }
        // the slot is free again: order this warp's reads before the next bulk write
        fence_proxy_async_smem();
        __syncwarp();
        if (k + kSlotsFor<FP8, GP> < nk) {
            issue(k + kSlotsFor<FP8, GP>);
            ++issued;
        }
    }
    if (failed) {
        // drain this warp's copies still in flight (bounded) before the CTA exits
        WaitCtx drain{nullptr, a.status};
        for (int k = 0; k < issued; ++k) {
            if (lane == 0 && k + kSlotsFor<FP8, GP> >= issued)  // the last use of each slot
                (void)mbar_wait(&sm.full[warp][k % kSlotsFor<FP8, GP>], (uint32_t)((k / kSlotsFor<FP8, GP>) & 1), drain, 199);
        }
        __syncwarp();
    }

    // merge the four warp states of every query head
    if constexpr (kLaneGroups<D>) {  // the token groups' partial O (they share m_run)
#pragma unroll
        for (int i = 0; i < kGD; ++i)
#pragma unroll
            for (int off = kT; off < 32; off <<= 1) o4[i] += __shfl_xor_sync(0xffffffffu, o4[i], off);
    }
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        if (lane == 0) {
            sm.red_m[warp][g] = m_run[g];
            sm.red_l[warp][g] = l_run[g];
        }
        if constexpr (kLaneGroups<D>) {
            if (gq == 0) {
#pragma unroll
                for (int i = 0; i < kGD; ++i) sm.red_o[warp][g][kGD * cq + i] = o4[i];
            }
        } else {
#pragma unroll
            for (int i = 0; i < DPL; ++i)
                if (LD::has(lane, i)) sm.red_o[warp][g][LD::dim(lane, i)] = o[g][i];
        }
    }
    __syncthreads();
    if (sm.abort_flag) return;
    for (int e = threadIdx.x; e < GP * D; e += blockDim.x) {
        const int g = e / D, dd = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.red_m[w][g]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float wgt = ex2_approx(sm.red_m[w][g] - M);
                L += sm.red_l[w][g] * wgt;
                O += sm.red_o[w][g][dd] * wgt;
            }
        }
        float *ws = reinterpret_cast<float *>(a.workspace) +
                    (((size_t)b * a.H + qh0 + g) * max_splits + split) * (size_t)ws_stride<D>();
        ws[dd] = FP8 ? O * a.v_scale : O;
        if (dd == 0) {
            ws[D] = M;
            ws[D + 1] = L;
        }
    }
    griddep_launch_dependents();
}

// ------------------------------------------------------------------ grouped-query decode on mma
// With GP query heads per key/value head the scalar kernel spends about 12 warp-instructions per
// (token, query head) on dot products, shuffles and broadcasts, and becomes compute-bound.  Here
// each warp runs the two products of a 16-token page on the tensor cores with mma.sync
// (m16n8k16, bf16 -> fp32): S = Q K^T with the group's query heads as the M rows (padded to 16),
// and O += P V with P taken straight from the score fragments (the C layout of two n8 tiles is
// the A layout of one k16 step).  K and V fragments come from the page blocks in shared memory
// through ldmatrix (transposed for V).  Softmax per row over the quad of lanes that holds it,
// with the same lazy reference max as the prefill (O and l are rescaled only when a row max
// grows by more than 2^8).  The page blocks arrive by TMA in 128-byte-swizzled boxes of 16 rows x
// 64 columns (the 16-byte chunk c of row r sits at chunk c ^ (r & 7)), so the eight rows of every
// ldmatrix read fall in different banks.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
// d (+)= a b: a 16x16 bf16 (row-major fragment), b 16x8 bf16 (column-major fragment), d 16x8 fp32.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// The same product over f16 fragments.
__device__ __forceinline__ void mma_16816_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Byte permute: byte i of the result is byte (sel >> 4i) & 7 of {hi:lo}.
__device__ __forceinline__ uint32_t prmt(uint32_t lo, uint32_t hi, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(lo), "r"(hi), "r"(sel));
    return r;
}

// Byte offset of the 16-byte chunk holding column col (a multiple of 8) of row r in a page block
// stored as 128-byte-swizzled boxes of 16 rows x 64 bf16 columns.
__device__ __forceinline__ uint32_t swz_off(int r, int col) {
    return (uint32_t)((col >> 6) * (16 * 128) + r * 128 + ((((col & 63) >> 3) ^ (r & 7)) << 4));
}

// An e4m3 cache takes the same path with f16 products.  Each page block arrives by TMA as one
// 128-byte-swizzled box of 16 rows x 128 codes, and ldmatrix hands every lane its codes in
// fragment order, so they are widened in registers (one conversion per two codes, exact) with no
// staging copy:
//  - K (plain ldmatrix of 8 tokens x 16 codes): lane (g, t) gets dims 16c + 4t .. 16c + 4t + 3 of
//    token g, the B fragment of k-step c when the k-step's logical index 2t + {0, 1} stands for dims
//    16c + 4t + {0, 1} and 2t + 8 + {0, 1} for 16c + 4t + 2 + {0, 1}.  Q's A fragments are loaded in
//    the same order (a permutation of the contraction index leaves Q K^T unchanged).
//  - V (transposed ldmatrix, codes taken in pairs): lane (g, t) gets tokens 2t, 2t + 1 of dims
//    16c + 2g and 16c + 2g + 1; one byte permute splits them into the B fragments of two n-tiles,
//    one over the chunk's even dims and one over its odd dims, and the final write of O puts
//    column n of n-tile (c, parity) at dim 16c + 2n + parity.
// Q is rounded to f16 once per CTA after a power-of-two factor that keeps |Q| below 2^15 (exact
// for every bf16 value in f16's normal range); the factor, the key scale and the softmax scale fold
// into the score scale, the value scale into the partial O.
// Ring slots per warp of the grouped-query kernel: the page loads in flight per warp.  Measured
// on 32 sequences x 8 cache heads (4 query heads each), contexts U[512, 8192], fraction of HBM:
// bf16 pages 1 / 2 / 3 slots 0.853 / 0.880 / 0.844; e4m3 pages 2 / 3 / 4 slots 0.565 / 0.555 /
// 0.557, and with registers capped for four CTAs per SM 0.53 / 0.53 / 0.50.  More pages in flight
// do not help the e4m3 form: it is bound by the work per page (two products, the softmax), not by
// the bytes in flight.
template <bool FP8> constexpr int kGqaSlots = 2;

template <int D, int GP, bool FP8>
struct GqaMmaSmem {
    // The page ring and the final merge's arrays are never in use at the same time (the merge
    // starts after every warp has consumed its last page), so they share their bytes.
    union {
        // [warp][slot][0 = K, 1 = V][one page block]: swizzled TMA boxes (16 x 64 bf16 each, or one
        // of 16 x 128 e4m3 codes); 1024-byte aligned for the swizzle
        alignas(1024) uint8_t kv[kWarps][kGqaSlots<FP8>][2][kBoxSlotBytes<D, FP8>];
        struct {
            float o[kWarps][GP][D];
            float m[kWarps][GP];
            float l[kWarps][GP];
        } red;
    } u;
    uint64_t full[kWarps][kGqaSlots<FP8>];
    int abort_flag;
};

template <int D, int GP, bool FP8>
__global__ void __launch_bounds__(kWarps * 32) decode_gqa_mma_kernel(const __grid_constant__ CUtensorMap tmK,
                                                                     const __grid_constant__ CUtensorMap tmV,
                                                                     const DecodeArgs a, int max_splits, int Hkv,
                                                                     int gsplit) {
    static_assert(GP >= 1 && GP <= 16, "query heads per CTA");
    static_assert(D % 16 == 0, "k-steps of 16");
    constexpr int kSl = kGqaSlots<FP8>;
    constexpr int kBx = FP8 ? 1 : kBoxes<D>;              // TMA boxes per page block (128-byte rows)
    constexpr uint32_t kBoxBytesAll = kBx * kPS * 128;    // a block's boxes (zero-filled past D)
    constexpr int KS = D / 16;  // k-steps of S = Q K^T
    constexpr int NT = D / 8;   // n-tiles of O += P V (even: n-tiles go in pairs)
    static_assert(NT % 2 == 0, "pairs of n-tiles");
    constexpr float kThresh = 8.0f;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    // the swizzled boxes need 1024-byte alignment
    GqaMmaSmem<D, GP, FP8> &sm =
        *reinterpret_cast<GqaMmaSmem<D, GP, FP8> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int split = blockIdx.x, b = blockIdx.z;
    const int kvh = (int)blockIdx.y / gsplit;
    const int qh0 = kvh * (a.H / Hkv) + ((int)blockIdx.y % gsplit) * GP;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cap = a.max_pages * kPS;
    const int ctx = min(max(a.ctx_lens[b], 0), cap);
    const int tok0 = split * kGqaChunkTokens;
    if (tok0 >= ctx) return;
    const int tok1 = min(ctx, tok0 + kGqaChunkTokens);
    const int page0 = tok0 / kPS;
    const int npages = (tok1 - tok0 + kPS - 1) / kPS;  // <= 64: at most 16 per warp, one per lane
    const int nk = npages > warp ? (npages - warp + kWarps - 1) / kWarps : 0;

    if (threadIdx.x == 0) {
        for (int w = 0; w < kWarps; ++w)
            for (int s2 = 0; s2 < kSl; ++s2) mbar_init(&sm.full[w][s2], 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    WaitCtx wc{&sm.abort_flag, a.status};

    int my_pid = -1;
    if (lane < nk) my_pid = a.page_table[(size_t)b * a.max_pages + page0 + warp + kWarps * lane];
    const bool my_ok = (my_pid >= 0 && my_pid < a.num_pages);
    if (lane == 0) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
    }
    auto issue = [&](int k) {
        const int pid = __shfl_sync(0xffffffffu, my_pid, k);
        const bool ok = __shfl_sync(0xffffffffu, my_ok ? 1 : 0, k) != 0;
        if (lane == 0) {
            uint64_t *bar = &sm.full[warp][k % kSl];
            if (ok) {
                const int row = pid * Hkv + kvh;  // page block in the pool viewed as [num_pages * Hkv, 16, D]
                mbar_arrive_expect_tx(bar, 2 * kBoxBytesAll);
#pragma unroll
                for (int i = 0; i < kBx; ++i) {  // box i: columns 64 i .. 64 i + 63 (bf16) or all 128 codes (e4m3)
                    tma_load_3d(sm.u.kv[warp][k % kSl][0] + i * (16 * 128), &tmK, bar, i * 64, 0, row);
                    tma_load_3d(sm.u.kv[warp][k % kSl][1] + i * (16 * 128), &tmV, bar, i * 64, 0, row);
                }
            } else {
                mbar_arrive(bar);
            }
        }
    };
    const int first = nk < kSl ? nk : kSl;
    for (int k = 0; k < first; ++k) issue(k);

    // Q as A fragments: rows r0 = lane / 4 and r0 + 8 (query heads qh0 + row; zero past GP)
    const int r0 = lane >> 2, kq = (lane & 3) * 2;
    const uint32_t *q32 = reinterpret_cast<const uint32_t *>(reinterpret_cast<const __nv_bfloat16 *>(a.q) +
                                                             ((size_t)b * a.H + qh0) * D);
    uint32_t qa[KS][4];
    float c = a.scale * kLog2e;
    if constexpr (FP8) {
        // dims 16 ks + 2 kq + {0, 1} (a0, a1) and + {2, 3} (a2, a3): the order of the K fragments
        float amax = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int rr = r0 + 8 * h;
                const uint2 u = rr < GP ? *reinterpret_cast<const uint2 *>(q32 + (rr * D + ks * 16 + 2 * kq) / 2)
                                        : make_uint2(0u, 0u);
                qa[ks][h] = u.x;
                qa[ks][h + 2] = u.y;
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(__uint_as_float(u.x << 16)), fabsf(__uint_as_float(u.x & 0xffff0000u))),
                                         fmaxf(fabsf(__uint_as_float(u.y << 16)), fabsf(__uint_as_float(u.y & 0xffff0000u)))));
            }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        // 2^-sh * |Q| < 2^15: sh = e - 14 when |Q| >= 2^15 (e its binary exponent); at most 113
        const int e = (int)((__float_as_uint(amax) >> 23) & 0xffu) - 127;
        const int sh = e >= 15 ? min(e - 14, 113) : 0;
        const float f = __uint_as_float((uint32_t)(127 - sh) << 23);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                qa[ks][i] = pack_f16x2(__uint_as_float(qa[ks][i] << 16) * f, __uint_as_float(qa[ks][i] & 0xffff0000u) * f);
        c *= a.k_scale * __uint_as_float((uint32_t)(127 + sh) << 23);
    } else {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int c0 = ks * 16 + kq;
            qa[ks][0] = r0 < GP ? q32[(r0 * D + c0) / 2] : 0u;
            qa[ks][1] = r0 + 8 < GP ? q32[((r0 + 8) * D + c0) / 2] : 0u;
            qa[ks][2] = r0 < GP ? q32[(r0 * D + c0 + 8) / 2] : 0u;
            qa[ks][3] = r0 + 8 < GP ? q32[((r0 + 8) * D + c0 + 8) / 2] : 0u;
        }
    }

    float o[NT][4];
#pragma unroll
    for (int nd = 0; nd < NT; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    float m_ref[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};  // rows r0, r0 + 8

    // ldmatrix: lane l gives row (l & 7) of 8x8 matrix l >> 3
    const int mi = lane >> 3, mr = lane & 7;
    const int k_row = (mi >> 1) * 8 + mr, k_col = (mi & 1) * 8;  // + ks * 16 columns
    const int v_row = (mi & 1) * 8 + mr, v_col = (mi >> 1) * 8;  // + nd * 8 columns
    // e4m3 boxes: matrices {tokens 0-7, tokens 8-15} x {chunk c, chunk c + 1} (16 codes a chunk)
    const int f_row = (mi & 1) * 8 + mr, f_chunk = mi >> 1;
    auto f_off = [](int r, int chunk) { return (uint32_t)(r * 128 + ((chunk ^ (r & 7)) << 4)); };

    int issued = first;
    bool failed = false;
    for (int k = 0; k < nk; ++k) {
        const int slot = k % kSl;
        if (!mbar_wait(&sm.full[warp][slot], (uint32_t)((k / kSl) & 1), wc, 120 + warp)) {
            failed = true;
            break;
        }
        const bool ok = __shfl_sync(0xffffffffu, my_ok ? 1 : 0, k) != 0;
        const int page_tok0 = tok0 + (warp + kWarps * k) * kPS;
        const int ntok = min(kPS, tok1 - page_tok0);
        if (ok) {
            const uint32_t Ks = smem_u32(sm.u.kv[warp][slot][0]);
            const uint32_t Vs = smem_u32(sm.u.kv[warp][slot][1]);
            if (ntok < kPS) {
                // slots past the context end: zero their V rows (every box) so P = 0 meets finite values
                const int per_box = (kPS - ntok) * 8;  // 16-byte chunks of the dead rows of one box
                for (int i = lane; i < per_box * kBx; i += 32) {
                    const int box = i / per_box, j = i % per_box;
                    *reinterpret_cast<uint4 *>(sm.u.kv[warp][slot][1] + box * (16 * 128) + ntok * 128 + j * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
            }
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            if constexpr (FP8) {
                // even and odd chunks accumulate in separate tiles (two shorter dependency chains)
                float sc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int ks = 0; ks < KS; ks += 2) {
                    uint32_t bk[4];  // tokens 0-7 / 8-15 of chunk ks, then of chunk ks + 1 (zeros past D)
                    ldsm_x4(Ks + f_off(f_row, ks + f_chunk), bk);
                    uint32_t b[4][2];
#pragma unroll
                    for (int i = 0; i < 4; ++i) e4m3x4_to_f16x2x2(bk[i], b[i][0], b[i][1]);
                    mma_16816_f16(sc[0], qa[ks], b[0][0], b[0][1]);
                    mma_16816_f16(sc[1], qa[ks], b[1][0], b[1][1]);
                    if (ks + 1 < KS) {
                        mma_16816_f16(sc2[0], qa[ks + 1], b[2][0], b[2][1]);
                        mma_16816_f16(sc2[1], qa[ks + 1], b[3][0], b[3][1]);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) sc[nt][i] += sc2[nt][i];
            } else {
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    uint32_t bk[4];
                    ldsm_x4(Ks + swz_off(k_row, ks * 16 + k_col), bk);
                    mma_16816(sc[0], qa[ks], bk[0], bk[1]);
                    mma_16816(sc[1], qa[ks], bk[2], bk[3]);
                }
            }
            // this lane holds the scores of tokens nt*8 + (lane&3)*2 + {0,1} of rows r0 / r0+8; slots
            // past the context end (only on a sequence's last page) become -inf
            if (ntok < kPS) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (nt * 8 + kq + (i & 1) >= ntok) sc[nt][i] = -INFINITY;
            }
            // row maxima of the raw scores, then the log2 domain (c > 0 keeps the order)
            float mx[2];
            mx[0] = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
            mx[1] = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
                mx[h] *= c;
            }
            float al[2] = {1.f, 1.f};
            bool resc = false;
#pragma unroll
            for (int h = 0; h < 2; ++h)
                if (mx[h] > m_ref[h] + kThresh) {
                    al[h] = ex2_approx(m_ref[h] - mx[h]);
                    m_ref[h] = mx[h];
                    l_run[h] *= al[h];
                    resc = true;
                }
            if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
                for (int nd = 0; nd < NT; ++nd) {
                    o[nd][0] *= al[0];
                    o[nd][1] *= al[0];
                    o[nd][2] *= al[1];
                    o[nd][3] *= al[1];
                }
            }
            float p[2][4], ps[2] = {0.f, 0.f};
            const float nm[2] = {-m_ref[0], -m_ref[1]};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    p[nt][i] = ex2_approx(fmaf(sc[nt][i], c, nm[i >> 1]));
                    ps[i >> 1] += p[nt][i];
                }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                ps[h] += __shfl_xor_sync(0xffffffffu, ps[h], 1);
                ps[h] += __shfl_xor_sync(0xffffffffu, ps[h], 2);
                l_run[h] += ps[h];
            }
            if constexpr (FP8) {
                const uint32_t pa[4] = {pack_f16x2(p[0][0], p[0][1]), pack_f16x2(p[0][2], p[0][3]),
                                        pack_f16x2(p[1][0], p[1][1]), pack_f16x2(p[1][2], p[1][3])};
#pragma unroll
                for (int ch = 0; ch < KS; ch += 2) {
                    uint32_t bv[4];  // per lane: tokens 2t, 2t+1 (+ 8) x dims 2g, 2g+1 of chunks ch, ch + 1
                    ldsm_x4_trans(Vs + f_off(f_row, ch + f_chunk), bv);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        if (ch + j < KS) {
                            // {tok 2t dim 2g, tok 2t+1 dim 2g} | {tok 2t dim 2g+1, tok 2t+1 dim 2g+1}
                            uint32_t e0, o0, e1, o1;  // even / odd dim of tokens 2t, 2t+1 and of 2t+8, 2t+9
                            e4m3x4_to_f16x2x2(prmt(bv[2 * j], 0u, 0x3120u), e0, o0);
                            e4m3x4_to_f16x2x2(prmt(bv[2 * j + 1], 0u, 0x3120u), e1, o1);
                            mma_16816_f16(o[2 * (ch + j)], pa, e0, e1);
                            mma_16816_f16(o[2 * (ch + j) + 1], pa, o0, o1);
                        }
                    }
                }
            } else {
                const uint32_t pa[4] = {pack_bf16x2(p[0][0], p[0][1]), pack_bf16x2(p[0][2], p[0][3]),
                                        pack_bf16x2(p[1][0], p[1][1]), pack_bf16x2(p[1][2], p[1][3])};
#pragma unroll
                for (int nd = 0; nd < NT; nd += 2) {
                    uint32_t bv[4];
                    ldsm_x4_trans(Vs + swz_off(v_row, nd * 8 + v_col), bv);
                    mma_16816(o[nd], pa, bv[0], bv[1]);
                    mma_16816(o[nd + 1], pa, bv[2], bv[3]);
                }
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (k + kSl < nk) {
            issue(k + kSl);
            ++issued;
        }
    }
    if (failed) {
        WaitCtx drain{nullptr, a.status};
        for (int k = 0; k < issued; ++k) {
            if (lane == 0 && k + kSl >= issued)
                (void)mbar_wait(&sm.full[warp][k % kSl], (uint32_t)((k / kSl) & 1), drain, 198);
        }
        __syncwarp();
    }

    // this warp's state of each query head -> shared memory (over the ring, once every warp is
    // done with its pages), then the merge of the kernel above
    __syncthreads();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int g = r0 + 8 * h;
        if (g < GP) {
            if ((lane & 3) == 0) {
                sm.u.red.m[warp][g] = m_ref[h];
                sm.u.red.l[warp][g] = l_run[h];
            }
#pragma unroll
            for (int nd = 0; nd < NT; ++nd) {
                // columns kq, kq + 1 of n-tile nd: dims nd * 8 + kq + {0, 1}, or for e4m3 pages
                // 16 (nd / 2) + 2 kq + (nd % 2) + {0, 2}
                const int d0 = FP8 ? (nd >> 1) * 16 + 2 * kq + (nd & 1) : nd * 8 + kq;
                sm.u.red.o[warp][g][d0] = o[nd][2 * h];
                sm.u.red.o[warp][g][d0 + (FP8 ? 2 : 1)] = o[nd][2 * h + 1];
            }
        }
    }
    __syncthreads();
    if (sm.abort_flag) return;
    for (int e = threadIdx.x; e < GP * D; e += blockDim.x) {
        const int g = e / D, dd = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.u.red.m[w][g]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float wgt = ex2_approx(sm.u.red.m[w][g] - M);
                L += sm.u.red.l[w][g] * wgt;
                O += sm.u.red.o[w][g][dd] * wgt;
            }
        }
        float *ws = reinterpret_cast<float *>(a.workspace) +
                    (((size_t)b * a.H + qh0 + g) * max_splits + split) * (size_t)ws_stride<D>();
        ws[dd] = FP8 ? O * a.v_scale : O;
        if (dd == 0) {
            ws[D] = M;
            ws[D + 1] = L;
        }
    }
    griddep_launch_dependents();
}

// Merge of one (sequence, query head)'s chunk partials.  The splits' maxima, weights and
// normalisers come from loads spread over the block and block reductions; each thread then
// walks the splits for its O column with independent loads (the weights of the first
// kCombineWeights splits from shared memory).  A walk with two dependent global loads per
// split took about 9.5 us per call at 16 splits.
constexpr int kCombineWeights = 256;
// One thread per O column, in whole warps (D = 80 has 16 threads without a column).
template <int D> constexpr int kCombineThreads = (D + 31) / 32 * 32;
template <int D>
__device__ __forceinline__ float block_reduce(float v, bool is_max, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float w = __shfl_xor_sync(0xffffffffu, v, o);
        v = is_max ? fmaxf(v, w) : v + w;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();  // red[] is free (an earlier reduction has been read)
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float r = red[0];
#pragma unroll
    for (int w = 1; w < kCombineThreads<D> / 32; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
    return r;
}

template <int D>
__global__ void __launch_bounds__(kCombineThreads<D>) decode_combine_kernel(const DecodeArgs a, int max_splits,
                                                                             int chunk) {
    constexpr int kT = kCombineThreads<D>;
    __shared__ float red[kT / 32];
    __shared__ float wgt[kCombineWeights];
    griddep_wait();  // the split kernel's partials are complete and visible
    const int h = blockIdx.x, b = blockIdx.y, dd = threadIdx.x;
    const int cap = a.max_pages * kPS;
    const int ctx = min(max(a.ctx_lens[b], 0), cap);
    const int nsplit = (ctx + chunk - 1) / chunk;
    const size_t stride = (size_t)ws_stride<D>();
    const float *ws = reinterpret_cast<const float *>(a.workspace) + ((size_t)b * a.H + h) * max_splits * stride;
    float m = -INFINITY;
    for (int s = dd; s < nsplit; s += kT) m = fmaxf(m, ws[(size_t)s * stride + D]);
    const float M = block_reduce<D>(m, true, red);
    float lsum = 0.f;
    if (M != -INFINITY) {
        for (int s = dd; s < nsplit; s += kT) {
            const float w = ex2_approx(ws[(size_t)s * stride + D] - M);
            if (s < kCombineWeights) wgt[s] = w;
            lsum += ws[(size_t)s * stride + D + 1] * w;
        }
    }
    const float L = block_reduce<D>(lsum, false, red);  // its barriers also publish wgt[]
    if (dd >= D) return;  // no O column (after the block's last barrier)
    float O = 0.f;
    if (M != -INFINITY) {
#pragma unroll 8
        for (int s = 0; s < nsplit; ++s) {
            const float *w = ws + (size_t)s * stride;
            const float ws_wgt = s < kCombineWeights ? wgt[s] : ex2_approx(w[D] - M);
            O += w[dd] * ws_wgt;
        }
    }
    const size_t row = (size_t)b * a.H + h;
    __nv_bfloat16 *op = reinterpret_cast<__nv_bfloat16 *>(a.o) + row * D;
    const bool any = L > 0.f;
    op[dd] = __float2bfloat16_rn(any ? O / L : 0.f);
    if (dd == 0 && a.lse) a.lse[row] = any ? kLn2 * (M + __log2f(L)) : -INFINITY;
}

template <int D, int GP, bool FP8>
cudaError_t launch_decode_g(const DecodeArgs &a, int max_splits, int chunk, cudaStream_t stream) {
    const size_t smem = sizeof(DecodeSmem<D, GP, FP8>);
    cudaError_t e =
        ensure_max_dynamic_smem(reinterpret_cast<const void *>(decode_split_kernel<D, GP, FP8>), (int)smem);
    if (e != cudaSuccess) return e;
    const int gsplit = (a.H / a.Hkv) / GP;  // CTAs per key/value head
    dim3 g1(max_splits, a.Hkv * gsplit, a.B);
    decode_split_kernel<D, GP, FP8><<<g1, kWarps * 32, smem, stream>>>(a, max_splits, a.Hkv, gsplit, chunk);
    return cudaGetLastError();
}

template <int D, int GP, bool FP8>
cudaError_t launch_decode_mma(const DecodeArgs &a, int max_splits, cudaStream_t stream) {
    // page pool [num_pages * Hkv, 16, D]: bf16 pages in 16 x 64 boxes (one per 64 columns), e4m3
    // pages in one 16 x 128-code box per page block
    CUtensorMap tk{}, tv{};
    const int rows = a.num_pages * a.Hkv;
    const bool ok = FP8 ? (encode_page_map_u8(&tk, a.k_pages, rows, kPS, D) &&
                           encode_page_map_u8(&tv, a.v_pages, rows, kPS, D))
                        : (encode_qkv_map(&tk, a.k_pages, rows, kPS, D, kPS) &&
                           encode_qkv_map(&tv, a.v_pages, rows, kPS, D, kPS));
    if (!ok) return cudaErrorInvalidValue;
    const size_t smem = sizeof(GqaMmaSmem<D, GP, FP8>) + 1024;
    cudaError_t e =
        ensure_max_dynamic_smem(reinterpret_cast<const void *>(decode_gqa_mma_kernel<D, GP, FP8>), (int)smem);
    if (e != cudaSuccess) return e;
    const int gsplit = (a.H / a.Hkv) / GP;
    dim3 g1(max_splits, a.Hkv * gsplit, a.B);
    decode_gqa_mma_kernel<D, GP, FP8><<<g1, kWarps * 32, smem, stream>>>(tk, tv, a, max_splits, a.Hkv, gsplit);
    return cudaGetLastError();
}

// Multi-head attention (one query head per CTA) runs on the tensor-core kernel where that measured
// faster than the scalar kernel.  Fraction of HBM on 32 sequences x 32 heads, contexts U[512, 8192],
// scalar / tensor-core: bf16 d = 32 0.90 / 0.64, 64 0.96 / 0.97, 80 0.96 / 0.96, 96 1.00 / 1.00; e4m3
// d = 32 0.51 / 0.45, 64 0.71 / 0.66, 80 0.63 / 0.52, 96 0.81 / 0.84 (d = 32 and 64 on the scalar
// kernel's lane groups).  Both split at 1024 tokens below d = 128.
template <int D, bool FP8> constexpr bool kMhaOnMma = FP8 ? (D == 96) : (D == 64);

template <int D, bool FP8>
cudaError_t launch_decode_gf(const DecodeArgs &a, int max_splits, int chunk, cudaStream_t stream) {
    static_assert(!kMhaOnMma<D, FP8> || mha_chunk_tokens(D) == kGqaChunkTokens, "the workspace's split length");
    if constexpr (kMhaOnMma<D, FP8>) return launch_decode_mma<D, 1, FP8>(a, max_splits, stream);
    else return launch_decode_g<D, 1, FP8>(a, max_splits, chunk, stream);
}

template <int D, int GP>
cudaError_t launch_decode_gk(const DecodeArgs &a, int max_splits, int chunk, cudaStream_t stream) {
    if constexpr (GP >= 2) {
        return a.kv_fp8 ? launch_decode_mma<D, GP, true>(a, max_splits, stream)
                        : launch_decode_mma<D, GP, false>(a, max_splits, stream);
    } else {
        return a.kv_fp8 ? launch_decode_gf<D, true>(a, max_splits, chunk, stream)
                        : launch_decode_gf<D, false>(a, max_splits, chunk, stream);
    }
}

template <int D>
cudaError_t launch_decode_d(const DecodeArgs &a, cudaStream_t stream) {
    // query heads per CTA: the largest of 8, 4, 2, 1 dividing the group size; groups of two or more
    // run the grouped-query kernel and its longer chunks
    const int group = a.H / a.Hkv;
    const int chunk = decode_chunk_tokens(a.H, a.Hkv, D);
    const int max_splits = (a.max_pages * kPS + chunk - 1) / chunk;
    cudaError_t e;
    if (group % 8 == 0) e = launch_decode_gk<D, 8>(a, max_splits, chunk, stream);
    else if (group % 4 == 0) e = launch_decode_gk<D, 4>(a, max_splits, chunk, stream);
    else if (group % 2 == 0) e = launch_decode_gk<D, 2>(a, max_splits, chunk, stream);
    else e = launch_decode_gk<D, 1>(a, max_splits, chunk, stream);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.H, a.B);
    cfg.blockDim = dim3(kCombineThreads<D>);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, a, max_splits, chunk);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

size_t decode_workspace_bytes(int B, int H, int Hkv, int d, int max_pages, int page_size) {
    if (B <= 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0 || max_pages <= 0 || page_size != kPS ||
        (d != 32 && d != 64 && d != 80 && d != 96 && d != 128))
        return 0;
    const size_t chunk = (size_t)decode_chunk_tokens(H, Hkv, d);
    const size_t max_splits = ((size_t)max_pages * kPS + chunk - 1) / chunk;
    return (size_t)B * H * max_splits * (size_t)(d + 4) * sizeof(float);
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream) {
    switch (a.d) {
        case 32: return launch_decode_d<32>(a, stream);
        case 64: return launch_decode_d<64>(a, stream);
        case 80: return launch_decode_d<80>(a, stream);
        case 96: return launch_decode_d<96>(a, stream);
        case 128: return launch_decode_d<128>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace attn

// ---------------------------------------------------------------------------
// Decode without any device allocation by the caller.
//
// Some callers cannot call cudaMalloc at the point where they decode: code that
// runs inside a memory pool or allocator that forbids nested allocation, a
// real-time serving loop that must not take the allocator's lock or risk an
// out-of-memory error mid-step, or a host that only hands over input and output
// buffers.  For them the chunk partials live in a fixed array in this library's
// own device memory.  Every GPU that loads the library holds this array until
// the process exits.  All calls share it: its contents are whatever the last
// call left.  Nothing in it needs clearing: a call that completes normally
// writes every slot it later reads.  A split CTA whose bounded wait runs out
// returns without writing its partial, so the merge of that call may read an
// earlier call's partial; the call's status (ATTN_ERR_DEVICE_TIMEOUT) already
// marks its result invalid.  Calls that overlap on the GPU (different streams,
// or different host threads without ordering) race on it.
namespace {

constexpr size_t kNoAllocScratchBytes = 12u << 20;  // 12 MiB: e.g. B=32, H=32, d=128, 8192-token contexts
static __device__ __align__(256) float g_decode_scratch[kNoAllocScratchBytes / sizeof(float)];

constexpr int kMaxScratchDevices = 64;
float *g_scratch_ptr[kMaxScratchDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device.  Looked up once per
// device (the first call on each device does it; make that call before any
// stream capture).  In host code g_decode_scratch names a host-side stand-in,
// not device memory, so only this address may be handed to a kernel.
cudaError_t scratch_address(float **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxScratchDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        if (!p) return cudaErrorInvalidSymbol;
        g_scratch_ptr[dev] = static_cast<float *>(p);
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

namespace attn {

size_t decode_noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

cudaError_t launch_decode_noalloc(const DecodeArgs &a_in, cudaStream_t stream) {
    float *scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) return e;
    DecodeArgs a = a_in;
    a.workspace = scratch;
    return launch_decode(a, stream);
}

}  // namespace attn

// ---------------------------------------------------------------------------
// Self-test of the bounded-wait machinery: one warp waits on an mbarrier that
// nothing ever arrives on.  The wait gives up after its time limit, raises the
// device status word (site 250) and the kernel returns; the context stays usable.
namespace attn {
namespace {
__global__ void selftest_wait_kernel(int *status) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        WaitCtx wc{&abort_flag, status};
        (void)mbar_wait(&bar, 0, wc, 250);
    }
    __syncthreads();
}
}  // namespace

cudaError_t launch_selftest_wait(int *status, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(status);
    return cudaGetLastError();
}
}  // namespace attn
