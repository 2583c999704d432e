// prefill.cu -- FlashAttention-style prefill forward on the sm_103a tensor cores.
//
// The method (NanoInfer README, Flash Attention bullets; gpu-inference blog,
// section 02; llm-kernel-lib README, kernel 1; Kernel-Inference-Engine README,
// tile-loop flowchart): a 128-row Q tile stays resident while 128-key K/V tiles
// stream past it; per tile S = Q K^T * scale, mask, online softmax with a
// running max m and normaliser l, O rescaled by exp(m_old - m_new), O += P V;
// at the end O / l and LSE = m + ln l are stored.  The score matrix never
// reaches global memory, and K/V tiles wholly above the causal diagonal (or
// past the key-padding length) are never visited.
//
// GB300 mapping (one CTA = one (batch, head, 128-row query tile), 6 warps):
//   warp 4     TMA producer: Q once, then K and V tiles into 2-stage rings
//              (128-byte swizzled boxes of 128 rows x 64 columns).
//   warp 5     TMEM owner and MMA issuer (one thread): S_j = Q K_j^T into one
//              of two TMEM score buffers (128 lanes x 128 fp32 columns), and
//              O += P_j V_j into a TMEM accumulator (128 lanes x d columns),
//              each followed by tcgen05.commit onto an mbarrier.
//   warps 0-3  softmax: thread r owns query row r (TMEM lane r).  It loads its
//              128 scores from TMEM, masks, takes the row max, and keeps the
//              reference max stale until the new max exceeds it by more than
//              2^8 (O and l always share the same reference, so the final O / l
//              is unchanged; only then is O in TMEM rescaled).  P = 2^(x - m)
//              goes to shared memory as bf16 in the 128-byte swizzled K-major
//              layout the MMA reads.  The same warps run the epilogue.
// S_{j+1} runs on the tensor core while the softmax warps work on S_j.
#include <cmath>
#include <mutex>

#include "launch.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per tile
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr int kThreads = 192;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kBoxBytes = 128 * 64 * 2;  // one 128-row x 64-column bf16 box (16 KB)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 2^8

struct PrefillParams {
    __nv_bfloat16 *o;
    float *lse;
    const int32_t *kv_lens;
    int *status;
    int B, H, Nq, Nkv, causal, n_qtiles;
    float scale_log2;
};

template <int D>
struct alignas(1024) PrefillSmem {
    __nv_bfloat16 q[kBM * D];               // D/64 boxes
    __nv_bfloat16 k[kKStages][kBN * D];     // D/64 boxes each
    __nv_bfloat16 v[kVStages][kBN * D];     // D/64 boxes each
    __nv_bfloat16 p[kBM * kBN];             // 2 boxes (keys 0-63, 64-127)
    uint64_t q_full;
    uint64_t k_full[kKStages], k_empty[kKStages];
    uint64_t v_full[kVStages], v_empty[kVStages];
    uint64_t s_full[2];
    uint64_t p_full;
    uint64_t o_done;
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

// ------------------------------------------------------------------ producer
template <int D>
__device__ void run_producer(PrefillSmem<D> &sm, const CUtensorMap *tmQ, const CUtensorMap *tmK,
                             const CUtensorMap *tmV, int bh, int q0, int n_tiles, WaitCtx wc) {
    constexpr int kBoxes = D / 64;
    prefetch_tensormap(tmQ);
    prefetch_tensormap(tmK);
    prefetch_tensormap(tmV);
    mbar_arrive_expect_tx(&sm.q_full, kBoxes * kBoxBytes);
#pragma unroll
    for (int i = 0; i < kBoxes; ++i) tma_load_3d(sm.q + i * (kBM * 64), tmQ, &sm.q_full, i * 64, q0, bh);
    int k_fills = 0, v_fills = 0;
    for (int j = 0; j < n_tiles; ++j) {
        const int ks = j % kKStages, kuse = j / kKStages;
        if (kuse > 0 && !mbar_wait(&sm.k_empty[ks], (uint32_t)((kuse - 1) & 1), wc, 1)) break;
        mbar_arrive_expect_tx(&sm.k_full[ks], kBoxes * kBoxBytes);
#pragma unroll
        for (int i = 0; i < kBoxes; ++i)
            tma_load_3d(sm.k[ks] + i * (kBN * 64), tmK, &sm.k_full[ks], i * 64, j * kBN, bh);
        ++k_fills;
        const int vs = j % kVStages, vuse = j / kVStages;
        if (vuse > 0 && !mbar_wait(&sm.v_empty[vs], (uint32_t)((vuse - 1) & 1), wc, 2)) break;
        mbar_arrive_expect_tx(&sm.v_full[vs], kBoxes * kBoxBytes);
#pragma unroll
        for (int i = 0; i < kBoxes; ++i)
            tma_load_3d(sm.v[vs] + i * (kBN * 64), tmV, &sm.v_full[vs], i * 64, j * kBN, bh);
        ++v_fills;
    }
    if (*wc.abort_flag) {
        // unwinding: let every copy still in flight land before the CTA exits
        WaitCtx drain{nullptr, wc.status};
        (void)mbar_wait(&sm.q_full, 0, drain, 90);
        for (int f = (k_fills > kKStages ? k_fills - kKStages : 0); f < k_fills; ++f)
            (void)mbar_wait(&sm.k_full[f % kKStages], (uint32_t)((f / kKStages) & 1), drain, 91);
        for (int f = (v_fills > kVStages ? v_fills - kVStages : 0); f < v_fills; ++f)
            (void)mbar_wait(&sm.v_full[f % kVStages], (uint32_t)((f / kVStages) & 1), drain, 92);
    }
}

// ------------------------------------------------------------------ MMA issuer
template <int D>
__device__ void run_mma(PrefillSmem<D> &sm, uint32_t tmem, int n_tiles, WaitCtx wc) {
    constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN, false, false);
    constexpr uint32_t idPV = idesc_bf16_f32(kBM, D, false, true);
    const uint32_t tO = tmem + 256;
    const uint32_t q_addr = smem_u32(sm.q);
    const uint32_t p_addr = smem_u32(sm.p);

    auto issue_S = [&](int j) -> bool {
        const int ks = j % kKStages;
        if (!mbar_wait(&sm.k_full[ks], (uint32_t)((j / kKStages) & 1), wc, 10)) return false;
        tc_fence_after_sync();
        const uint32_t k_addr = smem_u32(sm.k[ks]);
        const uint32_t tS = tmem + (uint32_t)((j & 1) * kBN);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (uint32_t)((kk >> 2) * kBoxBytes + (kk & 3) * 32);
            tc_mma_ss(tS, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(k_addr + off, 16, 1024), idS,
                      kk > 0 ? 1u : 0u);
        }
        tc_commit(&sm.s_full[j & 1]);
        tc_commit(&sm.k_empty[ks]);
        return true;
    };

    if (mbar_wait(&sm.q_full, 0, wc, 11) && issue_S(0)) {
        for (int j = 0; j < n_tiles; ++j) {
            if (j + 1 < n_tiles && !issue_S(j + 1)) break;
            if (!mbar_wait(&sm.p_full, (uint32_t)(j & 1), wc, 12)) break;
            const int vs = j % kVStages;
            if (!mbar_wait(&sm.v_full[vs], (uint32_t)((j / kVStages) & 1), wc, 13)) break;
            tc_fence_after_sync();
            const uint32_t v_addr = smem_u32(sm.v[vs]);
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk) {
                // A = P (K-major, keys contiguous); B = V (MN-major: d contiguous, 16 keys = 2048 B)
                const uint32_t a_off = (uint32_t)((kk >> 2) * kBoxBytes + (kk & 3) * 32);
                const uint32_t b_off = (uint32_t)(kk * 16 * 128);
                tc_mma_ss(tO, sdesc_sw128(p_addr + a_off, 16, 1024), sdesc_sw128(v_addr + b_off, kBoxBytes, 1024),
                          idPV, (j > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(&sm.o_done);
            tc_commit(&sm.v_empty[vs]);
        }
    }
    // wait (bounded) until every MMA issued above has finished with TMEM and smem
    tc_commit(&sm.drain);
    WaitCtx drain{nullptr, wc.status};
    (void)mbar_wait(&sm.drain, 0, drain, 19);
}

// ------------------------------------------------------------------ softmax + epilogue
template <int D>
__device__ void run_softmax(PrefillSmem<D> &sm, const PrefillParams &p, uint32_t tmem, int bh, int q0,
                            int n_tiles, int kv_end, WaitCtx wc) {
    const int t = threadIdx.x;  // 0..127 = query row in the tile = TMEM lane
    const int warp = t >> 5;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const int row = q0 + t;
    const int delta = p.Nkv - p.Nq;
    const float c = p.scale_log2;

    float m_ref = -INFINITY;  // reference max (log2 domain) shared by l and O
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
        // every decision that guards a .sync.aligned tcgen05 instruction is made warp-uniform
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.s_full[j & 1], (uint32_t)((j >> 1) & 1), wc, 20))) {
            ok = false;
            break;
        }
        tc_fence_after_sync();
        uint32_t s[4][32];
        const uint32_t tS = lane_base + (uint32_t)((j & 1) * kBN);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(tS + cc * 32, s[cc]);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_wait_ld(s[cc]);

        // mask keys that are invalid for this row (only tiles that straddle a boundary)
        const int key0 = j * kBN;
        const bool need_mask = (key0 + kBN > kv_end) || (p.causal && key0 + kBN - 1 > q0 + delta);
        if (need_mask) {
            int lim = kv_end;
            if (p.causal) lim = min(lim, row + delta + 1);
            const int nvalid = lim - key0;  // keys key0 .. key0+nvalid-1 are valid
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (cc * 32 + i >= nvalid) s[cc][i] = __float_as_uint(-INFINITY);
        }
        float mx = -INFINITY;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
            for (int i = 0; i < 32; ++i) mx = fmaxf(mx, __uint_as_float(s[cc][i]));
        const float m_cand = mx * c;  // -inf stays -inf (c > 0)
        const bool resc = m_cand > m_ref + kRescaleThreshold;
        float alpha = 1.f;
        if (resc) {
            alpha = ex2_approx(m_ref - m_cand);  // 0 when m_ref = -inf
            m_ref = m_cand;
            l *= alpha;
        }
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;

        // P = 2^(s*c - m_use), packed to bf16 pairs in place; l sums the fp32 values
        // (the exact normaliser the log-sum-exp needs).
        float rowsum = 0.f;
        uint32_t pk[64];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const float p0 = ex2_approx(fmaf(__uint_as_float(s[cc][i]), c, -m_use));
                const float p1 = ex2_approx(fmaf(__uint_as_float(s[cc][i + 1]), c, -m_use));
                rowsum += p0 + p1;
                pk[cc * 16 + i / 2] = pack_bf16x2(p0, p1);
            }
        l += rowsum;

        // O and the P buffer are free once PV(j-1) has completed
        if (j > 0) {
            if (!__all_sync(0xffffffffu, mbar_wait(&sm.o_done, (uint32_t)((j - 1) & 1), wc, 21))) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            if (__any_sync(0xffffffffu, resc)) {
                const uint32_t tO = lane_base + 256;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t ov[32];
                    tmem_ld32(tO + cc * 32, ov);
                    tmem_wait_ld(ov);
#pragma unroll
                    for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
                    tmem_st32(tO + cc * 32, ov);
                }
                tmem_wait_st();
            }
        }
        // P row -> shared memory, 128-byte swizzle: 16-byte chunk ch of row t lands at chunk ch ^ (t & 7)
        {
            const uint32_t pbase = smem_u32(sm.p) + (uint32_t)t * 128;
#pragma unroll
            for (int c16 = 0; c16 < 16; ++c16) {
                const uint32_t box = (uint32_t)(c16 >> 3) * kBoxBytes;
                const uint32_t ch = (uint32_t)((c16 & 7) ^ (t & 7));
                st_shared_v4(pbase + box + ch * 16, pk[c16 * 4 + 0], pk[c16 * 4 + 1], pk[c16 * 4 + 2],
                             pk[c16 * 4 + 3]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        mbar_arrive(&sm.p_full);
    }

    // epilogue: O / l -> bf16, LSE = ln2 * (m_ref + log2 l)
    if (ok && n_tiles > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.o_done, (uint32_t)((n_tiles - 1) & 1), wc, 22))) ok = false;
        else tc_fence_after_sync();
    }
    if (!ok) return;
    const bool have = (n_tiles > 0) && (l > 0.f);
    const float inv_l = have ? 1.f / l : 0.f;
    __nv_bfloat16 *orow = p.o + ((size_t)bh * p.Nq + row) * D;
    const bool store = row < p.Nq;
#pragma unroll
    for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t ov[32];
        if (n_tiles > 0) {
            tmem_ld32(lane_base + 256 + cc * 32, ov);
            tmem_wait_ld(ov);
        }
        if (store) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                pk[i] = have ? pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l)
                             : 0u;
            uint4 *dst = reinterpret_cast<uint4 *>(orow + cc * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
    }
    if (store && p.lse) p.lse[(size_t)bh * p.Nq + row] = have ? kLn2 * (m_ref + __log2f(l)) : -INFINITY;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
    extern __shared__ uint8_t smem_raw[];
    PrefillSmem<D> &sm =
        *reinterpret_cast<PrefillSmem<D> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BH = p.B * p.H;
    const int qt = p.n_qtiles - 1 - (int)(blockIdx.x / BH);  // heaviest (last) query tiles first
    const int bh = (int)(blockIdx.x % BH);
    const int b = bh / p.H;
    const int q0 = qt * kBM;
    int kv_end = p.Nkv;
    if (p.kv_lens) kv_end = min(max(p.kv_lens[b], 0), p.Nkv);
    int limit = kv_end;  // keys < limit may be valid for some row of this tile
    if (p.causal) limit = min(limit, min(q0 + kBM, p.Nq) + (p.Nkv - p.Nq));
    const int n_tiles = limit > 0 ? (limit + kBN - 1) / kBN : 0;

    if (threadIdx.x == 0) {
        mbar_init(&sm.q_full, 1);
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&sm.k_full[s], 1);
            mbar_init(&sm.k_empty[s], 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(&sm.v_full[s], 1);
            mbar_init(&sm.v_empty[s], 1);
        }
        mbar_init(&sm.s_full[0], 1);
        mbar_init(&sm.s_full[1], 1);
        mbar_init(&sm.p_full, kBM);
        mbar_init(&sm.o_done, 1);
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sm.tmem_base;
    WaitCtx wc{&sm.abort_flag, p.status};

    if (warp == kProducerWarp) {
        if (lane == 0 && n_tiles > 0) run_producer<D>(sm, &tmQ, &tmK, &tmV, bh, q0, n_tiles, wc);
    } else if (warp == kMmaWarp) {
        if (lane == 0 && n_tiles > 0) run_mma<D>(sm, tmem, n_tiles, wc);
    } else {
        run_softmax<D>(sm, p, tmem, bh, q0, n_tiles, kv_end, wc);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
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
bool encode_qkv_map(CUtensorMap *m, const void *ptr, int BH, int N, int D) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_prefill_d(const PrefillArgs &a, cudaStream_t stream) {
    CUtensorMap tq, tk, tv;
    const int BH = a.B * a.H;
    if (!encode_qkv_map(&tq, a.q, BH, a.Nq, D) || !encode_qkv_map(&tk, a.k, BH, a.Nkv, D) ||
        !encode_qkv_map(&tv, a.v, BH, a.Nkv, D))
        return cudaErrorInvalidValue;
    PrefillParams p;
    p.o = reinterpret_cast<__nv_bfloat16 *>(a.o);
    p.lse = a.lse;
    p.kv_lens = a.kv_lens;
    p.status = a.status;
    p.B = a.B;
    p.H = a.H;
    p.Nq = a.Nq;
    p.Nkv = a.Nkv;
    p.causal = a.causal;
    p.n_qtiles = (a.Nq + kBM - 1) / kBM;
    p.scale_log2 = a.scale * kLog2e;
    const size_t smem = sizeof(PrefillSmem<D>) + 1024;
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)((size_t)p.n_qtiles * BH);
    prefill_kernel<D><<<grid, kThreads, smem, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t stream) {
    if (a.d == 128) return launch_prefill_d<128>(a, stream);
    return launch_prefill_d<64>(a, stream);
}

}  // namespace attn
