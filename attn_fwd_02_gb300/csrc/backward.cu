// backward.cu -- attention backward on the sm_103a tensor cores.
//
// The method (gpu-inference blog, section 02 "FlashAttention-2 in Triton"): the backward keeps
// no probability matrix; it recomputes the probabilities tile by tile from the log-sum-exp the
// forward saved, and it is split into three kernels: a pass that computes the row term
// D_i = dO_i . O_i, a dK/dV kernel and a dQ kernel.  With P = exp(s - LSE) on the valid keys
// (s = scale q.k), dP = dO V^T and dS = P * (dP - D):
//     dV = P^T dO,   dK = scale dS^T Q,   dQ = scale dS K.
//
// GB300 mapping of the two tile kernels (d in {32, 64, 80, 96, 128}):
//   * One CTA owns a 128-row tile of what it accumulates (dK and dV of 128 keys, or dQ of 128
//     queries) in TMEM, and streams the other side's 128-row tiles through a 2-slot TMA ring
//     (128-byte swizzled boxes of 128 rows x 64 columns).
//   * 10 warps.  Warps 0-7 are two compute warpgroups: thread r of warpgroup w owns TMEM lane r
//     (row r of the CTA's own tile) and columns 64w .. 64w+63 of each 128 x 128 score tile.
//     Warp 8 loads; warp 9 owns the TMEM and one of its threads issues every MMA.
//   * dK/dV: S^T = K Q^T and dP^T = V dO^T land in TMEM with lane = key.  The warpgroups write
//     P^T and dS^T (bf16 pairs) back over the columns they read, where dV += P^T dO and
//     dK += dS^T Q take them as the A operand straight from TMEM.  Each Q or dO tile is the
//     K-major B operand of a score product and the MN-major B operand of an accumulation.
//     TMEM: S^T 128 | dP^T 128 | dV d | dK d columns.
//   * dQ: S = Q K^T and dP = dO V^T with lane = query; dS (bf16) over dP feeds dQ += dS K.
//     TMEM: S 128 | dP 128 | dQ d columns.
//   * Issue order per step j.  dK/dV: dV(j), S^T(j+1), then dK(j), dP^T(j+1).  dQ: S(j+1),
//     then dQ(j), dP(j+1).  The tensor core computes the next scores while the warpgroups turn
//     dP(j) into dS(j), and the next dP while they turn S(j+1) into P(j+1).  The MMAs of one
//     thread run in issue order, so a product that overwrites a TMEM buffer never overtakes the
//     earlier product that reads the same columns as its operand.
#include <cmath>

#include "launch.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kT = 128;  // rows of every tile (queries or keys)
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kStages = 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kBoxBytes = 128 * 64 * 2;  // one 128-row x 64-column bf16 box
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;
// Tiles are padded to 64 (d <= 64) or 128 columns of 64-column TMA boxes, which read zeros past d:
// the score products run over d/16 k-steps and the accumulations over N = d columns, so the padding
// costs shared memory only.  Accumulators in TMEM sit at padded column offsets.
template <int D> constexpr int kBPad = D <= 64 ? 64 : 128;
template <int D> constexpr int kBBoxes = kBPad<D> / 64;
// dQ columns of the first warpgroup (the second takes the rest): halves in multiples of 16
template <int D> constexpr int kDqSplit = ((D / 16 + 1) / 2) * 16;

struct BwdParams {
    const float *lse, *dterm;
    __nv_bfloat16 *dq, *dk, *dv;
    const int32_t *kv_lens;
    int *status;
    int B, Hq, Hkv, group, Nq, Nkv, causal;
    int units_per_head;   // query tiles (dQ kernel) or key tiles (dK/dV kernel) of one head
    int heads_per_chunk;  // heads whose streamed operands share L2 at a time
    float scale, scale_log2;
};

// CTA order (as in the forward): heads in chunks small enough that the chunk's streamed tiles
// stay in L2; inside a chunk, unit levels in order (level 0 = the heaviest unit of a head
// under the causal mask) across the chunk's heads.
__device__ __forceinline__ void unit_of(const BwdParams &p, int n_heads, int &head, int &level) {
    const int per_chunk = p.heads_per_chunk * p.units_per_head;
    const int chunk = (int)(blockIdx.x / per_chunk);
    const int h0 = chunk * p.heads_per_chunk;
    const int heads = min(p.heads_per_chunk, n_heads - h0);
    const int in_chunk = (int)(blockIdx.x % per_chunk);
    level = in_chunk / heads;
    head = h0 + in_chunk % heads;
}

__device__ __forceinline__ int kv_end_for(const BwdParams &p, int b) {
    return p.kv_lens ? min(max(p.kv_lens[b], 0), p.Nkv) : p.Nkv;
}

// 128 x 128 score tile: D[tmem] = A B^T over the head dimension (both operands K-major tiles).
template <int D>
__device__ __forceinline__ void mma_scores(uint32_t d_tmem, const __nv_bfloat16 *a, const __nv_bfloat16 *b) {
    constexpr uint32_t id = idesc_bf16_f32(kT, kT, false, false);
    const uint64_t da = sdesc_sw128(smem_u32(a), 16, 1024), db = sdesc_sw128(smem_u32(b), 16, 1024);
    static_assert(kBoxBytes == 16384, "k-step layout of the grouped issue");
    tc_mma_ss_ksteps<D / 16>(d_tmem, da, db, id, 0u);
}

// 128 x d accumulation: D[tmem] (+)= A[tmem] B, A = 128 x 128 bf16 written by the two warpgroups
// (columns 0-31 and 64-95 of a_tmem hold the bf16 pairs of k-indices 0-63 and 64-127), B = a
// 128-row tile read MN-major (k-index = tile row).
template <int D>
__device__ __forceinline__ void mma_accum(uint32_t d_tmem, uint32_t a_tmem, const __nv_bfloat16 *b, bool first) {
    constexpr uint32_t id = idesc_bf16_f32(kT, D, false, true);
    const uint64_t db = sdesc_sw128(smem_u32(b), kBoxBytes, 1024);
    static_assert(kT / 16 == 8, "one group of eight k-steps");
    tc_mma_ts_k8_halves(d_tmem, a_tmem, db, id, first ? 0u : 1u);
}

// 64 TMEM columns of this thread's lane -> registers.
__device__ __forceinline__ void load64(uint32_t taddr, uint32_t (&x)[2][32]) {
    tmem_ld32(taddr, x[0]);
    tmem_ld32(taddr + 32, x[1]);
    tmem_wait_ld(x[0]);
    tmem_wait_ld(x[1]);
}

// Writes NCOLS (a multiple of 16) columns of this thread's row of an fp32 TMEM accumulator,
// times `mul`, as bf16 to dst (`store` false skips the write).  Zeros if !have.
template <int NCOLS>
__device__ __forceinline__ void store_rows(uint32_t tacc, bool have, bool store, float mul, __nv_bfloat16 *dst) {
    static_assert(NCOLS % 16 == 0, "16-column steps");
#pragma unroll
    for (int cc = 0; cc < NCOLS / 32; ++cc) {
        uint32_t v[32];
        if (have) {
            tmem_ld32(tacc + cc * 32, v);
            tmem_wait_ld(v);
        }
        if (store) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                pk[i] = have ? pack_bf16x2(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul) : 0u;
            uint4 *o = reinterpret_cast<uint4 *>(dst + cc * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) o[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
    }
    if constexpr (NCOLS % 32 != 0) {  // the last 16 columns
        constexpr int c0 = NCOLS / 32 * 32;
        uint32_t v[16];
        if (have) {
            tmem_ld16(tacc + c0, v);
            tmem_wait_ld16(v);
        }
        if (store) {
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                pk[i] = have ? pack_bf16x2(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul) : 0u;
            uint4 *o = reinterpret_cast<uint4 *>(dst + c0);
            o[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            o[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
    }
}

// ================================================================== row term D = rowsum(dO * O)
// kTpr threads per row (d / 8 rounded up to a power of two), one 16-byte load of O and of dO each
// for the threads whose 8 columns lie inside d, then a shuffle reduction.
template <int D> constexpr int kRowThreads = D / 8 <= 4 ? 4 : (D / 8 <= 8 ? 8 : 16);
template <int D>
__global__ void __launch_bounds__(256) bwd_rowdot_kernel(const __nv_bfloat16 *o, const __nv_bfloat16 *dout,
                                                         float *dterm, long long rows) {
    constexpr int kTpr = kRowThreads<D>;
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long row = gid / kTpr;
    const int part = (int)(gid % kTpr);
    float acc = 0.f;
    if (row < rows && part * 8 < D) {
        const uint4 a = *reinterpret_cast<const uint4 *>(o + row * D + part * 8);
        const uint4 b = *reinterpret_cast<const uint4 *>(dout + row * D + part * 8);
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&av[i]));
            const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&bv[i]));
            acc = fmaf(fa.x, fb.x, acc);
            acc = fmaf(fa.y, fb.y, acc);
        }
    }
#pragma unroll
    for (int off = kTpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
    if (row < rows && part == 0) dterm[row] = acc;
}

// ================================================================== dK / dV
template <int D>
struct alignas(1024) DkvSmem {
    __nv_bfloat16 k[kT * kBPad<D>];              // the CTA's 128 keys (kBBoxes boxes)
    __nv_bfloat16 v[kT * kBPad<D>];
    __nv_bfloat16 q[kStages][kT * kBPad<D>];     // streamed query tiles
    __nv_bfloat16 dout[kStages][kT * kBPad<D>];  // and their upstream gradients
    float nlse2[kStages][kT];             // minus the log2-domain LSE of each streamed query (0 past Nq)
    float dterm[kStages][kT];             // row term D of each streamed query (0 past Nq)
    uint64_t kv_full;
    uint64_t u_full[kStages], u_empty[kStages];
    uint64_t s_full, p_full, dp_full, ds_full, acc_done, drain;
    uint32_t tmem_base;
    int abort_flag;
};

// Query tiles a key tile [k0, k0+128) must visit: queries i >= k0 - delta can see its keys
// under the causal mask (query i sees key j iff j <= i + delta).
__device__ __forceinline__ void dkdv_range(const BwdParams &p, int k0, int kv_end, int delta, int &qi_start,
                                           int &nqt) {
    const int n_qt = (p.Nq + kT - 1) / kT;
    qi_start = 0;
    nqt = 0;
    if (k0 >= kv_end) return;
    if (p.causal) {
        const int first = k0 - delta;
        if (first >= p.Nq) return;
        qi_start = first > 0 ? first / kT : 0;
    }
    nqt = n_qt - qi_start;
}

template <int D>
__device__ void dkdv_producer(DkvSmem<D> &sm, const BwdParams &p, const CUtensorMap *tmQ, const CUtensorMap *tmdO,
                              const CUtensorMap *tmK, const CUtensorMap *tmV, int b, int hkv, int bh_kv, int k0,
                              int qi_start, int nqt, int n, WaitCtx wc) {
    constexpr int kBoxes = kBBoxes<D>;
    const int lane = threadIdx.x & 31;
    if (lane == 0) {
        prefetch_tensormap(tmQ);
        prefetch_tensormap(tmdO);
        mbar_arrive_expect_tx(&sm.kv_full, 2 * kBoxes * kBoxBytes);
#pragma unroll
        for (int i = 0; i < kBoxes; ++i) {
            tma_load_3d(sm.k + i * (kT * 64), tmK, &sm.kv_full, i * 64, k0, bh_kv);
            tma_load_3d(sm.v + i * (kT * 64), tmV, &sm.kv_full, i * 64, k0, bh_kv);
        }
    }
    // the row statistics of unit u's 128 queries, four per lane (plain loads, zeros past Nq); they
    // are loaded one unit ahead so their latency hides behind the ring wait
    auto load_stats = [&](int u, float (&l4)[4], float (&d4)[4]) {
        const int bh_q = b * p.Hq + hkv * p.group + u / nqt;
        const int q0 = (qi_start + u % nqt) * kT;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int row = q0 + lane * 4 + t;
            l4[t] = 0.f;
            d4[t] = 0.f;
            if (row < p.Nq) {
                l4[t] = p.lse[(size_t)bh_q * p.Nq + row];
                d4[t] = p.dterm[(size_t)bh_q * p.Nq + row];
            }
        }
    };
    float l4n[4], d4n[4];
    load_stats(0, l4n, d4n);
    int fills = 0;
    for (int u = 0; u < n; ++u) {
        const int slot = u % kStages, use = u / kStages;
        if (use > 0 && !__all_sync(kFull, mbar_wait(&sm.u_empty[slot], (uint32_t)((use - 1) & 1), wc, 60))) break;
        const int g = u / nqt, qi = qi_start + u % nqt;
        const int bh_q = b * p.Hq + hkv * p.group + g;
        const int q0 = qi * kT;
        *reinterpret_cast<float4 *>(&sm.nlse2[slot][lane * 4]) =
            make_float4(l4n[0] * -kLog2e, l4n[1] * -kLog2e, l4n[2] * -kLog2e, l4n[3] * -kLog2e);
        *reinterpret_cast<float4 *>(&sm.dterm[slot][lane * 4]) = make_float4(d4n[0], d4n[1], d4n[2], d4n[3]);
        if (u + 1 < n) load_stats(u + 1, l4n, d4n);
        if (lane == 0) {
            mbar_arrive_expect_tx(&sm.u_full[slot], 2 * kBoxes * kBoxBytes);
#pragma unroll
            for (int i = 0; i < kBoxes; ++i) {
                tma_load_3d(sm.q[slot] + i * (kT * 64), tmQ, &sm.u_full[slot], i * 64, q0, bh_q);
                tma_load_3d(sm.dout[slot] + i * (kT * 64), tmdO, &sm.u_full[slot], i * 64, q0, bh_q);
            }
        } else {
            mbar_arrive(&sm.u_full[slot]);
        }
        ++fills;
    }
    if (lane == 0 && *wc.abort_flag) {
        // unwinding: let every copy still in flight land before the CTA exits
        WaitCtx drain{nullptr, wc.status};
        (void)mbar_wait(&sm.kv_full, 0, drain, 61);
        for (int f = (fills > kStages ? fills - kStages : 0); f < fills; ++f)
            (void)mbar_wait(&sm.u_full[f % kStages], (uint32_t)((f / kStages) & 1), drain, 62);
    }
}

template <int D>
__device__ void dkdv_mma(DkvSmem<D> &sm, uint32_t tmem, int n, WaitCtx wc) {
    const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + kBPad<D>;
    bool ok = mbar_wait(&sm.kv_full, 0, wc, 63) && mbar_wait(&sm.u_full[0], 0, wc, 64);
    if (ok) {
        tc_fence_after_sync();
        mma_scores<D>(tS, sm.k, sm.q[0]);
        tc_commit(&sm.s_full);
        mma_scores<D>(tdP, sm.v, sm.dout[0]);
        tc_commit(&sm.dp_full);
        for (int j = 0; j < n; ++j) {
            const int slot = j % kStages;
            if (!(ok = mbar_wait(&sm.p_full, (uint32_t)(j & 1), wc, 65))) break;
            tc_fence_after_sync();
            mma_accum<D>(tdV, tS, sm.dout[slot], j == 0);  // dV += P^T dO
            if (j + 1 < n) {
                const int u = j + 1;
                if (!(ok = mbar_wait(&sm.u_full[u % kStages], (uint32_t)((u / kStages) & 1), wc, 66))) break;
                mma_scores<D>(tS, sm.k, sm.q[u % kStages]);  // S^T(j+1), after dV(j) read P^T(j)
                tc_commit(&sm.s_full);
            }
            if (!(ok = mbar_wait(&sm.ds_full, (uint32_t)(j & 1), wc, 67))) break;
            tc_fence_after_sync();
            mma_accum<D>(tdK, tdP, sm.q[slot], j == 0);  // dK += dS^T Q
            tc_commit(&sm.u_empty[slot]);
            if (j == n - 1) tc_commit(&sm.acc_done);
            if (j + 1 < n) {
                mma_scores<D>(tdP, sm.v, sm.dout[(j + 1) % kStages]);  // dP^T(j+1), after dK(j) read dS^T(j)
                tc_commit(&sm.dp_full);
            }
        }
    }
    tc_commit(&sm.drain);
    WaitCtx drain{nullptr, wc.status};
    (void)mbar_wait(&sm.drain, 0, drain, 68);
}

template <int D>
__device__ void dkdv_compute(DkvSmem<D> &sm, const BwdParams &p, uint32_t tmem, int w, int bh_kv, int k0,
                             int kv_end, int delta, int qi_start, int nqt, int n, WaitCtx wc) {
    const int r = threadIdx.x & 127;
    const uint32_t lane_base = tmem + ((uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16);
    const uint32_t tS = lane_base + (uint32_t)(w * 64);
    const uint32_t tdP = lane_base + 128u + (uint32_t)(w * 64);
    const int key = k0 + r;
    const bool key_ok = key < kv_end;
    const uint64_t c2 = f32x2_pack(p.scale_log2, p.scale_log2);
    bool ok = true;
    for (int j = 0; j < n; ++j) {
        const int slot = j % kStages;
        const int col0 = (qi_start + j % nqt) * kT + w * 64;  // query of this half's column 0
        // valid columns lo <= c < hi: query < Nq, key < kv_end, and key <= query + delta if causal
        int lo = 0, hi = min(64, p.Nq - col0);
        if (p.causal) lo = max(0, key - delta - col0);
        if (!key_ok) hi = 0;
        const bool need_mask = lo > 0 || hi < 64;

        // The columns' statistics are read before the score waits so that their latency hides
        // behind them.  The producer wrote them before arriving on the unit's full barrier; waiting
        // on that barrier (without arriving) orders these reads after its writes.  The slot cannot
        // be refilled before this step ends (the refill waits for dK(j), which needs this step's dS).
        if (!__all_sync(kFull, mbar_wait(&sm.u_full[slot], (uint32_t)((j / kStages) & 1), wc, 73))) {
            ok = false;
            break;
        }
        float4 L4[16];
        const float4 *l2 = reinterpret_cast<const float4 *>(sm.nlse2[slot] + w * 64);
#pragma unroll
        for (int i = 0; i < 16; ++i) L4[i] = l2[i];
        if (!__all_sync(kFull, mbar_wait(&sm.s_full, (uint32_t)(j & 1), wc, 70))) {
            ok = false;
            break;
        }
        tc_fence_after_sync();
        uint32_t x[2][32];
        load64(tS, x);
        // P^T = 2^(s * scale * log2e - lse2): bf16 pairs over the scores, fp32 kept in x
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const float4 L = L4[(h * 32 + i) / 4];
                const uint64_t e01 = f32x2_fma(f32x2_pack(__uint_as_float(x[h][i]), __uint_as_float(x[h][i + 1])), c2,
                                               f32x2_pack(L.x, L.y));
                const uint64_t e23 = f32x2_fma(f32x2_pack(__uint_as_float(x[h][i + 2]), __uint_as_float(x[h][i + 3])),
                                               c2, f32x2_pack(L.z, L.w));
                float e[4];
                f32x2_unpack(e01, e[0], e[1]);
                f32x2_unpack(e23, e[2], e[3]);
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    float pv = ex2_approx(e[t]);
                    if (need_mask) {
                        const int c = h * 32 + i + t;
                        pv = (c >= lo && c < hi) ? pv : 0.f;
                    }
                    x[h][i + t] = __float_as_uint(pv);
                }
                pk[i / 2] = pack_bf16x2(__uint_as_float(x[h][i]), __uint_as_float(x[h][i + 1]));
                pk[i / 2 + 1] = pack_bf16x2(__uint_as_float(x[h][i + 2]), __uint_as_float(x[h][i + 3]));
            }
            tmem_st16(tS + (uint32_t)(h * 16), pk);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        mbar_arrive(&sm.p_full);

        float4 D4[16];
        const float4 *dd = reinterpret_cast<const float4 *>(sm.dterm[slot] + w * 64);
#pragma unroll
        for (int i = 0; i < 16; ++i) D4[i] = dd[i];
        if (!__all_sync(kFull, mbar_wait(&sm.dp_full, (uint32_t)(j & 1), wc, 71))) {
            ok = false;
            break;
        }
        tc_fence_after_sync();
        uint32_t y[2][32];
        load64(tdP, y);
        // dS^T = P^T * (dP^T - D): bf16 pairs over dP^T
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const float4 Dv = D4[(h * 32 + i) / 4];
                const float s0 = __uint_as_float(x[h][i]) * (__uint_as_float(y[h][i]) - Dv.x);
                const float s1 = __uint_as_float(x[h][i + 1]) * (__uint_as_float(y[h][i + 1]) - Dv.y);
                const float s2 = __uint_as_float(x[h][i + 2]) * (__uint_as_float(y[h][i + 2]) - Dv.z);
                const float s3 = __uint_as_float(x[h][i + 3]) * (__uint_as_float(y[h][i + 3]) - Dv.w);
                pk[i / 2] = pack_bf16x2(s0, s1);
                pk[i / 2 + 1] = pack_bf16x2(s2, s3);
            }
            tmem_st16(tdP + (uint32_t)(h * 16), pk);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        mbar_arrive(&sm.ds_full);
    }

    if (ok && n > 0) {
        if (!__all_sync(kFull, mbar_wait(&sm.acc_done, 0, wc, 72))) ok = false;
        else tc_fence_after_sync();
    }
    if (!ok) return;
    // warpgroup 0 writes dV, warpgroup 1 writes dK (times scale); rows past Nkv are not stored
    const bool store = key < p.Nkv;
    __nv_bfloat16 *dst = (w == 0 ? p.dv : p.dk) + ((size_t)bh_kv * p.Nkv + (store ? key : 0)) * D;
    store_rows<D>(lane_base + 256u + (uint32_t)(w * kBPad<D>), n > 0, store, w == 0 ? 1.f : p.scale, dst);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    DkvSmem<D> &sm =
        *reinterpret_cast<DkvSmem<D> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    int bh_kv, level;
    unit_of(p, p.B * p.Hkv, bh_kv, level);
    const int b = bh_kv / p.Hkv, hkv = bh_kv % p.Hkv;
    const int k0 = level * kT;  // level 0 = key tile 0, seen by the most queries when causal
    const int kv_end = kv_end_for(p, b);
    const int delta = p.Nkv - p.Nq;
    int qi_start, nqt;
    dkdv_range(p, k0, kv_end, delta, qi_start, nqt);
    const int n = nqt * p.group;  // steps: every query tile of every query head of the group

    if (threadIdx.x == 0) {
        mbar_init(&sm.kv_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.u_full[s], 32);
            mbar_init(&sm.u_empty[s], 1);
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.p_full, 256);
        mbar_init(&sm.dp_full, 1);
        mbar_init(&sm.ds_full, 256);
        mbar_init(&sm.acc_done, 1);
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
        if (n > 0) dkdv_producer<D>(sm, p, &tmQ, &tmdO, &tmK, &tmV, b, hkv, bh_kv, k0, qi_start, nqt, n, wc);
    } else if (warp == kMmaWarp) {
        if (lane == 0 && n > 0) dkdv_mma<D>(sm, tmem, n, wc);
    } else {
        dkdv_compute<D>(sm, p, tmem, warp >> 2, bh_kv, k0, kv_end, delta, qi_start, nqt, n, wc);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ================================================================== dQ
template <int D>
struct alignas(1024) DqSmem {
    __nv_bfloat16 q[kT * kBPad<D>];  // the CTA's 128 queries
    __nv_bfloat16 dout[kT * kBPad<D>];
    __nv_bfloat16 k[kStages][kT * kBPad<D>];  // streamed key tiles
    __nv_bfloat16 v[kStages][kT * kBPad<D>];
    uint64_t qd_full;
    uint64_t u_full[kStages], u_empty[kStages];
    uint64_t s_full, s_free, dp_full, ds_full, acc_done, drain;
    uint32_t tmem_base;
    int abort_flag;
};

template <int D>
__device__ void dq_producer(DqSmem<D> &sm, const CUtensorMap *tmQ, const CUtensorMap *tmdO, const CUtensorMap *tmK,
                            const CUtensorMap *tmV, int bh, int bh_kv, int q0, int n, WaitCtx wc) {
    constexpr int kBoxes = kBBoxes<D>;
    prefetch_tensormap(tmK);
    prefetch_tensormap(tmV);
    mbar_arrive_expect_tx(&sm.qd_full, 2 * kBoxes * kBoxBytes);
#pragma unroll
    for (int i = 0; i < kBoxes; ++i) {
        tma_load_3d(sm.q + i * (kT * 64), tmQ, &sm.qd_full, i * 64, q0, bh);
        tma_load_3d(sm.dout + i * (kT * 64), tmdO, &sm.qd_full, i * 64, q0, bh);
    }
    int fills = 0;
    for (int u = 0; u < n; ++u) {
        const int slot = u % kStages, use = u / kStages;
        if (use > 0 && !mbar_wait(&sm.u_empty[slot], (uint32_t)((use - 1) & 1), wc, 80)) break;
        mbar_arrive_expect_tx(&sm.u_full[slot], 2 * kBoxes * kBoxBytes);
#pragma unroll
        for (int i = 0; i < kBoxes; ++i) {
            tma_load_3d(sm.k[slot] + i * (kT * 64), tmK, &sm.u_full[slot], i * 64, u * kT, bh_kv);
            tma_load_3d(sm.v[slot] + i * (kT * 64), tmV, &sm.u_full[slot], i * 64, u * kT, bh_kv);
        }
        ++fills;
    }
    if (*wc.abort_flag) {
        WaitCtx drain{nullptr, wc.status};
        (void)mbar_wait(&sm.qd_full, 0, drain, 81);
        for (int f = (fills > kStages ? fills - kStages : 0); f < fills; ++f)
            (void)mbar_wait(&sm.u_full[f % kStages], (uint32_t)((f / kStages) & 1), drain, 82);
    }
}

template <int D>
__device__ void dq_mma(DqSmem<D> &sm, uint32_t tmem, int n, WaitCtx wc) {
    const uint32_t tS = tmem, tdP = tmem + 128, tdQ = tmem + 256;
    bool ok = mbar_wait(&sm.qd_full, 0, wc, 83) && mbar_wait(&sm.u_full[0], 0, wc, 84);
    if (ok) {
        tc_fence_after_sync();
        mma_scores<D>(tS, sm.q, sm.k[0]);
        tc_commit(&sm.s_full);
        mma_scores<D>(tdP, sm.dout, sm.v[0]);
        tc_commit(&sm.dp_full);
        for (int j = 0; j < n; ++j) {
            const int slot = j % kStages;
            if (j + 1 < n) {
                const int u = j + 1;
                if (!(ok = mbar_wait(&sm.s_free, (uint32_t)(j & 1), wc, 85))) break;
                if (!(ok = mbar_wait(&sm.u_full[u % kStages], (uint32_t)((u / kStages) & 1), wc, 86))) break;
                tc_fence_after_sync();
                mma_scores<D>(tS, sm.q, sm.k[u % kStages]);  // S(j+1): the warpgroups have read S(j)
                tc_commit(&sm.s_full);
            }
            if (!(ok = mbar_wait(&sm.ds_full, (uint32_t)(j & 1), wc, 87))) break;
            tc_fence_after_sync();
            mma_accum<D>(tdQ, tdP, sm.k[slot], j == 0);  // dQ += dS K
            tc_commit(&sm.u_empty[slot]);
            if (j == n - 1) tc_commit(&sm.acc_done);
            if (j + 1 < n) {
                mma_scores<D>(tdP, sm.dout, sm.v[(j + 1) % kStages]);  // dP(j+1), after dQ(j) read dS(j)
                tc_commit(&sm.dp_full);
            }
        }
    }
    tc_commit(&sm.drain);
    WaitCtx drain{nullptr, wc.status};
    (void)mbar_wait(&sm.drain, 0, drain, 88);
}

template <int D>
__device__ void dq_compute(DqSmem<D> &sm, const BwdParams &p, uint32_t tmem, int w, int bh, int q0, int kv_end,
                           int delta, int n, WaitCtx wc) {
    const int r = threadIdx.x & 127;
    const uint32_t lane_base = tmem + ((uint32_t)(((threadIdx.x >> 5) & 3) * 32) << 16);
    const uint32_t tS = lane_base + (uint32_t)(w * 64);
    const uint32_t tdP = lane_base + 128u + (uint32_t)(w * 64);
    const int row = q0 + r;
    const bool row_ok = row < p.Nq;
    const float lse2 = row_ok ? p.lse[(size_t)bh * p.Nq + row] * kLog2e : 0.f;
    const float drow = row_ok ? p.dterm[(size_t)bh * p.Nq + row] : 0.f;
    // keys < lim are valid for this row
    int lim = row_ok ? kv_end : 0;
    if (p.causal) lim = min(lim, row + delta + 1);
    const uint64_t c2 = f32x2_pack(p.scale_log2, p.scale_log2);
    const uint64_t nl2 = f32x2_pack(-lse2, -lse2);
    bool ok = true;
    for (int j = 0; j < n; ++j) {
        const int nvalid = lim - (j * kT + w * 64);  // columns c < nvalid are valid
        const bool need_mask = nvalid < 64;
        if (!__all_sync(kFull, mbar_wait(&sm.s_full, (uint32_t)(j & 1), wc, 90))) {
            ok = false;
            break;
        }
        tc_fence_after_sync();
        uint32_t x[2][32];
        load64(tS, x);
        tc_fence_before_sync();
        mbar_arrive(&sm.s_free);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const uint64_t e2 = f32x2_fma(f32x2_pack(__uint_as_float(x[h][i]), __uint_as_float(x[h][i + 1])), c2,
                                              nl2);
                float e0, e1;
                f32x2_unpack(e2, e0, e1);
                float p0 = ex2_approx(e0), p1 = ex2_approx(e1);
                if (need_mask) {
                    const int c = h * 32 + i;
                    p0 = c < nvalid ? p0 : 0.f;
                    p1 = c + 1 < nvalid ? p1 : 0.f;
                }
                x[h][i] = __float_as_uint(p0);
                x[h][i + 1] = __float_as_uint(p1);
            }

        if (!__all_sync(kFull, mbar_wait(&sm.dp_full, (uint32_t)(j & 1), wc, 91))) {
            ok = false;
            break;
        }
        tc_fence_after_sync();
        uint32_t y[2][32];
        load64(tdP, y);
        // dS = P * (dP - D): bf16 pairs over dP
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const float s0 = __uint_as_float(x[h][i]) * (__uint_as_float(y[h][i]) - drow);
                const float s1 = __uint_as_float(x[h][i + 1]) * (__uint_as_float(y[h][i + 1]) - drow);
                pk[i / 2] = pack_bf16x2(s0, s1);
            }
            tmem_st16(tdP + (uint32_t)(h * 16), pk);
        }
        tmem_wait_st();
        tc_fence_before_sync();
        mbar_arrive(&sm.ds_full);
    }

    if (ok && n > 0) {
        if (!__all_sync(kFull, mbar_wait(&sm.acc_done, 0, wc, 92))) ok = false;
        else tc_fence_after_sync();
    }
    if (!ok) return;
    // warpgroup 0 writes columns 0 .. kDqSplit - 1 of dQ, warpgroup 1 the rest (times scale)
    __nv_bfloat16 *dst = p.dq + ((size_t)bh * p.Nq + (row_ok ? row : 0)) * D + (w ? kDqSplit<D> : 0);
    if (w == 0) store_rows<kDqSplit<D>>(lane_base + 256u, n > 0, row_ok, p.scale, dst);
    else store_rows<D - kDqSplit<D>>(lane_base + 256u + (uint32_t)kDqSplit<D>, n > 0, row_ok, p.scale, dst);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    DqSmem<D> &sm = *reinterpret_cast<DqSmem<D> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    int bh, level;
    unit_of(p, p.B * p.Hq, bh, level);
    const int qt = p.units_per_head - 1 - level;  // level 0 = the last query tile (most keys if causal)
    const int b = bh / p.Hq;
    const int bh_kv = b * p.Hkv + (bh % p.Hq) / p.group;
    const int q0 = qt * kT;
    const int kv_end = kv_end_for(p, b);
    const int delta = p.Nkv - p.Nq;
    int limit = kv_end;
    if (p.causal) limit = min(limit, min(q0 + kT, p.Nq) + delta);
    const int n = limit > 0 ? (limit + kT - 1) / kT : 0;

    if (threadIdx.x == 0) {
        mbar_init(&sm.qd_full, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.u_full[s], 1);
            mbar_init(&sm.u_empty[s], 1);
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.s_free, 256);
        mbar_init(&sm.dp_full, 1);
        mbar_init(&sm.ds_full, 256);
        mbar_init(&sm.acc_done, 1);
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
        if (lane == 0 && n > 0) dq_producer<D>(sm, &tmQ, &tmdO, &tmK, &tmV, bh, bh_kv, q0, n, wc);
    } else if (warp == kMmaWarp) {
        if (lane == 0 && n > 0) dq_mma<D>(sm, tmem, n, wc);
    } else {
        dq_compute<D>(sm, p, tmem, warp >> 2, bh, q0, kv_end, delta, n, wc);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

int heads_per_chunk(double bytes_per_head, int n_heads) {
    // about 48 MB of streamed tiles per chunk: the chunk finishing and the one starting fit in
    // the 126 MB L2 together
    int h = (int)(48.0e6 / bytes_per_head);
    return h < 1 ? 1 : (h > n_heads ? n_heads : h);
}

template <int D>
cudaError_t launch_bwd_d(const BwdArgs &a, cudaStream_t stream) {
    const long long rows = (long long)a.B * a.Hq * a.Nq;
    {
        const long long threads = rows * kRowThreads<D>;
        const unsigned grid = (unsigned)((threads + 255) / 256);
        bwd_rowdot_kernel<D><<<grid, 256, 0, stream>>>(reinterpret_cast<const __nv_bfloat16 *>(a.o),
                                                       reinterpret_cast<const __nv_bfloat16 *>(a.dout), a.dterm, rows);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    CUtensorMap tq, tdo, tk, tv;
    const int BHq = a.B * a.Hq, BHkv = a.B * a.Hkv;
    if (!encode_qkv_map(&tq, a.q, BHq, a.Nq, D) || !encode_qkv_map(&tdo, a.dout, BHq, a.Nq, D) ||
        !encode_qkv_map(&tk, a.k, BHkv, a.Nkv, D) || !encode_qkv_map(&tv, a.v, BHkv, a.Nkv, D))
        return cudaErrorInvalidValue;
    BwdParams p;
    p.lse = a.lse;
    p.dterm = a.dterm;
    p.dq = reinterpret_cast<__nv_bfloat16 *>(a.dq);
    p.dk = reinterpret_cast<__nv_bfloat16 *>(a.dk);
    p.dv = reinterpret_cast<__nv_bfloat16 *>(a.dv);
    p.kv_lens = a.kv_lens;
    p.status = a.status;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.group = a.Hq / a.Hkv;
    p.Nq = a.Nq;
    p.Nkv = a.Nkv;
    p.causal = a.causal;
    p.scale = a.scale;
    p.scale_log2 = a.scale * kLog2e;

    // dK/dV: one CTA per (batch, key/value head, key tile); streams Q and dO of the group's heads
    {
        BwdParams pk = p;
        pk.units_per_head = (a.Nkv + kT - 1) / kT;
        pk.heads_per_chunk = heads_per_chunk(2.0 * p.group * a.Nq * D * 2.0, BHkv);
        const size_t smem = sizeof(DkvSmem<D>) + 1024;
        cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void *>(bwd_dkdv_kernel<D>), (int)smem);
        if (e != cudaSuccess) return e;
        const unsigned grid = (unsigned)((size_t)pk.units_per_head * BHkv);
        bwd_dkdv_kernel<D><<<grid, kThreads, smem, stream>>>(tq, tdo, tk, tv, pk);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // dQ: one CTA per (batch, query head, query tile); streams K and V of its key/value head
    {
        BwdParams pq = p;
        pq.units_per_head = (a.Nq + kT - 1) / kT;
        pq.heads_per_chunk = heads_per_chunk(2.0 * a.Nkv * D * 2.0 / p.group, BHq);
        const size_t smem = sizeof(DqSmem<D>) + 1024;
        cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void *>(bwd_dq_kernel<D>), (int)smem);
        if (e != cudaSuccess) return e;
        const unsigned grid = (unsigned)((size_t)pq.units_per_head * BHq);
        bwd_dq_kernel<D><<<grid, kThreads, smem, stream>>>(tq, tdo, tk, tv, pq);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd(const BwdArgs &a, cudaStream_t stream) {
    switch (a.d) {
        case 32: return launch_bwd_d<32>(a, stream);
        case 64: return launch_bwd_d<64>(a, stream);
        case 80: return launch_bwd_d<80>(a, stream);
        case 96: return launch_bwd_d<96>(a, stream);
        case 128: return launch_bwd_d<128>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

size_t bwd_workspace_bytes(int B, int Hq, int Nq) {
    if (B <= 0 || Hq <= 0 || Nq <= 0) return 0;
    const size_t n = (size_t)B * (size_t)Hq * (size_t)Nq * sizeof(float);
    return (n + 255) & ~(size_t)255;
}

}  // namespace attn
