// prefill.cu -- FlashAttention-style prefill forward on the sm_103a tensor cores.
//
// The method (NanoInfer README, Flash Attention bullets; gpu-inference blog,
// section 02; llm-kernel-lib README, kernel 1; Kernel-Inference-Engine README,
// tile-loop flowchart): a Q tile stays resident while 128-key K/V tiles stream
// past it; per tile S = Q K^T * scale, mask, online softmax with a running max
// m and normaliser l, O rescaled by exp(m_old - m_new), O += P V; at the end
// O / l and LSE = m + ln l are stored.  The score matrix never reaches global
// memory, and K/V tiles wholly above the causal diagonal (or past the
// key-padding length) are never visited.
//
// GB300 mapping (d = 128; d <= 64 uses one query tile per CTA, 64-key tiles and four CTAs per SM,
// see Cfg).  One CTA = one (batch, head) and 256 query rows held as two 128-row tiles Q0, Q1 that
// share every K/V tile.  12 warps (three warpgroups):
//   warps 0-3  softmax warpgroup 0 (rows of Q0), warps 4-7  softmax warpgroup 1
//              (rows of Q1).  Thread r of a warpgroup owns query row r = TMEM
//              lane r: it loads its 128 scores from TMEM, masks, takes the row
//              max, and keeps a reference max that only moves when the new max
//              exceeds it by more than 2^8 (O and l always share the reference,
//              so the final O / l is unchanged; only then is O rescaled in TMEM).
//              P = 2^(x - m) is rounded to bf16 (f16 over an e4m3 cache) and written back into TMEM over
//              the scores it came from, where the PV product reads it as its A
//              operand.  The same warps run the epilogue.
//   warp 8     TMA producer: Q0, Q1 once, then K and V tiles through a 2-slot ring
//              (128-byte swizzled boxes of 128 rows x 64 columns).
//   warp 9     TMEM owner and MMA issuer (one thread).  TMEM (512 columns):
//              S0 | S1 (128 fp32 columns each; P_t aliases the first 64 columns
//              of S_t as packed bf16 pairs) | O0 | O1 (d columns each).
//   warps 10-11 idle: the third warpgroup hands its registers to the softmax
//              warpgroups (setmaxnreg), so a thread holds its whole 128-score row.
//              Over an e4m3 cache they and a fourth warpgroup (warps 12-15) widen the
//              codes, which the producer loads into the ring slots (run_convert).
// Issue order per K/V tile j:  PV0(j), S0(j+1), PV1(j), S1(j+1) -- while one
// warpgroup turns S_t(j+1) into P, the tensor core works for the other.
// Every tcgen05 op of the MMA thread completes in issue order, so the commit
// that signals S_t(j) also tells warpgroup t that PV_t(j-1) has finished with
// O_t and with the P_t columns.

#include <cmath>

#include "launch.h"
#include "sm103_ptx.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;  // query rows per tile
// Head dims 32, 64, 80, 96 and 128 (the set the Kernel-Inference-Engine README instantiates its
// attention kernel for).  Tiles are laid out at a padded width kPad<D> (64 up to d = 64, else
// 128) in 64-column boxes; TMA fills the columns past d with zeros, the S product runs over d/16
// k-steps and the PV product has N = d, so the padding costs shared memory but no tensor work.
template <int D> constexpr int kPad = D <= 64 ? 64 : 128;
// Shape of the CTA per padded head dimension.
//   128: two 128-row query tiles per CTA (ping-pong softmax warpgroups), 128-key tiles, 12 warps
//        with a per-warpgroup register split, one CTA per SM (192 KB smem, all 512 TMEM columns).
//   64:  one query tile per CTA and 64-key tiles, four CTAs per SM.  At d <= 64 the softmax (one
//        exponential per 256 tensor FLOPs) bounds each step, and a CTA's chain per key tile (S,
//        scores loaded, row max, exponentials, PV) is mostly latency; four CTAs give each SM
//        sub-partition four softmax warps to interleave instead of two.  A CTA needs 128 TMEM
//        columns (S 64 | O 64, P over S) and 48 KB of shared memory (Q 16 KB, a 2-slot ring of
//        8 KB K and V tiles).  8 warps: softmax warpgroup, producer, MMA issuer, two idle warps
//        whose registers go to the softmax warpgroup.
// Register split (setmaxnreg) per warpgroup, within the block's launch pool (threads x
// registers at launch):
//   128: launched at 168 (384 x 168 = 64512): 128 x (64 + 216 + 216) = 63488.
//   64:  launched at 64 (four CTAs of 256 per SM): 128 x (32 + 96) = 16384 = 256 x 64.
template <int P> struct CfgPad;
template <int D> struct Cfg : CfgPad<kPad<D>> {};
template <> struct CfgPad<128> {
    static constexpr int QT = 2, BN = 128, kThreads = 384, kProducerWarp = 8, kMmaWarp = 9, kMinBlocks = 1;
    static constexpr int kStages = 2;
    static constexpr uint32_t kTmemCols = 512;
    static constexpr bool kSplitRegs = true;
    static constexpr uint32_t kRegsSoftmax = 216, kRegsOther = 64;
};
template <> struct CfgPad<64> {
    static constexpr int QT = 1, BN = 64, kThreads = 256, kProducerWarp = 4, kMmaWarp = 5;
    static constexpr int kMinBlocks = 4, kStages = 2;
    static constexpr uint32_t kTmemCols = 128;
    static constexpr bool kSplitRegs = true;
    // launch allocation of kMinBlocks CTAs per SM, and its split over the two warpgroups
    static constexpr uint32_t kRegsLaunch = (65536 / (256 * kMinBlocks)) / 8 * 8;
    static constexpr uint32_t kRegsOther = kMinBlocks >= 4 ? 32 : (kMinBlocks == 3 ? 48 : 64);
    static constexpr uint32_t kRegsSoftmax = 2 * kRegsLaunch - kRegsOther;
};
static_assert(128 * (Cfg<128>::kRegsOther + 2 * Cfg<128>::kRegsSoftmax) <= 384 * 168, "d=128 register split");
static_assert(128 * (Cfg<64>::kRegsOther + Cfg<64>::kRegsSoftmax) <= 256 * Cfg<64>::kRegsLaunch, "d=64 register split");
static_assert(Cfg<64>::QT * (Cfg<64>::BN + 64) <= (int)Cfg<64>::kTmemCols, "d=64 TMEM layout");
static_assert(Cfg<128>::QT * (128 + 128) <= (int)Cfg<128>::kTmemCols, "d=128 TMEM layout");
// keys per tile
template <int D> constexpr int kBNd = Cfg<D>::BN;
constexpr int kQTilesMax = 2;
constexpr uint32_t kBoxBytes = 128 * 64 * 2;  // one 128-row x 64-column bf16 box (16 KB)
template <int D> constexpr uint32_t kKvBoxBytes = kBNd<D> * 64 * 2;  // one K or V box (kBNd rows)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 2^8
constexpr int kPageTokens = 16;            // tokens per page of the paged KV cache

// Where K/V come from (a compile-time parameter of the kernel, so that each form carries only
// its own code): contiguous [B, Hkv, Nkv, d] tensors; bf16 pages of a paged KV cache; or e4m3
// pages, widened to f16 in shared memory before the products.
enum KvMode : int { kContig = 0, kPagedBf16 = 1, kPagedE4m3 = 2 };

// CTAs per SM and the register split per KV mode.  e4m3 pages at d <= 64: the two converter warps
// (the non-softmax warpgroup's idle pair) need more than the 32 registers that four CTAs per SM
// would leave them, so three CTAs share an SM, launched at 80 registers (128 x (104 + 56) = 20480 =
// 256 x 80).
template <int D, int M> struct Occ {
    static constexpr int kMinBlocks = Cfg<D>::kMinBlocks, kThreads = Cfg<D>::kThreads;
    static constexpr uint32_t kRegsSoftmax = Cfg<D>::kRegsSoftmax, kRegsOther = Cfg<D>::kRegsOther;
};
// e4m3 pages at d > 64: a fourth warpgroup widens with the third's two idle warps -- six converter
// warps -- launched at 128 registers (512 threads); the two non-softmax warpgroups keep 64 each:
// 128 x (2 x 192 + 2 x 64) = 65536.  Measured (TFLOP/s on the chunked prefill over e4m3 pages) for
// softmax / other: 216 / 40 889, 208 / 48 914, 200 / 56 993, 192 / 64 995, 184 / 72 985, 168 / 88 976
// (at 40 the producer and converters spill).
template <int D> struct OccWide {
    static constexpr int kMinBlocks = 1, kThreads = 512;
    static constexpr uint32_t kRegsSoftmax = 192, kRegsOther = 64;
};
template <> struct Occ<80, kPagedE4m3> : OccWide<80> {};
template <> struct Occ<96, kPagedE4m3> : OccWide<96> {};
template <> struct Occ<128, kPagedE4m3> : OccWide<128> {};
static_assert(128 * (2 * OccWide<128>::kRegsSoftmax + 2 * OccWide<128>::kRegsOther) <= 65536, "wide e4m3 split");
template <> struct Occ<32, kPagedE4m3> {
    static constexpr int kMinBlocks = Cfg<32>::kMinBlocks < 3 ? Cfg<32>::kMinBlocks : 3;
    static constexpr int kThreads = Cfg<32>::kThreads;
    static constexpr uint32_t kLaunch = (65536 / (256 * kMinBlocks)) / 8 * 8;
    static constexpr uint32_t kRegsOther = kMinBlocks == 3 ? 56 : 64;
    static constexpr uint32_t kRegsSoftmax = 2 * kLaunch - kRegsOther;
};
template <> struct Occ<64, kPagedE4m3> : Occ<32, kPagedE4m3> {};
static_assert(128 * (Occ<64, kPagedE4m3>::kRegsSoftmax + Occ<64, kPagedE4m3>::kRegsOther) <=
                  256 * Occ<64, kPagedE4m3>::kLaunch,
              "e4m3 d<=64 register split");


struct PrefillParams {
    __nv_bfloat16 *o;
    float *lse;
    const int32_t *kv_lens;
    int *status;
    int B, H, Nq, Nkv, causal, n_units;  // n_units = ceil(Nq / 256) per (b, h)
    int Hkv, group;                      // key/value heads; query heads per key/value head
    // paged mode (chunked prefill into a paged KV cache): K/V come from 16-token pages
    // [num_pages, Hkv, 16, d] found through page_table [B, max_pages]; sequence b holds
    // ctx_lens[b] tokens and the queries are its last Nq positions
    const int32_t *page_table, *ctx_lens;
    int max_pages, num_pages;
    const uint8_t *k8, *v8;              // e4m3 pages [num_pages, Hkv, 16, d] (kPagedE4m3)
    int heads_per_chunk;                 // heads whose K/V share L2 at a time (see the CTA order)
    float scale_log2;                    // scale * log2(e) (times the key scale of e4m3 pages)
    float o_scale;                       // multiplies O in the epilogue (the value scale of e4m3 pages)
};

// K/V ring.  Step j of the MMA issuer (PV(j) then S(j+1)) needs V(j) and K(j+1) together,
// so they travel as one ring unit: unit u = {K(u), V(u-1)} (unit 0 has only K(0), unit n only
// V(n-1)); with S = kStagesOf<D> slots, K(j) sits in slot j % S, V(j) in slot (j+1) % S.  One
// full and one empty barrier per unit keeps the single MMA-issuing thread's synchronisation per
// step at one wait and one commit for the ring.
template <int D> constexpr int kStagesOf = Cfg<D>::kStages;

// e4m3 pages: a ring unit's codes land by TMA in its own slots -- in each tile's last 64-column
// box, one 128-byte row per key (zeros past d) -- and the converter warps widen them to f16 in place
// (code_off is that box's byte offset).
template <int D> constexpr int kCodeOff = (kPad<D> / 64 - 1) * kBNd<D> * 128;

template <int D, int M>
struct alignas(1024) PrefillSmem {
    // q, k, v: tiles of kBM x kPad elements back to back (the MMA issuer steps between them by
    // a constant)
    __nv_bfloat16 q[Cfg<D>::QT][kBM * kPad<D>];  // kPad/64 boxes each
    __nv_bfloat16 k[kStagesOf<D>][kBNd<D> * kPad<D>];  // kPad/64 boxes each
    __nv_bfloat16 v[kStagesOf<D>][kBNd<D> * kPad<D>];  // kPad/64 boxes each
    uint64_t q_full;
    uint64_t u_full[kStagesOf<D>], u_empty[kStagesOf<D>];
    uint64_t c_full[kStagesOf<D>];  // e4m3 pages: the unit's codes have landed
    uint64_t v_full[kStagesOf<D>];  // e4m3 pages: the unit's V tile is widened (u_full: its K tile)
    uint64_t s_full[kQTilesMax];
    uint64_t p_full[kQTilesMax];
    uint64_t o_done[kQTilesMax];
    uint64_t o_staged[kQTilesMax];  // the warpgroup's O rows are in shared memory
    uint64_t q_conv[kQTilesMax];    // e4m3 pages: the warpgroup's Q rows are f16 in shared memory
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};

// Cached tokens of sequence b in paged mode (clamped to the table's capacity).
__device__ __forceinline__ int kv_end_of(const PrefillParams &p, int b) {
    return min(max(p.ctx_lens[b], 0), p.max_pages * kPageTokens);
}

// TMEM columns: S_t at BN t; O_t after all S buffers; P_t (bf16 pairs) over the first BN/2
// columns of S_t.
template <int D> __device__ __forceinline__ uint32_t o_col(int t) {
    return (uint32_t)(Cfg<D>::QT * kBNd<D> + t * kPad<D>);
}
template <int D> __device__ __forceinline__ uint32_t p_col(int t) { return (uint32_t)(t * kBNd<D>); }

// Key tiles query tile t of this CTA must visit: keys < limit can be valid for some of its rows.
template <int BN>
__device__ __forceinline__ int tiles_for(const PrefillParams &p, int qs, int kv_end, int delta) {
    if (qs >= p.Nq) return 0;  // no rows in this tile (ragged end)
    int limit = kv_end;
    if (p.causal) limit = min(limit, min(qs + kBM, p.Nq) + delta);
    return limit > 0 ? (limit + BN - 1) / BN : 0;
}

// ------------------------------------------------------------------ producer
// Contiguous K/V: the loads that need no ring wait -- Q and the first kStages units -- issued by
// the producer thread before the CTA's start-up barrier, so they overlap the TMEM allocation and
// the other warps' start (at d = 64 this took the start of a CTA from about 5000 to 4200 cycles
// and the decoder workload's span from 28.4 to 25.1 us in a timestamped copy).  Returns the first
// unit left for run_producer.
template <int D, int M>
__device__ int producer_start(PrefillSmem<D, M> &sm, const PrefillParams &p, const CUtensorMap *tmQ,
                              const CUtensorMap *tmK, const CUtensorMap *tmV, int bh, int bh_kv, int q0, int n_all) {
    static_assert(M == kContig, "contiguous K/V only");
    constexpr int kBoxes = kPad<D> / 64;
    constexpr int kBN = kBNd<D>;
    prefetch_tensormap(tmQ);
    prefetch_tensormap(tmK);
    prefetch_tensormap(tmV);
    mbar_arrive_expect_tx(&sm.q_full, Cfg<D>::QT * kBoxes * kBoxBytes);
#pragma unroll
    for (int t = 0; t < Cfg<D>::QT; ++t)
#pragma unroll
        for (int i = 0; i < kBoxes; ++i)
            tma_load_3d(sm.q[t] + i * (kBM * 64), tmQ, &sm.q_full, i * 64, q0 + t * kBM, bh);
    const int first = n_all + 1 < kStagesOf<D> ? n_all + 1 : kStagesOf<D>;
    for (int u = 0; u < first; ++u) {
        const bool has_k = u < n_all, has_v = u > 0;
        mbar_arrive_expect_tx(&sm.u_full[u], ((has_k ? 1 : 0) + (has_v ? 1 : 0)) * kBoxes * kKvBoxBytes<D>);
#pragma unroll
        for (int i = 0; i < kBoxes; ++i) {
            if (has_k) tma_load_3d(sm.k[u] + i * (kBN * 64), tmK, &sm.u_full[u], i * 64, u * kBN, bh_kv);
            if (has_v) tma_load_3d(sm.v[u] + i * (kBN * 64), tmV, &sm.u_full[u], i * 64, (u - 1) * kBN, bh_kv);
        }
    }
    return first;
}

template <int D, int M>
__device__ void run_producer(PrefillSmem<D, M> &sm, const PrefillParams &p, const CUtensorMap *tmQ,
                             const CUtensorMap *tmK, const CUtensorMap *tmV, int b, int bh, int bh_kv, int q0,
                             int n_all, int u_begin, WaitCtx wc) {
    constexpr int kBoxes = kPad<D> / 64;
    if (u_begin == 0) {  // Q not yet issued (paged modes)
        prefetch_tensormap(tmQ);
        prefetch_tensormap(tmK);
        prefetch_tensormap(tmV);
        mbar_arrive_expect_tx(&sm.q_full, Cfg<D>::QT * kBoxes * kBoxBytes);
#pragma unroll
        for (int t = 0; t < Cfg<D>::QT; ++t)
#pragma unroll
            for (int i = 0; i < kBoxes; ++i)
                tma_load_3d(sm.q[t] + i * (kBM * 64), tmQ, &sm.q_full, i * 64, q0 + t * kBM, bh);
    }
    // paged modes: the page ids of each tile (-1 past the sequence's last page), fetched one
    // ring unit ahead of their use, so the global loads stay in flight across the ring wait
    constexpr int kBN = kBNd<D>;
    constexpr int kTilePages = kBN / kPageTokens;
    const int kvh = bh_kv % p.Hkv;
    const int pages_used = (M != kContig) ? (kv_end_of(p, b) + kPageTokens - 1) / kPageTokens : 0;
    auto fetch_ids = [&](int tile, int (&ids)[kTilePages]) {
#pragma unroll
        for (int pg = 0; pg < kTilePages; ++pg) {
            const int lp = tile * kTilePages + pg;
            ids[pg] = lp < pages_used ? p.page_table[(size_t)b * p.max_pages + lp] : -1;
        }
    };
    int ids_prev[kTilePages], ids_cur[kTilePages], ids_next[kTilePages];
#pragma unroll
    for (int pg = 0; pg < kTilePages; ++pg) ids_prev[pg] = ids_cur[pg] = ids_next[pg] = -1;
    if constexpr (M != kContig) fetch_ids(0, ids_next);

    // K/V by TMA into the ring slots.  Paged: pool row (page * Hkv + head) of each page of a tile;
    // pages past the sequence's last page, or with an id outside the pool (an unmapped page, whose
    // keys the softmax masks), get an out-of-range row, which TMA reads as zeros.  bf16 pages: one
    // 16-row box per page and 64-column block; e4m3 pages: one box of 16 rows x 128 codes per page,
    // into the tile's code rows (kCodeOff), for the converters to widen.
    auto load_tile = [&](__nv_bfloat16 *dst, const CUtensorMap *map, uint64_t *bar, const int (&ids)[kTilePages]) {
#pragma unroll
        for (int pg = 0; pg < kTilePages; ++pg) {
            const int id = ids[pg];
            const int row = (id >= 0 && id < p.num_pages) ? id * p.Hkv + kvh : p.num_pages * p.Hkv;
            if constexpr (M == kPagedE4m3) {
                tma_load_3d(reinterpret_cast<uint8_t *>(dst) + kCodeOff<D> + pg * (kPageTokens * 128), map, bar, 0, 0,
                            row);
            } else {
#pragma unroll
                for (int i = 0; i < kBoxes; ++i)
                    tma_load_3d(dst + i * (kBN * 64) + pg * (kPageTokens * 64), map, bar, i * 64, 0, row);
            }
        }
    };
    int fills = u_begin;
    for (int u = u_begin; u <= n_all; ++u) {
        const int slot = u % kStagesOf<D>, use = u / kStagesOf<D>;
        if (use > 0 && !mbar_wait(&sm.u_empty[slot], (uint32_t)((use - 1) & 1), wc, 1)) break;
        const bool has_k = u < n_all, has_v = u > 0;
        // e4m3 pages: the codes complete c_full, and the converters then complete u_full
        uint64_t *full = (M == kPagedE4m3) ? &sm.c_full[slot] : &sm.u_full[slot];
        constexpr uint32_t kTileBytes = (M == kPagedE4m3) ? (uint32_t)kBN * 128 : kBoxes * kKvBoxBytes<D>;
        mbar_arrive_expect_tx(full, ((has_k ? 1 : 0) + (has_v ? 1 : 0)) * kTileBytes);
        if constexpr (M == kContig) {
            if (has_k) {
#pragma unroll
                for (int i = 0; i < kBoxes; ++i)
                    tma_load_3d(sm.k[slot] + i * (kBN * 64), tmK, &sm.u_full[slot], i * 64, u * kBN, bh_kv);
            }
            if (has_v) {
#pragma unroll
                for (int i = 0; i < kBoxes; ++i)
                    tma_load_3d(sm.v[slot] + i * (kBN * 64), tmV, &sm.u_full[slot], i * 64, (u - 1) * kBN, bh_kv);
            }
        } else {
            // a tile is kBN / 16 pages of 16 keys: one 16-row box per page and 64-column block,
            // stacked in the tile's 128-byte-swizzled rows.  K(u) uses the pages of tile u,
            // V(u-1) those of tile u-1 (already looked up for K(u-1)); tile u+1's page ids are
            // fetched here, one unit ahead of their use.
#pragma unroll
            for (int pg = 0; pg < kTilePages; ++pg) {
                ids_prev[pg] = ids_cur[pg];
                ids_cur[pg] = ids_next[pg];
            }
            if (u + 1 < n_all) fetch_ids(u + 1, ids_next);
            if (has_k) load_tile(sm.k[slot], tmK, full, ids_cur);
            if (has_v) load_tile(sm.v[slot], tmV, full, ids_prev);
        }
        ++fills;
    }
    if (*wc.abort_flag) {
        // unwinding: let every copy still in flight land before the CTA exits
        WaitCtx drain{nullptr, wc.status};
        (void)mbar_wait(&sm.q_full, 0, drain, 90);
        for (int f = (fills > kStagesOf<D> ? fills - kStagesOf<D> : 0); f < fills; ++f)
            (void)mbar_wait(M == kPagedE4m3 ? &sm.c_full[f % kStagesOf<D>] : &sm.u_full[f % kStagesOf<D>],
                            (uint32_t)((f / kStagesOf<D>) & 1), drain, 91);
    }
}

// ------------------------------------------------------------------ e4m3 converters
// The converter warps widen each ring unit's e4m3 codes to f16 in place, into the layout a TMA
// load with the 128-byte swizzle gives (16-byte chunk c of row r of a 64-column box at chunk
// c ^ (r % 8)), so the MMA issuer reads the tile exactly as a loaded bf16 one.  Each e4m3 value is
// an f16 value (the widening is exact, one conversion per pair); the tensor scales fold elsewhere
// (the key scale into the score scale, the value scale into the epilogue), and Q is rounded to f16
// by the softmax warps (run_softmax).
// Widens one tile in place.  Row r's codes (128 bytes at kCodeOff + 128 r) lie inside the bytes of
// row r of the tile's last box, and nothing else of the f16 tile overlaps them, so a warp that owns
// whole rows reads a row's codes, meets at __syncwarp, and writes the row over them: no other warp
// touches those bytes.  Lanes take 16-code chunks, kPad/16 lanes per row.
template <int D, int kCW>
__device__ __forceinline__ void widen_in_place(__nv_bfloat16 *tile, int cw, int lane) {
    constexpr int kBN = kBNd<D>;
    constexpr int kLanesPerRow = kPad<D> / 16;  // the chunks that carry columns < kPad
    constexpr int kRowsPerStep = 32 / kLanesPerRow;
    static_assert(kBN % kRowsPerStep == 0, "whole steps of rows");
    uint8_t *t8 = reinterpret_cast<uint8_t *>(tile);
    const int rsub = lane / kLanesPerRow, c16 = lane % kLanesPerRow;
    const int box = c16 >> 2, k0 = (c16 & 3) * 2;  // the row's 16-byte f16 chunks k0, k0 + 1 of this box
#pragma unroll 2
    for (int r0 = cw * kRowsPerStep; r0 < kBN; r0 += kCW * kRowsPerStep) {
        const int r = r0 + rsub;
        const uint4 v = *reinterpret_cast<const uint4 *>(t8 + kCodeOff<D> + r * 128 + c16 * 16);
        __syncwarp();
        uint4 lo, hi;
        e4m3x4_to_f16x2x2(v.x, lo.x, lo.y);
        e4m3x4_to_f16x2x2(v.y, lo.z, lo.w);
        e4m3x4_to_f16x2x2(v.z, hi.x, hi.y);
        e4m3x4_to_f16x2x2(v.w, hi.z, hi.w);
        uint8_t *row = t8 + box * (kBN * 128) + r * 128;
        *reinterpret_cast<uint4 *>(row + ((k0 ^ (r & 7)) << 4)) = lo;
        *reinterpret_cast<uint4 *>(row + (((k0 + 1) ^ (r & 7)) << 4)) = hi;
    }
}

// NCV converter threads (the warps after the MMA issuer's).
template <int D> constexpr int kConverters = Occ<D, kPagedE4m3>::kThreads - (Cfg<D>::kMmaWarp + 1) * 32;

// Per ring unit u = {K(u), V(u-1)}: wait for its codes; widen V(u-1) first, fence the writes for
// the async proxy and arrive (one lane per warp) on the unit's V barrier; then K(u) and the unit's
// full barrier.  Each completes when every converter warp has arrived (unit 0 has no V and the
// last unit no K: the arrivals keep the barriers' phases in step).
template <int D>
__device__ void run_convert(PrefillSmem<D, kPagedE4m3> &sm, int n_all, int ct, WaitCtx wc) {
    constexpr int kCW = kConverters<D> / 32;
    const int cw = ct >> 5, lane = ct & 31;
    for (int u = 0; u <= n_all; ++u) {
        const int slot = u % kStagesOf<D>, use = u / kStagesOf<D>;
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.c_full[slot], (uint32_t)(use & 1), wc, 5))) break;
        if (u > 0) widen_in_place<D, kCW>(sm.v[slot], cw, lane);
        fence_proxy_async_smem();  // this thread's tile writes, before the MMA's reads
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.v_full[slot]);
        if (u < n_all) widen_in_place<D, kCW>(sm.k[slot], cw, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.u_full[slot]);
    }
}

// ------------------------------------------------------------------ MMA issuer
template <int D, int M>
__device__ void run_mma(PrefillSmem<D, M> &sm, uint32_t tmem, const int (&n)[kQTilesMax], int n_all, WaitCtx wc) {
    constexpr int kBN = kBNd<D>;
    // e4m3 pages: Q, K and V are f16 in shared memory and P is packed as f16, so both products run
    // f16 x f16
    constexpr uint32_t idS =
        M == kPagedE4m3 ? idesc_f16_f32(kBM, kBN, false, false) : idesc_bf16_f32(kBM, kBN, false, false);
    constexpr uint32_t idPV =
        M == kPagedE4m3 ? idesc_f16_f32(kBM, D, false, true) : idesc_bf16_f32(kBM, D, false, true);

    // Descriptors of the operand buffers, built once (the Q tiles, the K tiles and the V tiles
    // are each equally spaced: kQTile and kKvTile descriptor units); each MMA advances one by a
    // constant.
    constexpr uint64_t kQTile = (uint64_t)(kBM * kPad<D> * 2) >> 4;
    constexpr uint64_t kKvTile = (uint64_t)(kBN * kPad<D> * 2) >> 4;
    const uint64_t dq = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);
    const uint64_t dk = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);
    const uint64_t dv = sdesc_sw128(smem_u32(sm.v[0]), kKvBoxBytes<D>, 1024);

    // S_t(j) = Q_t K_j^T  (A = Q_t, B = K_j: both K-major, 128-byte swizzle), d/16 k-steps
    // issued in groups from single asm statements (the second 64-column box of a 128-row tile
    // starts 16 KB on, which the grouped issue assumes)
    static_assert(kPad<D> == 64 || kBN * 128 == 16384, "k-step layout of the grouped issue");
    auto issue_S = [&](int t, int j) {
        const uint64_t a = dq + (t ? kQTile : 0);
        const uint64_t b = dk + (uint64_t)(j % kStagesOf<D>) * kKvTile;  // K(j) sits in slot j % S
        const uint32_t tS = tmem + (uint32_t)(t * kBN);
        tc_mma_ss_ksteps<D / 16>(tS, a, b, idS, 0u);
        tc_commit(&sm.s_full[t]);
    };
    // O_t += P_t V_j  (A = P_t from TMEM, 8 columns per 16 keys; B = V_j MN-major, 16 keys = 2048 B)
    static_assert(kBN == 128 || kBN == 64, "PV is one group of eight or four k-steps");
    auto issue_PV = [&](int t, int j) {
        const uint64_t b = dv + (uint64_t)((j + 1) % kStagesOf<D>) * kKvTile;  // V(j) sits in slot (j + 1) % S
        const uint32_t tP = tmem + p_col<D>(t);
        const uint32_t tO = tmem + o_col<D>(t);
        if constexpr (kBN == 128) tc_mma_ts_k8(tO, tP, b, idPV, j > 0 ? 1u : 0u);
        else tc_mma_ts_k4(tO, tP, b, idPV, j > 0 ? 1u : 0u);
    };

    // The data waits below (Q, ring units) need no tcgen05 fence: TMA writes and the MMA's
    // operand reads are both async-proxy traffic ordered by the mbarrier.  The P waits do
    // (P was written to TMEM by other threads).
    bool ok = mbar_wait(&sm.q_full, 0, wc, 11);
    if constexpr (M == kPagedE4m3)  // the Q tiles rounded to f16 in place (generic-proxy writes, fenced)
        for (int t = 0; t < Cfg<D>::QT && ok; ++t) ok = mbar_wait(&sm.q_conv[t], 0, wc, 14);
    ok = ok && mbar_wait(&sm.u_full[0], 0, wc, 10);
    if (ok) {
        tc_fence_after_sync();
        for (int t = 0; t < Cfg<D>::QT; ++t)
            if (n[t] > 0) issue_S(t, 0);
        tc_commit(&sm.u_empty[0]);
        for (int j = 0; j < n_all && ok; ++j) {
            const int u = j + 1;  // unit with V(j) and K(j+1)
            const uint32_t ph = (uint32_t)((u / kStagesOf<D>) & 1);
            // e4m3 pages: V(j) is widened before K(j+1) and signalled on its own barrier, so the
            // first PV can start while the converters still widen the keys
            ok = mbar_wait(M == kPagedE4m3 ? &sm.v_full[u % kStagesOf<D>] : &sm.u_full[u % kStagesOf<D>], ph, wc, 13);
            if (!ok) break;
            bool k_ready = (M != kPagedE4m3);
            // P over S: PV_t(j) must be issued before S_t(j+1) overwrites its buffer
            for (int t = 0; t < Cfg<D>::QT; ++t) {
                if (j < n[t]) {
                    if (!(ok = mbar_wait(&sm.p_full[t], (uint32_t)(j & 1), wc, 12 + 8 * t))) break;
                    tc_fence_after_sync();
                    issue_PV(t, j);
                    if (j == n[t] - 1) tc_commit(&sm.o_done[t]);
                }
                if (j + 1 < n[t]) {
                    if (!k_ready) {
                        if (!(ok = mbar_wait(&sm.u_full[u % kStagesOf<D>], ph, wc, 15))) break;
                        k_ready = true;
                    }
                    issue_S(t, j + 1);
                }
            }
            if (!ok) break;
            tc_commit(&sm.u_empty[u % kStagesOf<D>]);
        }
    }
    // wait (bounded) until every MMA issued above has finished with TMEM and smem
    tc_commit(&sm.drain);
    WaitCtx drain{nullptr, wc.status};
    (void)mbar_wait(&sm.drain, 0, drain, 19);
}

// ------------------------------------------------------------------ softmax + epilogue
// O row *= alpha in TMEM (whole warp; alpha = 1 for rows that keep their reference max).
// Rare (only when a row max grows by more than 2^8); done 16 columns at a time so it adds
// few registers to the softmax loop.
template <int D>
__device__ __forceinline__ void rescale_o(uint32_t tO, float alpha) {
#pragma unroll 1
    for (int cc = 0; cc < D / 16; ++cc) {
        uint32_t ov[16];
        tmem_ld16(tO + cc * 16, ov);
        tmem_wait_ld16(ov);
#pragma unroll
        for (int i = 0; i < 16; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
        tmem_st16(tO + cc * 16, ov);
    }
}

// Scores at positions >= nvalid (relative to the first of the 64 held) become -inf.
__device__ __forceinline__ void mask_chunks(uint32_t (&s)[2][32], int nvalid) {
#pragma unroll
    for (int cc = 0; cc < 2; ++cc)
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (cc * 32 + i >= nvalid) s[cc][i] = __float_as_uint(-INFINITY);
}

// Paged mode: scores of keys whose page is unmapped (bit pg of `bad` set: keys 16 pg .. 16 pg + 15
// of the tile) become -inf, as a padded key would.
template <int H>
__device__ __forceinline__ void mask_pages(uint32_t (&s)[H][2][32], uint32_t bad) {
#pragma unroll
    for (int h = 0; h < H; ++h)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if ((bad >> (h * 4 + cc * 2 + (i >> 4))) & 1u) s[h][cc][i] = __float_as_uint(-INFINITY);
}

// Max of 64 scores: eight independent three-input chains, then a tree.
__device__ __forceinline__ float max64(const uint32_t (&s)[2][32]) {
    float m[8];
#pragma unroll
    for (int a = 0; a < 8; ++a) m[a] = fmaxf(__uint_as_float(s[0][a]), __uint_as_float(s[0][a + 8]));
#pragma unroll
    for (int a = 0; a < 8; ++a) m[a] = fmax3(m[a], __uint_as_float(s[0][a + 16]), __uint_as_float(s[0][a + 24]));
#pragma unroll
    for (int a = 0; a < 8; ++a) {
        m[a] = fmax3(m[a], __uint_as_float(s[1][a]), __uint_as_float(s[1][a + 8]));
        m[a] = fmax3(m[a], __uint_as_float(s[1][a + 16]), __uint_as_float(s[1][a + 24]));
    }
    return fmax3(fmax3(m[0], m[1], m[2]), fmax3(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}

// p = 2^(s*c - m) for 64 scores (two per packed FMA), summed into rs2 and stored to TMEM
// as 32 columns of bf16 pairs (f16 pairs when F16P) starting at tP.
template <bool F16P = false>
__device__ __forceinline__ void exp_store(const uint32_t (&s)[2][32], uint32_t tP, uint64_t c2, uint64_t negm2,
                                          uint64_t (&rs2)[4]) {
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            const uint64_t x2 =
                f32x2_fma(f32x2_pack(__uint_as_float(s[cc][i]), __uint_as_float(s[cc][i + 1])), c2, negm2);
            float x0, x1;
            f32x2_unpack(x2, x0, x1);
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            rs2[(i >> 1) & 3] = f32x2_add(rs2[(i >> 1) & 3], f32x2_pack(p0, p1));
            pk[i / 2] = F16P ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
        }
        tmem_st16(tP + cc * 16, pk);
    }
}

// Row r of a Q tile (kPad/64 boxes of kBM x 64 bf16, 128-byte swizzle) rounded to f16 in place after
// the factor 2^-sh, sh = 0 unless |q| reaches 2^15 (then the smallest that brings the row below 2^15,
// at most 113); returns 2^sh.  Chunk j of the row is read from position j ^ (r % 8) so that eight
// consecutive rows fall in different banks.
template <int D>
__device__ __forceinline__ float q_row_to_f16(__nv_bfloat16 *qt, int r) {
    constexpr int kBx = kPad<D> / 64;
    uint8_t *base = reinterpret_cast<uint8_t *>(qt) + r * 128;
    uint4 v[kBx * 8];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kBx * 8; ++i) {
        v[i] = *reinterpret_cast<const uint4 *>(base + (i >> 3) * (kBM * 128) + (((i & 7) ^ (r & 7)) << 4));
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[k] << 16)), fabsf(__uint_as_float(w[k] & 0xffff0000u))));
    }
    const int e = (int)((__float_as_uint(amax) >> 23) & 0xffu) - 127;
    const int sh = e >= 15 ? min(e - 14, 113) : 0;
    const float f = __uint_as_float((uint32_t)(127 - sh) << 23);
#pragma unroll
    for (int i = 0; i < kBx * 8; ++i) {
        uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = pack_f16x2(__uint_as_float(w[k] << 16) * f, __uint_as_float(w[k] & 0xffff0000u) * f);
        *reinterpret_cast<uint4 *>(base + (i >> 3) * (kBM * 128) + (((i & 7) ^ (r & 7)) << 4)) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
    return __uint_as_float((uint32_t)(127 + sh) << 23);
}

template <int D, int M>
__device__ void run_softmax(PrefillSmem<D, M> &sm, const PrefillParams &p, const CUtensorMap *tmO, uint32_t tmem,
                            int t, int bh, int q0, int n_tiles, int n_all, int kv_end, int delta, WaitCtx wc) {
    const int r = threadIdx.x & 127;  // query row in the tile = TMEM lane
    const int wq = (threadIdx.x >> 5) & 3;
    const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
    constexpr int kBN = kBNd<D>;
    constexpr int kHalves = kBN / 64;  // the row's scores of a tile, in halves of 64
    const uint32_t tS = lane_base + (uint32_t)(t * kBN);
    const uint32_t tO = lane_base + o_col<D>(t);
    const int qs = q0 + t * kBM;  // first row of this tile
    const int row = qs + r;
    float c = p.scale_log2;
    if constexpr (M == kPagedE4m3) {
        // Over e4m3 pages the products run in f16: each thread rounds its Q row to f16 in place once
        // Q has landed, after a power-of-two factor 2^-sh that keeps the row below 2^15 (exact for
        // every value in f16's normal range), and folds 2^sh into its score scale.
        if (n_all > 0) {
            if (!__all_sync(0xffffffffu, mbar_wait(&sm.q_full, 0, wc, 25))) return;
            c *= q_row_to_f16<D>(sm.q[t], r);
            fence_proxy_async_smem();  // before the MMA's reads of the tile
            mbar_arrive(&sm.q_conv[t]);
        }
    }
    const uint64_t c2 = f32x2_pack(c, c);

    float m_ref = -INFINITY;  // reference max (log2 domain) shared by l and O
    float l = 0.f;
    bool ok = true;
    // Paged mode: a page id outside the pool is an unmapped page that holds no token (the producer
    // loads zeros there; its keys are masked here).  The first lanes of each warp read the tile's
    // table entries (one per 16 keys) themselves, one tile ahead of its use, and a ballot turns
    // them into a warp-uniform mask of unmapped pages.
    constexpr bool kPaged = (M != kContig);
    const int lane = threadIdx.x & 31;
    const int pages_used = kPaged ? (kv_end + kPageTokens - 1) / kPageTokens : 0;
    const int32_t *table = kPaged ? p.page_table + (size_t)(bh / p.H) * p.max_pages : nullptr;
    auto table_entry = [&](int tile) {
        const int lp = tile * (kBN / kPageTokens) + lane;
        return (lane < kBN / kPageTokens && lp < pages_used) ? table[lp] : 0;
    };
    int next_id = 0;
    if constexpr (kPaged) next_id = table_entry(0);
    for (int j = 0; j < n_tiles; ++j) {
        uint32_t unmapped = 0;
        if constexpr (kPaged) {
            const int id = next_id;
            if (j + 1 < n_tiles) next_id = table_entry(j + 1);
            unmapped = __ballot_sync(0xffffffffu, id < 0 || id >= p.num_pages);
        }
        // every decision that guards a .sync.aligned tcgen05 instruction is warp-uniform
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.s_full[t], (uint32_t)(j & 1), wc, 20 + t))) {
            ok = false;
            break;
        }
        tc_fence_after_sync();

        // Keys key0 .. key0+nvalid-1 are valid for this row; masking is needed only on tiles
        // that straddle the causal diagonal or the key-padding length.
        const int key0 = j * kBN;
        const bool need_mask = (key0 + kBN > kv_end) || (p.causal && key0 + kBN - 1 > qs + delta);
        int nvalid = kBN;
        if (need_mask) {
            int lim = kv_end;
            if (p.causal) lim = min(lim, row + delta + 1);
            nvalid = lim - key0;
        }
        uint32_t s[kHalves][2][32];  // the row's scores as halves of 64
#pragma unroll
        for (int h = 0; h < kHalves; ++h) {
            tmem_ld32(tS + h * 64, s[h][0]);
            tmem_ld32(tS + h * 64 + 32, s[h][1]);
        }
#pragma unroll
        for (int h = 0; h < kHalves; ++h) {
            tmem_wait_ld(s[h][0]);
            tmem_wait_ld(s[h][1]);
        }
        if (need_mask) {
#pragma unroll
            for (int h = 0; h < kHalves; ++h) mask_chunks(s[h], nvalid - 64 * h);
        }
        if (kPaged && unmapped) mask_pages<kHalves>(s, unmapped);
        float mx = max64(s[0]);
#pragma unroll
        for (int h = 1; h < kHalves; ++h) mx = fmaxf(mx, max64(s[h]));
        const float m_cand = mx * c;  // -inf stays -inf (c > 0)
        const bool resc = m_cand > m_ref + kRescaleThreshold;
        float alpha = 1.f;
        if (resc) {
            alpha = ex2_approx(m_ref - m_cand);  // 0 when m_ref = -inf
            m_ref = m_cand;
            l *= alpha;
        }
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        const uint64_t negm2 = f32x2_pack(-m_use, -m_use);

        // P = 2^(s*c - m_use) as bf16 pairs (even key in the low half, as the TMEM A operand
        // expects): keys 64h .. 64h + 63 -> columns 32h .. 32h + 31, over the scores already
        // read into registers.  Over e4m3 pages P is packed as f16 pairs instead, the type of the
        // widened V tile (P <= 2^8 with the lazy reference max, well inside f16's range).
        uint64_t rs2[4] = {0, 0, 0, 0};
#pragma unroll
        for (int h = 0; h < kHalves; ++h) exp_store<M == kPagedE4m3>(s[h], tS + 32 * h, c2, negm2, rs2);
        {
            const uint64_t t01 = f32x2_add(rs2[0], rs2[1]);
            const uint64_t t23 = f32x2_add(rs2[2], rs2[3]);
            float a0, a1;
            f32x2_unpack(f32x2_add(t01, t23), a0, a1);
            l += a0 + a1;
        }

        // O_t is stable here: PV_t(j-1) completed before S_t(j) was signalled (the issuer's
        // commits complete in order, and S_t(j) is issued after PV_t(j-1))
        if (j > 0 && __any_sync(0xffffffffu, resc)) rescale_o<D>(tO, alpha);
        tmem_wait_st();
        tc_fence_before_sync();
        mbar_arrive(&sm.p_full[t]);
    }

    // epilogue: O / l -> bf16, LSE = ln2 * (m_ref + log2 l).  Each thread writes its row into the Q
    // tile's shared memory, free once the tile's last product has completed (o_done; if the tile had
    // no key, once its Q load has landed), in the 128-byte swizzled box layout of a TMA load; one
    // thread of the warpgroup then stores the tile with TMA (rows past Nq and columns past d are not
    // written).
    if (ok && n_tiles > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.o_done[t], 0, wc, 22 + t))) ok = false;
        else tc_fence_after_sync();
    } else if (ok && n_all > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(&sm.q_full, 0, wc, 24))) ok = false;
    }
    if (!ok) return;
    const bool have = (n_tiles > 0) && (l > 0.f);
    const float inv_l = have ? (M == kPagedE4m3 ? p.o_scale : 1.f) / l : 0.f;
    uint8_t *stage = reinterpret_cast<uint8_t *>(sm.q[t]) + r * 128;
    auto put = [&](int col0, const uint32_t *pk, int nchunks) {  // 16-byte chunks from column col0
#pragma unroll
        for (int q = 0; q < nchunks; ++q) {
            const int col = col0 + 8 * q;
            const int c = (col & 63) >> 3;
            *reinterpret_cast<uint4 *>(stage + (col >> 6) * (kBM * 128) + ((c ^ (r & 7)) << 4)) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
    };
#pragma unroll
    for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t ov[32];
        if (n_tiles > 0) {
            tmem_ld32(tO + cc * 32, ov);
            tmem_wait_ld(ov);
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            pk[i] = have ? pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l)
                         : 0u;
        put(cc * 32, pk, 4);
    }
    if constexpr (D % 32 != 0) {  // d = 80: the last 16 columns
        constexpr int c0 = D / 32 * 32;
        uint32_t ov[16];
        if (n_tiles > 0) {
            tmem_ld16(tO + c0, ov);
            tmem_wait_ld16(ov);
        }
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            pk[i] = have ? pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l)
                         : 0u;
        put(c0, pk, 2);
    }
    if (row < p.Nq && p.lse) p.lse[(size_t)bh * p.Nq + row] = have ? kLn2 * (m_ref + __log2f(l)) : -INFINITY;
    fence_proxy_async_smem();  // the staged rows, before the TMA store reads them
    mbar_arrive(&sm.o_staged[t]);
    if (r == 0 && qs < p.Nq) {
        if (mbar_wait(&sm.o_staged[t], 0, wc, 25 + t)) {
#pragma unroll
            for (int i = 0; i < kPad<D> / 64; ++i)
                if (i * 64 < D) tma_store_3d(tmO, reinterpret_cast<const uint8_t *>(sm.q[t]) + i * (kBM * 128), i * 64, qs, bh);
            bulk_commit_group();
            bulk_wait_group_all();
        }
    }
}

template <int D, int M>
__global__ void __launch_bounds__((Occ<D, M>::kThreads), (Occ<D, M>::kMinBlocks))
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                   const PrefillParams p) {
    extern __shared__ uint8_t smem_raw[];
    PrefillSmem<D, M> &sm =
        *reinterpret_cast<PrefillSmem<D, M> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // CTA order: heads are taken in chunks small enough that the chunk's K/V stays in L2
    // while its query units stream it; inside a chunk the units go heaviest first across
    // all its heads (the last query rows, which see the most keys under the causal mask).
    // The hardware dispatches CTAs in index order, so this is a longest-first schedule per
    // chunk: no heavy unit is left to start at the end of the launch.
    const int BH = p.B * p.H;
    const int per_chunk = p.heads_per_chunk * p.n_units;
    const int chunk = (int)(blockIdx.x / per_chunk);
    const int h0 = chunk * p.heads_per_chunk;
    const int heads = min(p.heads_per_chunk, BH - h0);  // the last chunk may be smaller
    const int in_chunk = (int)(blockIdx.x % per_chunk);
    const int level = in_chunk / heads;  // 0 = heaviest unit of a head
    const int bh = h0 + in_chunk % heads;
    const int unit = p.n_units - 1 - level;
    // key/value head of this query head (grouped-query attention; = bh for multi-head)
    const int bh_kv = (bh / p.H) * p.Hkv + (bh % p.H) / p.group;
    const int b = bh / p.H;
    const int q0 = unit * (kBM * Cfg<D>::QT);
    // keys of this sequence and the causal offset (query i sits at key position i + delta)
    int kv_end, delta;
    if constexpr (M != kContig) {
        kv_end = kv_end_of(p, b);
        delta = kv_end - p.Nq;
    } else {
        kv_end = p.kv_lens ? min(max(p.kv_lens[b], 0), p.Nkv) : p.Nkv;
        delta = p.Nkv - p.Nq;
    }
    int n[kQTilesMax] = {0, 0};
#pragma unroll
    for (int t = 0; t < Cfg<D>::QT; ++t) n[t] = tiles_for<kBNd<D>>(p, q0 + t * kBM, kv_end, delta);
    const int n_all = max(n[0], n[1]);

    // The producer thread initialises the barriers and, for contiguous K/V, issues the loads that
    // need no ring wait before the start-up barrier.
    const bool producer = (warp == Cfg<D>::kProducerWarp && lane == 0);
    int u_begin = 0;
    if (producer) {
        mbar_init(&sm.q_full, 1);
        for (int s = 0; s < kStagesOf<D>; ++s) {
            // e4m3 pages: the unit is full once every converter warp has widened its rows
            mbar_init(&sm.u_full[s], M == kPagedE4m3 ? kConverters<D> / 32 : 1);
            mbar_init(&sm.u_empty[s], 1);
            mbar_init(&sm.c_full[s], 1);
            mbar_init(&sm.v_full[s], M == kPagedE4m3 ? kConverters<D> / 32 : 1);
        }
        for (int t = 0; t < Cfg<D>::QT; ++t) {
            mbar_init(&sm.s_full[t], 1);
            mbar_init(&sm.p_full[t], kBM);
            mbar_init(&sm.o_done[t], 1);
            mbar_init(&sm.o_staged[t], kBM);
            mbar_init(&sm.q_conv[t], kBM);
        }
        mbar_init(&sm.drain, 1);
        sm.abort_flag = 0;
        fence_mbar_init();
        if constexpr (M == kContig) {
            if (n_all > 0) u_begin = producer_start<D, M>(sm, p, &tmQ, &tmK, &tmV, bh, bh_kv, q0, n_all);
        }
    }
    if (warp == Cfg<D>::kMmaWarp) {
        tmem_alloc(&sm.tmem_base, Cfg<D>::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sm.tmem_base;
    WaitCtx wc{&sm.abort_flag, p.status};

    if (warp >= 4 * Cfg<D>::QT) {
        if constexpr (Cfg<D>::kSplitRegs) setmaxnreg_dec<Occ<D, M>::kRegsOther>();
        if (warp == Cfg<D>::kProducerWarp) {
            if (lane == 0 && n_all > 0)
                run_producer<D, M>(sm, p, &tmQ, &tmK, &tmV, b, bh, bh_kv, q0, n_all, u_begin, wc);
        } else if (warp == Cfg<D>::kMmaWarp) {
            if (lane == 0 && n_all > 0) run_mma<D, M>(sm, tmem, n, n_all, wc);
        } else if constexpr (M == kPagedE4m3) {
            // the warps after the MMA issuer's convert e4m3 tiles into the ring
            if (n_all > 0) run_convert<D>(sm, n_all, (int)threadIdx.x - (Cfg<D>::kMmaWarp + 1) * 32, wc);
        }
    } else {
        if constexpr (Cfg<D>::kSplitRegs) setmaxnreg_inc<Occ<D, M>::kRegsSoftmax>();
        const int t = warp >> 2;  // warpgroup = query tile
        run_softmax<D, M>(sm, p, &tmO, tmem, t, bh, q0, n[t], n_all, kv_end, delta, wc);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == Cfg<D>::kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, Cfg<D>::kTmemCols);
    }
}

// The register split of the kernel's warpgroups (setmaxnreg) draws on the block's launch
// allocation; a split larger than it would wait forever.  Checked once per kernel against the
// register count the compiler gave it, before the first launch.
template <int D, int M>
cudaError_t check_register_split() {
    static int verdict = 0;  // 0 unknown, 1 fits, -1 does not
    if (verdict == 0) {
        cudaFuncAttributes fa;
        const cudaError_t e = cudaFuncGetAttributes(&fa, prefill_kernel<D, M>);
        if (e != cudaSuccess) return e;
        const long pool = (long)fa.numRegs * Occ<D, M>::kThreads;
        const long need = 128L * (Cfg<D>::QT * (long)Occ<D, M>::kRegsSoftmax +
                                  (Occ<D, M>::kThreads / 128 - Cfg<D>::QT) * (long)Occ<D, M>::kRegsOther);
        verdict = (!Cfg<D>::kSplitRegs || need <= pool) ? 1 : -1;
    }
    return verdict == 1 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

template <int D, int M>
cudaError_t launch_prefill_dm(const PrefillArgs &a, cudaStream_t stream) {
    CUtensorMap tq, tk, tv, to;
    const int BH = a.B * a.H, BHkv = a.B * a.Hkv;
    bool ok_maps = encode_qkv_map(&tq, a.q, BH, a.Nq, D) && encode_qkv_map(&to, a.o, BH, a.Nq, D);
    if constexpr (M == kPagedBf16)  // pages [num_pages * Hkv] of 16 x D, one 16-row box per page
        ok_maps = ok_maps && encode_qkv_map(&tk, a.k, a.num_pages * a.Hkv, kPageTokens, D, kPageTokens) &&
                  encode_qkv_map(&tv, a.v, a.num_pages * a.Hkv, kPageTokens, D, kPageTokens);
    else if constexpr (M == kContig)  // boxes of kBNd<D> key rows
        ok_maps = ok_maps && encode_qkv_map(&tk, a.k, BHkv, a.Nkv, D, kBNd<D>) &&
                  encode_qkv_map(&tv, a.v, BHkv, a.Nkv, D, kBNd<D>);
    else  // e4m3 pages: one box of 16 rows x 128 codes per page (zeros past d), unswizzled
        ok_maps = ok_maps && encode_page_map_u8(&tk, a.k, a.num_pages * a.Hkv, kPageTokens, D, false) &&
                  encode_page_map_u8(&tv, a.v, a.num_pages * a.Hkv, kPageTokens, D, false);
    if (!ok_maps) return cudaErrorInvalidValue;
    cudaError_t e = check_register_split<D, M>();
    if (e != cudaSuccess) return e;
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
    p.Hkv = a.Hkv;
    p.group = a.H / a.Hkv;
    p.page_table = a.page_table;
    p.ctx_lens = a.ctx_lens;
    p.max_pages = a.max_pages;
    p.num_pages = a.num_pages;
    p.k8 = static_cast<const uint8_t *>(a.k);
    p.v8 = static_cast<const uint8_t *>(a.v);
    p.n_units = (a.Nq + kBM * Cfg<D>::QT - 1) / (kBM * Cfg<D>::QT);
    {
        // about 48 MB of K/V per chunk: two chunks (the one finishing, the one starting) fit
        // in the 126 MB L2 together.  Query heads of one group share their K/V.
        const double elem = (M == kPagedE4m3) ? 1.0 : 2.0;
        const double kv_bytes_per_head = 2.0 * a.Nkv * D * elem / p.group;  // Nkv: capacity when paged
        int hpc = (int)(48.0e6 / kv_bytes_per_head);
        p.heads_per_chunk = hpc < 1 ? 1 : (hpc > BH ? BH : hpc);
    }
    p.scale_log2 = a.scale * kLog2e * (M == kPagedE4m3 ? a.k_scale : 1.f);
    p.o_scale = (M == kPagedE4m3) ? a.v_scale : 1.f;
    const size_t smem = sizeof(PrefillSmem<D, M>) + 1024;
    e = ensure_max_dynamic_smem(reinterpret_cast<const void *>(prefill_kernel<D, M>), (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)((size_t)p.n_units * BH);
    prefill_kernel<D, M><<<grid, Occ<D, M>::kThreads, smem, stream>>>(tq, tk, tv, to, p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_prefill_d(const PrefillArgs &a, cudaStream_t stream) {
    if (!a.paged) return launch_prefill_dm<D, kContig>(a, stream);
    if (a.kv_fp8) return launch_prefill_dm<D, kPagedE4m3>(a, stream);
    return launch_prefill_dm<D, kPagedBf16>(a, stream);
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t stream) {
    switch (a.d) {
        case 32: return launch_prefill_d<32>(a, stream);
        case 64: return launch_prefill_d<64>(a, stream);
        case 80: return launch_prefill_d<80>(a, stream);
        case 96: return launch_prefill_d<96>(a, stream);
        case 128: return launch_prefill_d<128>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace attn
