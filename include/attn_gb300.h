/*
 * attn_gb300.h -- C ABI of the GB300 (sm_103a) exact-attention library.
 *
 * Exact scaled-dot-product attention computed the
 * FlashAttention way (K/V streamed in tiles past a resident Q tile, running
 * max m and normaliser l, accumulator rescaled by exp(m_old - m_new), the
 * score matrix never written to memory):
 *
 *   attn_fwd / attn_fwd_kvlen -- prefill forward, causal or not, emitting O
 *       and the per-row log-sum-exp.  The method: NanoInfer README ("Flash
 *       Attention v1/v2" bullets and the naive-vs-flash paragraph);
 *       gpu-inference blog, section 02 (online softmax, rescale by
 *       exp(m_old - m_new), log-sum-exp saved, causal mask combined with the
 *       padding mask before the softmax); llm-kernel-lib README, kernel 1
 *       (causal tile skipping); Kernel-Inference-Engine README, the tile-loop
 *       flowchart (Q tile held, K/V tiles streamed, normalise and store).
 *
 *   attn_bwd -- the backward of the prefill forward (dQ, dK, dV from the
 *       saved log-sum-exp; gpu-inference blog, section 02).
 *
 *   paged_attn_decode -- one query token per sequence attending over a KV
 *       cache split into fixed-size pages reached through a page table; the
 *       result equals that of a contiguous cache (inference-kernel-cookbook
 *       README, recipes 02 "KV Cache" and 03 "Paged Attention").  Long
 *       contexts are split into chunks whose partial (m, l, O) are merged by
 *       their log-sum-exp weights in a second pass.
 *
 * Definition computed (per batch b, head h, query row i):
 *   J     = { j < Nkv : j < kv_len[b] and (not causal or j <= i + Nkv - Nq) }
 *   s_j   = scale * <q_i, k_j>
 *   O_i   = sum_J exp(s_j - m) v_j / sum_J exp(s_j - m),   m = max_J s_j
 *   LSE_i = m + ln(sum_J exp(s_j - m))        (natural log, of the scaled scores)
 *   A row with no valid key gets O_i = 0 and LSE_i = -inf.
 *   Causal alignment is bottom-right: with Nq < Nkv the queries are the last
 *   Nq positions of the key sequence.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller, contiguous
 *     row-major.  bf16 tensors are passed as void* (storage of __nv_bfloat16).
 *     Every tensor pointer must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  The library never allocates device memory, never copies
 *     between host and device and never synchronises the stream.
 *   - Host-side checks happen before any launch; on error nothing is launched
 *     and the outputs are untouched.
 *   - Device-resident lengths (kv_lens, ctx_lens, page_table) are not read on
 *     the host.  The kernels clamp lengths to [0, capacity] and treat a page id
 *     outside [0, num_pages) as an unmapped page that holds no token (its keys
 *     are skipped, on every paged entry point alike), so bad values give wrong
 *     numbers, never out-of-bounds accesses.
 *   - Every wait inside a kernel is bounded.  A wait that runs out records
 *     ATTN_ERR_DEVICE_TIMEOUT in a device status word and in a host-visible flag
 *     of that device, and the kernel exits cleanly.  The flag is reported without
 *     synchronising: once it is set, every later call that would launch work on
 *     that device returns ATTN_ERR_DEVICE_TIMEOUT and launches nothing, and
 *     attn_last_device_status() returns it, until attn_check_device_status()
 *     clears it.  (A kernel still running when a call is made has not reported
 *     yet; attn_check_device_status() synchronises first.)
 *   - The first call on each device does a one-time set-up with that device
 *     current: a check of the architecture, the lookup of the status word, the
 *     page-locking of the library's static page of host flags (once per process)
 *     and one small synchronous copy into the status word.  Make that first call
 *     before any stream capture.
 *   - Supported: head dim d in {32, 64, 80, 96, 128} for every entry point
 *     (prefill, decode, KV cache, backward); page_size 16.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st *attn_stream_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,     /* null pointer, non-positive size, size overflow */
    ATTN_ERR_UNSUPPORTED = 2,     /* head dim not supported by the call, page_size != 16, no sm_103 device */
    ATTN_ERR_MISALIGNED = 3,      /* a tensor pointer not 16-byte aligned */
    ATTN_ERR_WORKSPACE = 4,       /* workspace missing, misaligned or too small */
    ATTN_ERR_CUDA = 5,            /* a CUDA runtime/driver call or launch failed */
    ATTN_ERR_DEVICE_TIMEOUT = 6,  /* a bounded in-kernel wait ran out (see attn_check_device_status) */
    ATTN_ERR_SCRATCH_LIMIT = 7    /* paged_attn_decode_noalloc: sizes need more than its fixed scratch */
} attn_status_t;

/*
 * Prefill forward.
 *   q   [B, H, Nq,  d] bf16      k, v [B, H, Nkv, d] bf16
 *   o   [B, H, Nq,  d] bf16 (written, round-to-nearest-even from fp32)
 *   lse [B, H, Nq]     fp32 (written; may be NULL to skip)
 *   causal: 0 or 1 (bottom-right aligned).  scale: multiplier of q.k (e.g. 1/sqrt(d)).
 * Returns ATTN_OK or an attn_status_t error code.
 */
int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
             int B, int H, int Nq, int Nkv, int d, int causal, float scale,
             attn_stream_t stream);

/*
 * Prefill forward with per-sequence key padding: key j of sequence b is valid
 * only if j < kv_lens[b] (device int32 [B]; NULL means every key is valid).
 * The padding mask applies to every query row and is ANDed with the causal
 * mask.  Other arguments as attn_fwd.
 */
int attn_fwd_kvlen(const void *q, const void *k, const void *v, void *o, float *lse,
                   int B, int H, int Nq, int Nkv, int d, int causal, float scale,
                   const int32_t *kv_lens, attn_stream_t stream);

/*
 * Prefill forward with grouped-query (or multi-query) attention: Hq query heads
 * share Hkv key/value heads, query head h reading key/value head h / (Hq / Hkv)
 * (the MHA / GQA / MQA variants compared in the llm-kernel-lib README's
 * attention ablation).  q, o [B, Hq, Nq, d]; k, v [B, Hkv, Nkv, d]; lse
 * [B, Hq, Nq]; Hq % Hkv == 0 (else ATTN_ERR_INVALID_ARG).  Hkv == Hq is
 * attn_fwd_kvlen.  Other arguments as attn_fwd_kvlen.
 */
int attn_fwd_gqa(const void *q, const void *k, const void *v, void *o, float *lse,
                 int B, int Hq, int Hkv, int Nq, int Nkv, int d, int causal, float scale,
                 const int32_t *kv_lens, attn_stream_t stream);

/*
 * Bytes of device workspace paged_attn_decode needs for these sizes (0 on
 * invalid sizes).  The caller allocates it (16-byte aligned) and may reuse it
 * across calls on the same stream; calls that overlap on the GPU need
 * separate workspaces.  The size depends on the page table's capacity,
 * max_pages_per_seq * page_size tokens, because the split grid covers every
 * position the table can address.
 */
size_t paged_attn_decode_workspace_size(int B, int H, int d, int max_pages_per_seq,
                                        int page_size);

/*
 * The same size stated by the longest context: max_ctx_len tokens in 16-token
 * pages, i.e. paged_attn_decode_workspace_size(B, H, d, ceil(max_ctx_len / 16),
 * 16).  Pass the capacity of the table the decode will get (max_pages_per_seq *
 * 16), which is at least the longest context.
 */
size_t paged_attn_decode_workspace_size_ctx(int B, int H, int d, int max_ctx_len);

/*
 * Workspace of paged_attn_decode_gqa and paged_attn_decode_fp8 for H query heads
 * over Hkv cache heads.  Groups of two or more query heads run longer splits
 * (1024 tokens instead of 512) and need about half the multi-head size; the
 * multi-head size is always enough.
 */
size_t paged_attn_decode_gqa_workspace_size(int B, int H, int Hkv, int d, int max_pages_per_seq,
                                            int page_size);

/*
 * Paged-KV decode: one query per sequence over its cached tokens.
 *   q          [B, H, d] bf16
 *   k_pages    [num_pages, H, page_size, d] bf16 (one page of one head is a
 *   v_pages     contiguous page_size x d block)
 *   page_table [B, max_pages_per_seq] int32: physical page of logical page p of
 *              sequence b; token t of b is slot t % page_size of page
 *              page_table[b][t / page_size]
 *   ctx_lens   [B] int32: number of cached tokens of each sequence (the query
 *              attends to all of them; clamped to [0, max_pages_per_seq*page_size])
 *   o          [B, H, d] bf16 (written)      lse [B, H] fp32 (written; may be NULL)
 *   workspace  device scratch of at least paged_attn_decode_workspace_size() bytes
 */
int paged_attn_decode(const void *q, const void *k_pages, const void *v_pages,
                      const int32_t *page_table, const int32_t *ctx_lens, int page_size,
                      void *o, float *lse, int B, int H, int d, int max_pages_per_seq,
                      int num_pages, float scale, void *workspace, size_t workspace_bytes,
                      attn_stream_t stream);

/*
 * Paged decode with grouped-query attention: the cache has Hkv heads
 * (k_pages, v_pages [num_pages, Hkv, page_size, d]) shared by the H query heads
 * (q, o [B, H, d]; lse [B, H]); query head h reads cache head h / (H / Hkv), and
 * each cache page is read once for all the query heads that share it.  H % Hkv
 * must be 0.  The workspace is sized by paged_attn_decode_gqa_workspace_size(B,
 * H, Hkv, ...) with H the number of query heads.  Other arguments as
 * paged_attn_decode.
 */
int paged_attn_decode_gqa(const void *q, const void *k_pages, const void *v_pages,
                          const int32_t *page_table, const int32_t *ctx_lens, int page_size,
                          void *o, float *lse, int B, int H, int Hkv, int d, int max_pages_per_seq,
                          int num_pages, float scale, void *workspace, size_t workspace_bytes,
                          attn_stream_t stream);

/*
 * Chunked prefill over the paged KV cache (a prefill step writing into, then
 * attending over, a KV cache kept in pages: inference-kernel-cookbook README,
 * recipes 02 and 03).  Sequence b holds ctx_lens[b] tokens (device int32 [B],
 * clamped to [0, max_pages_per_seq * page_size]) in its pages; the Nq queries
 * q[b, :, i] are its LAST Nq positions (ctx_lens[b] - Nq + i), so with causal = 1
 * query i sees keys j <= i + ctx_lens[b] - Nq (bottom-right), and every query sees
 * only keys j < ctx_lens[b].  The new tokens' K/V must already be in the pages
 * (paged_kv_append).
 *   q, o [B, H, Nq, d] bf16; lse [B, H, Nq] fp32 (may be NULL)
 *   k_pages, v_pages [num_pages, Hkv, page_size, d] bf16; page_table [B, max_pages_per_seq]
 *   H % Hkv == 0 (grouped-query heads as attn_fwd_gqa); page_size 16; d in {32, 64, 80, 96, 128}.
 * A page id outside [0, num_pages) is an unmapped page, as in decode: the positions
 * it covers hold no token (their keys are masked out; the other positions keep their
 * places, so the causal alignment is unchanged), and a query that sees no mapped key
 * gets O = 0 and LSE = -inf.  Runs on the same tcgen05 pipeline as attn_fwd, with
 * each 128-key tile gathered page by page through TMA.
 */
int paged_attn_prefill(const void *q, const void *k_pages, const void *v_pages,
                       const int32_t *page_table, const int32_t *ctx_lens, int page_size,
                       void *o, float *lse, int B, int H, int Hkv, int Nq, int d,
                       int max_pages_per_seq, int num_pages, int causal, float scale,
                       attn_stream_t stream);

/*
 * Appends the K/V of Nnew new tokens to the paged cache: token t of sequence b
 * goes to position p = start_pos[b] + t, i.e. page page_table[b][p / page_size],
 * slot p % page_size, for every key/value head.
 *   k_new, v_new [B, Hkv, Nnew, d] bf16; k_pages, v_pages [num_pages, Hkv, page_size, d]
 *   start_pos [B] int32 (device; tokens already in the cache before this append)
 * Positions past max_pages_per_seq * page_size and page ids outside [0, num_pages)
 * are skipped (nothing written).  The caller reserves the pages in the table.
 */
int paged_kv_append(const void *k_new, const void *v_new, void *k_pages, void *v_pages,
                    const int32_t *page_table, const int32_t *start_pos, int page_size,
                    int B, int Hkv, int Nnew, int d, int max_pages_per_seq, int num_pages,
                    attn_stream_t stream);

/*
 * FP8 KV cache.  The NanoInfer README's roadmap names FP8 e4m3 storage (cuda_fp8.h
 * __nv_fp8_e4m3) as the successor of INT8 with the quantisation math unchanged;
 * here it is the storage of the paged KV cache, which halves the bytes a decode
 * step reads.  A cache tensor holds E4M3 codes (1 sign, 4 exponent bits with bias
 * 7, 3 mantissa bits, no infinities, largest finite 448) with one scale per
 * tensor:  value = e4m3(code) * scale.  Conversion from bf16:
 *   code = e4m3 nearest-even rounding of fp32(x) * fp32(1 / scale), saturating at
 *          +-448 (1 / scale is computed in fp32 on the host).
 *
 * paged_attn_prefill_fp8: paged_attn_prefill over an e4m3 cache (k_pages, v_pages
 *   [num_pages, Hkv, page_size, d] uint8 codes; k_scale, v_scale > 0 and finite): the
 *   chunked prefill of a serving loop that keeps its cache in e4m3.  q, o, lse, the
 *   table, the masks and the result are as in paged_attn_prefill, for the dequantised
 *   cache.  The codes are widened exactly to f16 in shared memory and both products run
 *   in f16 with fp32 accumulation: each query row is rounded to f16 after a power-of-two
 *   factor that keeps it below 2^15 (exact for bf16 values in f16's normal range).  The
 *   key scale multiplies the scores and the value scale the output.
 * paged_attn_decode_fp8: paged_attn_decode_gqa over an e4m3 cache (k_pages,
 *   v_pages [num_pages, Hkv, page_size, d] uint8 codes; k_scale, v_scale > 0
 *   and finite).  q, o, lse, the table, the workspace and the result are as in
 *   paged_attn_decode_gqa, for the dequantised cache.  The codes are widened exactly
 *   to f16 or fp32; where the products run on tensor cores they run in f16 with fp32
 *   accumulation, the query rounded to f16 after a power-of-two factor as above.
 * kv_quantize_fp8: n contiguous bf16 elements of src -> n codes in dst (n a
 *   multiple of 8; both 16-byte aligned).  Converts a whole bf16 page pool.
 * paged_kv_append_fp8: paged_kv_append into an e4m3 cache, converting each new
 *   element with the tensor's scale.
 */
int paged_attn_decode_fp8(const void *q, const void *k_pages, const void *v_pages, float k_scale,
                          float v_scale, const int32_t *page_table, const int32_t *ctx_lens,
                          int page_size, void *o, float *lse, int B, int H, int Hkv, int d,
                          int max_pages_per_seq, int num_pages, float scale, void *workspace,
                          size_t workspace_bytes, attn_stream_t stream);

int paged_attn_prefill_fp8(const void *q, const void *k_pages, const void *v_pages, float k_scale,
                           float v_scale, const int32_t *page_table, const int32_t *ctx_lens,
                           int page_size, void *o, float *lse, int B, int H, int Hkv, int Nq, int d,
                           int max_pages_per_seq, int num_pages, int causal, float scale,
                           attn_stream_t stream);

int kv_quantize_fp8(const void *src, void *dst, size_t n, float scale, attn_stream_t stream);

int paged_kv_append_fp8(const void *k_new, const void *v_new, void *k_pages, void *v_pages,
                        float k_scale, float v_scale, const int32_t *page_table,
                        const int32_t *start_pos, int page_size, int B, int Hkv, int Nnew, int d,
                        int max_pages_per_seq, int num_pages, attn_stream_t stream);

/*
 * Backward of attn_fwd_gqa: gradients of the loss with respect to q, k and v
 * given its gradient dout with respect to the forward output.  The method
 * (gpu-inference blog, section 02 "FlashAttention-2 in Triton"): the
 * probabilities are recomputed tile by tile from the forward's log-sum-exp
 * instead of being stored, and the work is three kernels -- the row term
 * D_i = dO_i . O_i, a dK/dV kernel and a dQ kernel.  With P_ij = exp(s_ij -
 * LSE_i) on the valid keys (0 elsewhere), dP = dO V^T and dS = P * (dP - D):
 *   dV = P^T dO,   dK = scale dS^T Q,   dQ = scale dS K;
 * for grouped-query heads dK and dV of a key/value head sum over the query
 * heads that read it.  A row with no valid key contributes nothing.
 *   q, o, dout, dq [B, Hq, Nq, d] bf16    k, v, dk, dv [B, Hkv, Nkv, d] bf16
 *   lse [B, Hq, Nq] fp32: the forward's log-sum-exp (natural log), required
 *   o: the forward's output for these inputs (used only for D)
 *   kv_lens, causal, scale, Hq % Hkv == 0: exactly as in the forward call
 *   workspace: device scratch of at least attn_bwd_workspace_size(B, Hq, Nq)
 *       bytes, 16-byte aligned; it holds D [B, Hq, Nq] fp32 when the call ends.
 * dq, dk and dv are fully written (rows past a sequence's key length get zero
 * dk/dv).  Products run on bf16 operands with fp32 accumulation: P and dS are
 * rounded to bf16 before they multiply dO, Q and K.  d in {32, 64, 80, 96, 128}.
 */
size_t attn_bwd_workspace_size(int B, int Hq, int Nq);

int attn_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
             const void *dout, void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int Nq,
             int Nkv, int d, int causal, float scale, const int32_t *kv_lens, void *workspace,
             size_t workspace_bytes, attn_stream_t stream);

/*
 * paged_attn_decode for callers that cannot allocate device memory.  The pages
 * describe no such variant; it exists for callers such as code running inside
 * a memory pool or allocator callback (where a nested cudaMalloc is not
 * allowed), serving loops that must not block on the allocator or risk an
 * out-of-memory failure in the middle of a step, and hosts that can only pass
 * the input and output buffers they already own.
 *
 * Arguments, layouts and results are those of paged_attn_decode without the
 * workspace: the chunk partials live in a fixed 12 MiB array inside the
 * library's device memory (every GPU that loads the library holds it until the
 * process exits).  Sizes whose workspace (paged_attn_decode_workspace_size)
 * exceeds 12 MiB are rejected with ATTN_ERR_SCRATCH_LIMIT before anything is
 * launched.  No call allocates or frees memory.
 *
 * The first call on each device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  All calls
 * share the one array: calls that may overlap on the GPU (other streams, other
 * host threads) race on it and must be ordered by the caller.  A call that
 * completes normally writes every part of the array it later reads, so what an
 * earlier call left there does not reach its result.  A call whose bounded wait
 * runs out (ATTN_ERR_DEVICE_TIMEOUT) is different: the split that gave up does
 * not write its partial, and the merge may then read an earlier call's partial
 * from the array, so that call's O and LSE are invalid (as the status says).
 */
int paged_attn_decode_noalloc(const void *q, const void *k_pages, const void *v_pages,
                              const int32_t *page_table, const int32_t *ctx_lens, int page_size,
                              void *o, float *lse, int B, int H, int d, int max_pages_per_seq,
                              int num_pages, float scale, attn_stream_t stream);

/*
 * Synchronises `stream`, then returns and clears the current device's status
 * (the device word and the host-visible flag): ATTN_OK,
 * ATTN_ERR_DEVICE_TIMEOUT if a kernel's bounded wait ran out since the last
 * check, or ATTN_ERR_CUDA if the synchronisation itself failed.  After it the
 * other entry points launch work again.
 */
int attn_check_device_status(attn_stream_t stream);

/*
 * The current device's host-visible timeout flag, read without synchronising
 * and without clearing it: ATTN_ERR_DEVICE_TIMEOUT if a kernel that has already
 * reached its timeout path recorded one since the last attn_check_device_status(),
 * else ATTN_OK.  The same condition makes the launching entry points return
 * ATTN_ERR_DEVICE_TIMEOUT.  (The op sequence of the Kernel-Inference-Engine
 * README reads the error state right after a launch, with no host round trip;
 * this is that check for the asynchronous in-kernel timeouts.)
 */
int attn_last_device_status(void);

/*
 * Self-test of the failure detection: launches one block whose only thread waits
 * on an mbarrier that nothing arrives on.  The wait gives up after its limit
 * (about two seconds), records ATTN_ERR_DEVICE_TIMEOUT in the device status word
 * and the kernel returns normally, so the CUDA context stays usable.  The next
 * attn_check_device_status() on this stream returns ATTN_ERR_DEVICE_TIMEOUT.
 * Returns ATTN_OK if the launch succeeded.
 */
int attn_selftest_bounded_wait(attn_stream_t stream);

/* Static, human-readable text for a status code. */
const char *attn_status_string(int status);

/* Library version as "major.minor.patch" (static string). */
const char *attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
