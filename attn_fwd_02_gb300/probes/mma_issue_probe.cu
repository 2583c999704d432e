// mma_issue_probe.cu -- how fast one thread can feed the sm_103a tensor core.
//
// Standalone measurement behind the prefill kernel's MMA-issuing code (not part of the
// library).  One CTA per SM; thread 0 issues a long run of 128 x 128 x 16 bf16 products
// (tcgen05.mma, fp32 accumulate in TMEM) with three styles of issue code, then commits
// and waits.  Printed per style: issue cycles per MMA (until the last one is accepted)
// and total cycles per MMA (until all have completed).  A 128 x 128 x 16 product is 64
// cycles of tensor work at the full rate (8192 dense bf16 FLOP per cycle per SM).
//
//   per-MMA descriptors: every MMA rebuilds both shared-memory descriptors from an address
//                        (and / shift / or) -- the form the kernels first used;
//   advanced descriptors: each buffer's descriptor is built once and advanced by a constant
//                        per MMA (sdesc_advance) -- the kernels' current form;
//   8-MMA asm block:     eight MMAs in one asm statement over precomputed descriptors.
// A last pair of lines runs the 8-MMA groups alone and with four other warps streaming the
// prefill softmax's TMEM traffic (score loads, P stores) on other columns.
//
// Build and run on a GB300 (from the repository root):
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//        -o /tmp/mma_issue_probe attn_fwd_02_gb300/probes/mma_issue_probe.cu && /tmp/mma_issue_probe
// Operands are zeros in shared memory; every access stays inside the 48 KB operand region
// (operand tiles of 16 KB at offsets up to 24.6 KB; 64 KB for the two-box groups of the last
// pair) and the 512 TMEM columns the CTA allocates; the waits and the streaming loop are bounded.
#include <cstdio>

#include <cuda_runtime.h>

#include "../csrc/sm103_ptx.cuh"

using namespace attn;

enum Style { kPerMma = 0, kAdvanced = 1, kBlock8 = 2 };

__global__ void __launch_bounds__(128, 1) issue_probe(long long *out, int *status, int nblk, int style, int ts) {
    extern __shared__ uint8_t raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar;
    __shared__ uint32_t tbase;
    const int warp = threadIdx.x / 32;
    for (int i = threadIdx.x; i < 48 * 1024 / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tbase, 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tbase;
    if (threadIdx.x == 0) {
        const uint32_t a = smem_u32(smem), b = smem_u32(smem + 16384);
        constexpr uint32_t id = idesc_bf16_f32(128, 128, false, false);
        const uint64_t da = sdesc_sw128(a, 16, 1024), db = sdesc_sw128(b, 16, 1024);
        const uint64_t da1 = sdesc_sw128(a + 4096, 16, 1024), db1 = sdesc_sw128(b + 4096, 16, 1024);
        const uint32_t ta = tmem + 384;  // A operand of the TMEM form: 8 columns per 16 k
        WaitCtx wc{nullptr, status};
        const long long t0 = clock64();
        for (int i = 0; i < nblk; ++i) {
            if (style == kBlock8 && !ts) {
                asm volatile(
                    "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, 1, 0;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %5, %3, p;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %7, %3, p;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %9, %3, p;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %5, %3, p;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %7, %3, p;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %9, %3, p;\n\t}" ::"r"(tmem),
                    "l"(da), "l"(db), "r"(id), "l"(da + 2), "l"(db + 2), "l"(da + 4), "l"(db + 4), "l"(da + 6),
                    "l"(db + 6)
                    : "memory");
            } else if (style == kBlock8) {
                asm volatile(
                    "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, 1, 0;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %5, %3, p;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], [%6], %7, %3, p;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], [%8], %9, %3, p;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %5, %3, p;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], [%6], %7, %3, p;\n\t"
                    "tcgen05.mma.cta_group::1.kind::f16 [%0], [%8], %9, %3, p;\n\t}" ::"r"(tmem),
                    "r"(ta), "l"(db), "r"(id), "r"(ta + 8), "l"(db + 2), "r"(ta + 16), "l"(db + 4), "r"(ta + 24),
                    "l"(db + 6)
                    : "memory");
            } else {
                // as in the kernels, the buffer changes from one group of 8 to the next (a ring
                // slot), so nothing can be hoisted out of the loop
                const uint32_t sel = (uint32_t)(i & 1) << 12;
                const uint64_t da_i = (i & 1) ? da1 : da, db_i = (i & 1) ? db1 : db;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (uint32_t)((kk >> 2) * 4096 + (kk & 3) * 32);
                    const uint64_t ad = style == kPerMma ? sdesc_sw128(a + sel + off, 16, 1024) : sdesc_advance(da_i, off);
                    const uint64_t bd = style == kPerMma ? sdesc_sw128(b + sel + off, 16, 1024) : sdesc_advance(db_i, off);
                    if (ts)
                        tc_mma_ts(tmem, ta + (uint32_t)((kk & 3) * 8), bd, id, 1u);
                    else
                        tc_mma_ss(tmem, ad, bd, id, 1u);
                }
            }
        }
        const long long t1 = clock64();
        tc_commit(&bar);
        (void)mbar_wait(&bar, 0, wc, 1);
        const long long t2 = clock64();
        out[blockIdx.x * 2 + 0] = t1 - t0;
        out[blockIdx.x * 2 + 1] = t2 - t0;
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}


// The same 8-MMA groups (A and B in shared memory, D in TMEM columns 0-127) while warps 4-7
// stream the prefill softmax's TMEM traffic on other columns: 128 fp32 columns loaded
// (256-383) and 64 columns of bf16 pairs stored (384-447) per round, as one tile of scores
// and its P.  Warp w accesses TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31.
__global__ void __launch_bounds__(256, 1) tmem_traffic_probe(long long *out, int *status, int nblk, int traffic) {
    extern __shared__ uint8_t raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar;
    __shared__ uint32_t tbase;
    __shared__ volatile int stop;
    const int warp = threadIdx.x / 32;
    for (int i = threadIdx.x; i < 48 * 1024 / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        stop = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tbase, 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tbase;
    if (threadIdx.x == 0) {
        const uint32_t a = smem_u32(smem), b = smem_u32(smem + 16384);
        constexpr uint32_t id = idesc_bf16_f32(128, 128, false, false);
        const uint64_t da = sdesc_sw128(a, 16, 1024), db = sdesc_sw128(b, 16, 1024);
        WaitCtx wc{nullptr, status};
        const long long t0 = clock64();
        for (int i = 0; i < nblk; ++i) tc_mma_ss_k8_box16k(tmem, da, db, id, 1u);
        tc_commit(&bar);
        (void)mbar_wait(&bar, 0, wc, 1);
        out[blockIdx.x] = clock64() - t0;
        stop = 1;
    } else if (warp >= 4 && traffic) {
        const uint32_t lane_base = tmem + ((uint32_t)((warp % 4) * 32) << 16);
        uint32_t acc = 0;
        for (int it = 0; !stop && it < (1 << 20); ++it) {
            uint32_t r[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + 256 + c * 32, r[c]);
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_wait_ld(r[c]);
            uint32_t pk[4][16];
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int i = 0; i < 16; ++i) pk[c][i] = r[c][2 * i] ^ r[c][2 * i + 1];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_st16(lane_base + 384 + c * 16, pk[c]);
            tmem_wait_st();
            acc ^= pk[0][0];
        }
        if (acc == 0x12345678u) status[1] = (int)acc;  // keeps the loop's work
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

int main() {
    const int grid = 152, nblk = 64, smem = 48 * 1024 + 1024;
    long long *d_out;
    int *d_status;
    cudaMalloc(&d_out, grid * 2 * sizeof(long long));
    cudaMalloc(&d_status, 2 * sizeof(int));
    cudaMemset(d_status, 0, 2 * sizeof(int));
    cudaFuncSetAttribute(issue_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    const char *names[] = {"per-MMA descriptors", "advanced descriptors", "8-MMA asm block"};
    printf("one thread per SM, %d x 128x128x16 bf16 MMAs (64 cycles each at the full rate)\n", nblk * 8);
    for (int ts = 0; ts < 2; ++ts)
        for (int style = 0; style < 3; ++style) {
            for (int rep = 0; rep < 2; ++rep) issue_probe<<<grid, 128, smem>>>(d_out, d_status, nblk, style, ts);
            if (cudaDeviceSynchronize() != cudaSuccess) {
                printf("launch failed\n");
                return 1;
            }
            long long h[grid * 2];
            cudaMemcpy(h, d_out, sizeof(h), cudaMemcpyDeviceToHost);
            double iss = 0, tot = 0;
            for (int g = 0; g < grid; ++g) {
                iss += h[2 * g];
                tot += h[2 * g + 1];
            }
            const double n = (double)grid * nblk * 8;
            printf("%s %-22s issue %6.1f  total %6.1f cycles per MMA\n", ts ? "A in TMEM " : "A in smem ", names[style],
                   iss / n, tot / n);
        }
    // the two-box groups read B up to 48.1 KB past the aligned base: 64 KB of operand space here
    const int smem_tt = 64 * 1024 + 1024;
    cudaFuncSetAttribute(tmem_traffic_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_tt);
    for (int traffic = 0; traffic < 2; ++traffic) {
        for (int rep = 0; rep < 2; ++rep) tmem_traffic_probe<<<grid, 256, smem_tt>>>(d_out, d_status, nblk, traffic);
        if (cudaDeviceSynchronize() != cudaSuccess) {
            printf("launch failed\n");
            return 1;
        }
        long long h[grid * 2];
        cudaMemcpy(h, d_out, grid * sizeof(long long), cudaMemcpyDeviceToHost);
        double tot = 0;
        for (int g = 0; g < grid; ++g) tot += h[g];
        printf("A in smem  8-MMA asm block, %-36s total %6.1f cycles per MMA\n",
               traffic ? "4 warps streaming TMEM loads/stores" : "TMEM otherwise idle", tot / ((double)grid * nblk * 8));
    }
    int st[2];
    cudaMemcpy(st, d_status, sizeof(st), cudaMemcpyDeviceToHost);
    printf("bounded-wait status %d\n", st[0]);
    return st[0] != 0;
}
