// tma_latency_probe.cu -- cycles per 64-KB K/V unit delivered by TMA into shared memory.
//
// Standalone measurement behind the prefill kernel's K/V ring (not part of the library).
// One CTA per SM; thread 0 streams units of four 128-row x 64-column bf16 boxes (128-byte
// swizzle, the kernel's K/V box) through a ring of R slots (R units in flight), and reports
// the cycles per unit.  Variants:
//   source:    a 50 MB tensor (resident in L2 after the first pass) or a 500 MB one (HBM);
//   in flight: R = 1 or 2;
//   pattern:   "staggered" (CTAs of one head read different tiles at a time) or "lockstep"
//              (all CTAs of a head read the same tile at the same time, as concurrently
//              running query units of one head do in the prefill);
//   neighbour: a second warp of the CTA issuing 128 x 128 x 16 MMAs with both operands in
//              shared memory back to back (about 120 B/clk of operand reads), or idle.
//
// Build and run on a GB300 (from the repository root):
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//        -o /tmp/tma_latency_probe attn_fwd_02_gb300/probes/tma_latency_probe.cu && /tmp/tma_latency_probe
// Every box lies inside the tensor (rows r0 .. r0+255 < 8192, heads < the tensor's count),
// the MMA operands lie in the third 64-KB slot (unused by the ring when R <= 2), the MMA
// loop ends when the loads are done or after 2^22 MMAs, and every wait is bounded.
#include <cstdio>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../csrc/sm103_ptx.cuh"

using namespace attn;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kN = 8192;      // rows per head
constexpr int kUnits = 256;   // units streamed per CTA
constexpr int kUnitBytes = 65536;

__global__ void __launch_bounds__(64, 1) ring_probe(const __grid_constant__ CUtensorMap tm, int R, int heads,
                                                   int lockstep, int with_mma, long long *out, int *status) {
    extern __shared__ uint8_t raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full[2];
    __shared__ uint64_t done;
    __shared__ uint32_t tbase;
    __shared__ volatile int stop;
    const int warp = threadIdx.x / 32;
    if (threadIdx.x == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(&done, 1);
        stop = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&tbase, 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tbase;
    WaitCtx wc{nullptr, status};
    if (threadIdx.x == 0) {
        const int head = blockIdx.x % heads, tiles = kN / 256;
        const long long t0 = clock64();
        for (int u = 0; u < kUnits; ++u) {
            const int slot = u % R, use = u / R;
            if (use > 0 && !mbar_wait(&full[slot], (uint32_t)((use - 1) & 1), wc, 1)) break;
            mbar_arrive_expect_tx(&full[slot], kUnitBytes);
            const int r0 = ((lockstep ? u : u + (int)blockIdx.x) % tiles) * 256;
            uint8_t *dst = smem + slot * kUnitBytes;
            tma_load_3d(dst, &tm, &full[slot], 0, r0, head);
            tma_load_3d(dst + 16384, &tm, &full[slot], 64, r0, head);
            tma_load_3d(dst + 32768, &tm, &full[slot], 0, r0 + 128, head);
            tma_load_3d(dst + 49152, &tm, &full[slot], 64, r0 + 128, head);
        }
        for (int u = (kUnits > R ? kUnits - R : 0); u < kUnits; ++u)
            (void)mbar_wait(&full[u % R], (uint32_t)((u / R) & 1), wc, 2);
        out[blockIdx.x] = clock64() - t0;
        stop = 1;
    } else if (threadIdx.x == 32 && with_mma) {
        const uint32_t a = smem_u32(smem + 2 * kUnitBytes), b = smem_u32(smem + 2 * kUnitBytes + 16384);
        constexpr uint32_t id = idesc_bf16_f32(128, 128, false, false);
        const uint64_t da = sdesc_sw128(a, 16, 1024), db = sdesc_sw128(b, 16, 1024);
        for (long long n = 0; !stop && n < (1 << 22); n += 8) {
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
        }
        tc_commit(&done);
        (void)mbar_wait(&done, 0, wc, 3);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

int main() {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return 1;
    EncodeTiledFn encode = reinterpret_cast<EncodeTiledFn>(fn);
    const int grid = 152, smem = 3 * kUnitBytes + 1024;
    long long *d_out;
    int *d_status;
    cudaMalloc(&d_out, grid * sizeof(long long));
    cudaMalloc(&d_status, 2 * sizeof(int));
    cudaMemset(d_status, 0, 2 * sizeof(int));
    cudaFuncSetAttribute(ring_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    printf("cycles per 64-KB unit (four 128x64 bf16 boxes), one CTA per SM, %d units each\n", kUnits);
    for (int heads : {24, 240}) {  // 50 MB: L2-resident after the first pass; 500 MB: from HBM
        void *buf = nullptr;
        const size_t bytes = (size_t)heads * kN * 128 * 2;
        if (cudaMalloc(&buf, bytes) != cudaSuccess) return 1;
        cudaMemset(buf, 0, bytes);
        CUtensorMap tm;
        cuuint64_t dims[3] = {128, (cuuint64_t)kN, (cuuint64_t)heads};
        cuuint64_t strides[2] = {256, (cuuint64_t)kN * 256};
        cuuint32_t box[3] = {64, 128, 1};
        cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, buf, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return 1;
        for (int with_mma = 0; with_mma < 2; ++with_mma)
            for (int lockstep = 0; lockstep < 2; ++lockstep)
                for (int R = 1; R <= 2; ++R) {
                    const int hx = heads == 24 ? 12 : heads;  // 12 CTAs per head on the L2 tensor
                    for (int rep = 0; rep < 2; ++rep)
                        ring_probe<<<grid, 64, smem>>>(tm, R, hx, lockstep, with_mma, d_out, d_status);
                    if (cudaDeviceSynchronize() != cudaSuccess) {
                        printf("launch failed\n");
                        return 1;
                    }
                    long long h[grid];
                    cudaMemcpy(h, d_out, sizeof(h), cudaMemcpyDeviceToHost);
                    double cyc = 0;
                    for (int g = 0; g < grid; ++g) cyc += h[g];
                    printf("%-4s R=%d %-9s %-16s %6.0f cycles per unit\n", heads == 24 ? "L2" : "HBM", R,
                           lockstep ? "lockstep" : "staggered", with_mma ? "SS MMAs alongside" : "loads alone",
                           cyc / grid / kUnits);
                }
        cudaFree(buf);
    }
    int st[2];
    cudaMemcpy(st, d_status, sizeof(st), cudaMemcpyDeviceToHost);
    printf("bounded-wait status %d\n", st[0]);
    return st[0] != 0;
}
