// host_link_probe.cu -- host<->device bandwidth over the CPU-GPU link of a Grace-Blackwell node.
//
// Standalone measurement behind the end-to-end figures (not part of the library): a step that copies
// its inputs from pinned host memory and its outputs back cannot run faster than this link.  Measures
// copy-engine transfers (cudaMemcpyAsync, one per chunk, the 512 MiB buffer split over 1-8 streams)
// host-to-device, device-to-host and both at once, and the same transfers done by SM loads and
// stores of the mapped pinned buffer (a grid-stride 16-byte copy kernel; every index < n16).
//
// Build and run on a GB300 (from the repository root):
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//        -o /tmp/host_link_probe attn_fwd_02_gb300/probes/host_link_probe.cu && /tmp/host_link_probe
#include <cstdio>
#include <cstring>
#include <cuda_runtime.h>

__global__ void kcopy(const int4 *__restrict__ src, int4 *__restrict__ dst, size_t n16) {
    size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x, stride = (size_t)gridDim.x * blockDim.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        int4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
        dst[i] = a; dst[i + stride] = b; dst[i + 2 * stride] = c; dst[i + 3 * stride] = d;
    }
    for (; i < n16; i += stride) dst[i] = src[i];
}

#define CK(x) do { cudaError_t e = (x); if (e != cudaSuccess) { printf("%s: %s\n", #x, cudaGetErrorString(e)); return 1; } } while (0)

int main() {
    const size_t bytes = 512ull << 20;
    void *h, *h2, *d, *d2;
    CK(cudaHostAlloc(&h, bytes, cudaHostAllocDefault));
    CK(cudaHostAlloc(&h2, bytes, cudaHostAllocDefault));
    CK(cudaMalloc(&d, bytes));
    CK(cudaMalloc(&d2, bytes));
    memset(h, 1, bytes); memset(h2, 2, bytes);
    CK(cudaMemset(d, 0, bytes)); CK(cudaMemset(d2, 0, bytes));
    cudaStream_t s[8];
    for (auto &x : s) CK(cudaStreamCreateWithFlags(&x, cudaStreamNonBlocking));
    cudaEvent_t e0, e1, ej[8];
    CK(cudaEventCreate(&e0)); CK(cudaEventCreate(&e1));
    for (auto &x : ej) CK(cudaEventCreateWithFlags(&x, cudaEventDisableTiming));
    int dev; CK(cudaGetDevice(&dev));
    int sms; CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    // mode: 0 = copy-engine H2D, 1 = copy-engine D2H, 2 = both at once; chunks split over streams
    for (int mode = 0; mode < 3; ++mode)
        for (int chunks : {1, 2, 4, 8}) {
            float best = 1e9;
            for (int rep = 0; rep < 4; ++rep) {
                CK(cudaDeviceSynchronize());
                CK(cudaEventRecord(e0, s[0]));
                for (int c = 1; c < 8; ++c) CK(cudaStreamWaitEvent(s[c], e0));
                const size_t per = bytes / chunks;
                for (int c = 0; c < chunks; ++c) {
                    const size_t off = c * per;
                    if (mode == 0 || mode == 2)
                        CK(cudaMemcpyAsync((char *)d + off, (char *)h + off, per, cudaMemcpyHostToDevice, s[c]));
                    if (mode == 1 || mode == 2)
                        CK(cudaMemcpyAsync((char *)h2 + off, (char *)d2 + off, per, cudaMemcpyDeviceToHost,
                                           s[mode == 2 ? (c + chunks) % 8 : c]));
                }
                for (int c = 1; c < 8; ++c) { CK(cudaEventRecord(ej[c], s[c])); CK(cudaStreamWaitEvent(s[0], ej[c])); }
                CK(cudaEventRecord(e1, s[0]));
                CK(cudaEventSynchronize(e1));
                float ms; CK(cudaEventElapsedTime(&ms, e0, e1));
                if (ms < best) best = ms;
            }
            printf("copy engine %-4s chunks=%d: %7.1f GB/s per direction (%.3f ms for 512 MiB)\n",
                   mode == 0 ? "H2D" : mode == 1 ? "D2H" : "both", chunks, bytes / best / 1e6, best);
        }
    // SM loads/stores of mapped pinned memory (the pinned pointer is valid on the device under UVA)
    for (int mode = 0; mode < 3; ++mode)
        for (int per_sm : {1, 2, 4, 8}) {
            float best = 1e9;
            const size_t n16 = bytes / 16;
            for (int rep = 0; rep < 4; ++rep) {
                CK(cudaDeviceSynchronize());
                CK(cudaEventRecord(e0, s[0]));
                CK(cudaStreamWaitEvent(s[1], e0));
                if (mode == 0 || mode == 2) kcopy<<<sms * per_sm, 512, 0, s[0]>>>((const int4 *)h, (int4 *)d, n16);
                if (mode == 1 || mode == 2) kcopy<<<sms * per_sm, 512, 0, s[1]>>>((const int4 *)d2, (int4 *)h2, n16);
                CK(cudaGetLastError());
                CK(cudaEventRecord(ej[1], s[1]));
                CK(cudaStreamWaitEvent(s[0], ej[1]));
                CK(cudaEventRecord(e1, s[0]));
                CK(cudaEventSynchronize(e1));
                float ms; CK(cudaEventElapsedTime(&ms, e0, e1));
                if (ms < best) best = ms;
            }
            printf("SM copy     %-4s CTAs/SM=%d: %7.1f GB/s per direction (%.3f ms)\n",
                   mode == 0 ? "H2D" : mode == 1 ? "D2H" : "both", per_sm, bytes / best / 1e6, best);
        }
    // check the SM copies moved the data
    unsigned char probe_d = 0, probe_h = ((unsigned char *)h2)[bytes - 1];
    CK(cudaMemcpy(&probe_d, (char *)d + bytes - 1, 1, cudaMemcpyDeviceToHost));
    printf("check: device byte %d (want 1), host byte %d (want 0)\n", probe_d, probe_h);
    return 0;
}
