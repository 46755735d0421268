// GB300 memory-path ceilings that the MSDA kernels are designed against.
//
// Measures, on one GPU: (1) gather throughput when each group of lanes reads a
// contiguous chunk of 16..512 bytes at a random chunk position, from an
// L1-resident, an L2-resident and a DRAM-sized footprint; (2) vector
// red.global.add throughput (f32 and bf16x2) versus chunk size and footprint;
// (3) shared-memory atomicAdd throughput; (4) TMA bulk reductions
// (cp.reduce.async.bulk ... add.f32) versus size.
// Build and run: nvcc -gencode arch=compute_103a,code=sm_103a -O3 -std=c++17 \
//                  -o /tmp/memprobe memprobe.cu && /tmp/memprobe
// Every index is masked into a power-of-two buffer, so every access is in
// bounds; no kernel waits on another.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>

#define CK(x) do { cudaError_t e = (x); if (e != cudaSuccess) { printf("CUDA %s at %d\n", cudaGetErrorString(e), __LINE__); return 1; } } while (0)

__device__ __forceinline__ uint32_t hsh(uint32_t x) {
    x ^= x >> 16; x *= 0x7feb352du; x ^= x >> 15; x *= 0x846ca68bu; x ^= x >> 16; return x;
}

// Each group of LPC lanes reads one chunk of LPC*16 contiguous bytes; PAIR:
// groups 2k, 2k+1 read the two halves of one 2*LPC*16-byte region.
template <int LPC, bool PAIR>
__global__ void gather(const uint4* __restrict__ buf, uint32_t mask, int iters, uint4* out, long long* cyc) {
    const int lane = threadIdx.x & 31, grp = lane / LPC, r = lane % LPC;
    const uint32_t wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    uint4 acc = make_uint4(0, 0, 0, 0);
    long long t0 = clock64();
    for (int it = 0; it < iters; it += 4) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            uint32_t key = PAIR ? (grp >> 1) : grp;
            uint32_t c = hsh(wid * 7919u + (uint32_t)(it + u) * 131u + key) & mask;
            if (PAIR) c = ((c >> 1) << 1) | (grp & 1);
            v[u] = __ldg(buf + (size_t)c * LPC + r);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) { acc.x ^= v[u].x; acc.y += v[u].y; acc.z ^= v[u].z; acc.w += v[u].w; }
    }
    long long t1 = clock64();
    out[blockIdx.x * blockDim.x + threadIdx.x] = acc;
    if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}

template <int LPC>
__global__ void redk(float* buf, uint32_t mask, int iters) {
    const int lane = threadIdx.x & 31, grp = lane / LPC, r = lane % LPC;
    const uint32_t wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    for (int it = 0; it < iters; ++it) {
        uint32_t c = hsh(wid * 7919u + (uint32_t)it * 131u + grp) & mask;
        float* p = buf + ((size_t)c * LPC + r) * 4;
        asm volatile("red.global.add.v4.f32 [%0], {%1,%1,%1,%1};" :: "l"(p), "f"(1.0f) : "memory");
    }
}

template <int LPC>
__global__ void redbf(uint4* buf, uint32_t mask, int iters) {
    const int lane = threadIdx.x & 31, grp = lane / LPC, r = lane % LPC;
    const uint32_t wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    for (int it = 0; it < iters; ++it) {
        uint32_t c = hsh(wid * 7919u + (uint32_t)it * 131u + grp) & mask;
        uint4* p = buf + (size_t)c * LPC + r;
        asm volatile("red.global.add.noftz.v4.bf16x2 [%0], {%1,%1,%1,%1};" :: "l"(p), "r"(0x3f803f80u) : "memory");
    }
}

__global__ void smem_red(int iters, float* out) {
    __shared__ float s[8192];
    for (int i = threadIdx.x; i < 8192; i += blockDim.x) s[i] = 0.f;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int it = 0; it < iters; ++it) {
        int idx = ((warp * 37 + it * 13) & 255) * 32 + lane;   // conflict-free rows of 32 words
        atomicAdd(&s[idx], 1.0f);
    }
    __syncthreads();
    if (threadIdx.x == 0) out[blockIdx.x] = s[0];
}


// One thread per bulk reduction of CB bytes of 1.0f from shared memory.
__global__ void bulk_red(float* g, uint32_t mask, int iters, int cb) {
    __shared__ __align__(128) float sm[256];
    for (int i = threadIdx.x; i < 256; i += blockDim.x) sm[i] = 1.0f;
    __syncthreads();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const uint32_t wid = (blockIdx.x * blockDim.x + threadIdx.x);
    const uint32_t src = (uint32_t)__cvta_generic_to_shared(sm);
    for (int it = 0; it < iters; ++it) {
        uint32_t c = hsh(wid * 7919u + (uint32_t)it * 131u) & mask;
        float* dst = g + (size_t)c * (cb / 4);
        asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;"
                     :: "l"(dst), "r"(src), "r"(cb) : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        if ((it & 7) == 7) asm volatile("cp.async.bulk.wait_group.read 8;" ::: "memory");
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

template <typename K>
float time_it(K launch) {
    cudaEvent_t a, b; cudaEventCreate(&a); cudaEventCreate(&b);
    launch(); cudaDeviceSynchronize();
    cudaEventRecord(a); launch(); cudaEventRecord(b); cudaEventSynchronize(b);
    float ms; cudaEventElapsedTime(&ms, a, b); return ms;
}

int main() {
    int sms; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    const int blocks = sms * 8, threads = 256, iters = 2048;
    const size_t big = 256ull << 20;   // 256 MiB
    uint4* buf; float* fbuf; uint4* out; long long* cyc; float* o2;
    CK(cudaMalloc(&buf, big)); CK(cudaMemset(buf, 1, big));
    CK(cudaMalloc(&fbuf, big)); CK(cudaMemset(fbuf, 0, big));
    CK(cudaMalloc(&out, (size_t)blocks * threads * sizeof(uint4)));
    CK(cudaMalloc(&cyc, blocks * sizeof(long long)));
    CK(cudaMalloc(&o2, blocks * sizeof(float)));
    printf("sms %d\n", sms);
    long long hc[4096];
    auto report = [&](const char* name, int lpc, size_t foot, float ms) {
        double bytes = (double)blocks * threads * iters * 16.0;
        cudaMemcpy(hc, cyc, blocks * sizeof(long long), cudaMemcpyDeviceToHost);
        double c = 0; for (int i = 0; i < blocks; ++i) c += hc[i]; c /= blocks;
        printf("%-26s chunk %4d B foot %9zu B: %8.3f ms  %8.1f GB/s  %6.1f B/clk/SM(at cycles/block %.0f)\n",
               name, lpc * 16, foot, ms, bytes / ms / 1e6, bytes / sms / (c * 1.0), c);
    };
#define G(LPC, PAIR, FOOT) { size_t chunks = (FOOT) / (LPC * 16); uint32_t mask = (uint32_t)chunks - 1; \
    float ms = time_it([&]{ gather<LPC, PAIR><<<blocks, threads>>>(buf, mask, iters, out, cyc); }); \
    CK(cudaGetLastError()); report(PAIR ? "gather-paired" : "gather", LPC, FOOT, ms); }
    for (size_t foot : {(size_t)32 << 10, (size_t)16 << 20, (size_t)256 << 20}) {
        G(1, false, foot) G(2, false, foot) G(4, false, foot) G(4, true, foot) G(8, false, foot)
        G(16, false, foot) G(32, false, foot)
    }
#define R(LPC, FOOT) { size_t chunks = (FOOT) / (LPC * 16); uint32_t mask = (uint32_t)chunks - 1; \
    float ms = time_it([&]{ redk<LPC><<<blocks, threads>>>(fbuf, mask, iters / 4); }); CK(cudaGetLastError()); \
    double bytes = (double)blocks * threads * (iters / 4) * 16.0; \
    printf("red.v4.f32     chunk %4d B foot %9zu B: %8.3f ms  %8.1f GB/s of red data  %.2f Gred-instr/s\n", LPC * 16, (size_t)(FOOT), ms, bytes / ms / 1e6, (double)blocks * threads / 32 * (iters / 4) / ms / 1e6); }
    for (size_t foot : {(size_t)16 << 10, (size_t)1 << 20, (size_t)64 << 20, (size_t)256 << 20}) { R(2, foot) R(4, foot) R(8, foot) }
#define RB(LPC, FOOT) { size_t chunks = (FOOT) / (LPC * 16); uint32_t mask = (uint32_t)chunks - 1; \
    float ms = time_it([&]{ redbf<LPC><<<blocks, threads>>>(buf, mask, iters / 4); }); CK(cudaGetLastError()); \
    double bytes = (double)blocks * threads * (iters / 4) * 16.0; \
    printf("red.v4.bf16x2  chunk %4d B foot %9zu B: %8.3f ms  %8.1f GB/s of red data\n", LPC * 16, (size_t)(FOOT), ms, bytes / ms / 1e6); }
    for (size_t foot : {(size_t)1 << 20, (size_t)64 << 20}) { RB(4, foot) RB(8, foot) }
    {
        float ms = time_it([&]{ smem_red<<<blocks, threads>>>(iters, o2); }); CK(cudaGetLastError());
        double ops = (double)blocks * threads * iters;
        printf("smem atomicAdd f32: %.3f ms  %.1f Gop/s  %.2f warp-instr/clk/SM at 2.0GHz\n", ms, ops / ms / 1e6, ops / 32 / (ms * 1e-3) / sms / 2.0e9);
    }
    for (int cb : {128, 256, 512, 1024}) {
        size_t foot = (size_t)64 << 20; uint32_t mask = (uint32_t)(foot / cb) - 1;
        for (int thr : {32, 256}) {
            int it2 = 256;
            float ms = time_it([&]{ bulk_red<<<blocks, thr>>>(fbuf, mask, it2, cb); }); CK(cudaGetLastError());
            double bytes = (double)blocks * thr * it2 * cb;
            printf("bulk-reduce f32 %4d B, %3d thr/blk: %8.3f ms  %8.1f GB/s of red data\n", cb, thr, ms, bytes / ms / 1e6);
        }
    }
    return 0;
}
