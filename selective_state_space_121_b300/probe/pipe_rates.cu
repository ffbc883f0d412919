// pipe_rates.cu -- throughput probes for the SM pipes the selective scan is bound by
// (libssmprobe.so, declared in include/ssm_probe.h). Measurement only: nothing in
// libssmscan.so calls it.
//
// Every probe kernel runs a fixed number of independent chains of one instruction
// per thread (shared loads are volatile so that none is merged or hoisted; each
// shuffle takes an integer add and a changing lane mask, so none cancels another), with enough warps per SM to cover its latency, and clocks itself
// with clock64() per block, from a barrier before the loop to a barrier after it.
// All blocks of a launch are resident at once (4 blocks of 256 threads per SM),
// so per-SM throughput = 4 * (work per block) / cycles.
//
// Probes (`which`), each reported as work per clock per SM:
//   0 ex2.approx.ftz.f32      lanes      1 lg2.approx.ftz.f32   lanes
//   2 rcp.approx.ftz.f32      lanes (with one FP32 add per rcp, on another pipe)
//   3 fma.rn.f32              lanes
//   4 fma.rn.f32x2            FP32 FMAs (2 per lane and instruction)
//   5 ld.shared.v4, every lane of the warp at one address          warp instructions
//   6 ld.shared.v4, two addresses (one per half-warp)               warp instructions
//   7 ld.shared.v4, four addresses (one per quarter-warp)           warp instructions
//   8 ld.shared.v4, 32 consecutive 16-byte vectors                  warp instructions
//   9 ld.shared.v2, one address                                     warp instructions
//  10 ld.shared.v2, two addresses (one per half-warp)               warp instructions
//  11 ld.shared.f32, one address                                    warp instructions
//  12 shfl.sync.bfly.b32 (plus one integer add)                    warp instructions
//  13 ld.shared.v4, eight addresses, the same eight in every quarter-warp  warp instructions
//  14 ld.shared.v4, sixteen addresses, the same sixteen in both half-warps warp instructions
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssm_probe.h"

namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerSM = 4;
constexpr int kChains = 8;
constexpr int kIters = 4096;

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2f(float x) {
    float y;
    asm volatile("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcpf(float x) {
    float y;
    asm volatile("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float ffma(float a, float b, float c) {
    float d;
    asm volatile("fma.rn.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
    unsigned long long d;
    asm volatile("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint32_t lds128(uint32_t addr) {
    uint32_t a, b, c, d;
    asm volatile("ld.volatile.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr));
    return a ^ b ^ c ^ d;
}
__device__ __forceinline__ uint32_t lds64(uint32_t addr) {
    uint32_t a, b;
    asm volatile("ld.volatile.shared.v2.u32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "r"(addr));
    return a ^ b;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t a;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(a) : "r"(addr));
    return a;
}

// byte offset a lane reads in the shared-memory probes
template <int which>
__device__ __forceinline__ uint32_t lane_offset(int lane) {
    switch (which) {
        case 6: case 10: return (lane >> 4) * 32;            // one address per half-warp
        case 7: return (lane >> 3) * 32;                     // one per quarter-warp
        case 8: return lane * 16;                            // consecutive vectors
        case 13: return (lane & 7) * 16;                     // eight, repeated per quarter
        case 14: return (lane & 15) * 16;                    // sixteen, repeated per half
        default: return 0;                                   // one address
    }
}

template <int which>
__global__ void __launch_bounds__(kThreads, kBlocksPerSM) probe_kernel(float seed, float* sink, long long* cycles) {
    __shared__ __align__(16) uint32_t s_buf[2048];   // 8 KB
    for (int i = threadIdx.x; i < 2048; i++) s_buf[i] = i * 2654435761u;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const uint32_t base = (uint32_t)__cvta_generic_to_shared(s_buf) + lane_offset<which>(lane);
    constexpr bool kF = which <= 3, kF2 = which == 4, kU = which >= 5;
    float x[kChains];
    unsigned long long x2[kChains];
    uint32_t acc[kChains];
#pragma unroll
    for (int k = 0; k < kChains; k++) {
        if constexpr (kF) x[k] = seed * (float)(k + 1 + threadIdx.x % 7);
        if constexpr (kF2) {
            const float lo = seed * (float)(k + 1), hi = lo + 1.f;
            x2[k] = ((unsigned long long)__float_as_uint(hi) << 32) | __float_as_uint(lo);
        }
        if constexpr (kU) acc[k] = (uint32_t)k;
    }
    const unsigned long long m2 = ((unsigned long long)__float_as_uint(0.999f) << 32) | __float_as_uint(0.999f);
    const unsigned long long a2 = ((unsigned long long)__float_as_uint(1e-3f) << 32) | __float_as_uint(1e-3f);
    __syncthreads();
    const long long t0 = clock64();
    for (int it = 0; it < kIters; it++) {
        const uint32_t off = (uint32_t)(it & 3) * 1024u;    // 4 shared-memory windows of 1 KB
#pragma unroll
        for (int k = 0; k < kChains; k++) {
            if constexpr (which == 0) x[k] = ex2f(-x[k]);
            else if constexpr (which == 1) x[k] = lg2f(x[k]);
            else if constexpr (which == 2) x[k] = rcpf(x[k] + 1.f);
            else if constexpr (which == 3) x[k] = ffma(x[k], 0.999f, 1e-3f);
            else if constexpr (which == 4) x2[k] = ffma2(x2[k], m2, a2);
            else if constexpr (which == 9 || which == 10) acc[k] += lds64(base + off + (uint32_t)k * 128u);
            else if constexpr (which == 11) acc[k] += lds32(base + off + (uint32_t)k * 128u);
            else if constexpr (which == 12) acc[k] = __shfl_xor_sync(0xffffffffu, acc[k] + 1u, 1 + ((it + k) & 15));
            else acc[k] += lds128(base + off + (uint32_t)k * 128u);
        }
    }
    __syncthreads();   // the block's time is its slowest warp's
    const long long t1 = clock64();
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < kChains; k++) {
        if constexpr (kF) s += x[k];
        if constexpr (kF2) s += __uint_as_float((uint32_t)x2[k]) + __uint_as_float((uint32_t)(x2[k] >> 32));
        if constexpr (kU) s += (float)acc[k];
    }
    sink[blockIdx.x * kThreads + threadIdx.x] = s;
    __syncthreads();
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

}  // namespace

extern "C" SSM_PROBE_API int ssm_probe_pipe_rate(int which, double* per_clock_per_sm, double* cycles_out, void* stream) {
    if (which < 0 || which > 14 || !per_clock_per_sm) return -1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -2;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -2;
    const int blocks = sms * kBlocksPerSM;
    float* sink = nullptr;
    long long* cyc = nullptr;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMallocAsync((void**)&sink, sizeof(float) * blocks * kThreads, s) != cudaSuccess) return -3;
    if (cudaMallocAsync((void**)&cyc, sizeof(long long) * blocks, s) != cudaSuccess) return -3;
    using K = void (*)(float, float*, long long*);
    const K kernels[15] = {probe_kernel<0>, probe_kernel<1>, probe_kernel<2>, probe_kernel<3>, probe_kernel<4>,
                           probe_kernel<5>, probe_kernel<6>, probe_kernel<7>, probe_kernel<8>, probe_kernel<9>,
                           probe_kernel<10>, probe_kernel<11>, probe_kernel<12>, probe_kernel<13>,
                           probe_kernel<14>};
    kernels[which]<<<blocks, kThreads, 0, s>>>(0.37f, sink, cyc);   // warm-up
    kernels[which]<<<blocks, kThreads, 0, s>>>(0.41f, sink, cyc);
    long long* host = new long long[blocks];
    int rc = 0;
    if (cudaGetLastError() != cudaSuccess ||
        cudaMemcpyAsync(host, cyc, sizeof(long long) * blocks, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        rc = -4;
    } else {
        long long mx = 0;
        for (int i = 0; i < blocks; i++) mx = host[i] > mx ? host[i] : mx;
        // work per block: threads x chains x iterations, counted per lane (pipes), per FP32
        // FMA (packed: 2 per lane) or per warp instruction (shared memory, shuffle)
        double work = (double)kThreads * kChains * kIters;
        if (which == 4) work *= 2.0;
        if (which >= 5) work /= 32.0;
        *per_clock_per_sm = work * kBlocksPerSM / (double)mx;
        if (cycles_out) *cycles_out = (double)mx;
    }
    delete[] host;
    cudaFreeAsync(sink, s);
    cudaFreeAsync(cyc, s);
    return rc;
}
