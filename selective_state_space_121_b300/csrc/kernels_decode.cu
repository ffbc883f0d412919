// kernels_decode.cu -- single-token state update (decode) for the selective scan.
//
// One token of the recurrence (Mamba SSM complete guide (youngju.dev), section 5,
// the selective_scan loop body; applied once per token it is the O(1)-per-token
// recurrent inference of the SM1 (Scalar Mamba1) page's section details):
//     s_n <- exp(dt*A_n) * s_n + dt*B_n*x ;  y = sum_n C_n s_n + D x ;  y *= silu(z)
// on a resident fp32 (batch, dim, dstate) state, in place.
//
// The kernel is HBM-bound: 8 bytes of state traffic per (b, d, n) (read + write)
// against one exp and four FP32 operations. Layout of the work:
//  * a thread owns NPL = min(dstate, 4) consecutive states of one channel d
//    (G = dstate/NPL lanes per channel, adjacent lanes), so a warp reads and writes
//    512 contiguous bytes of state per batch row with 16-byte accesses;
//  * the thread walks R batch rows (b0, b0 + gridDim.y, ...), keeping its A
//    values in registers, and issues all R state loads before using any, so R x 16
//    bytes per thread are in flight;
//  * a lane's 4 values of the B and C rows are one vector load each (8 bytes of
//    bf16, 16 of fp32) when aligned; x, delta, z are per (b, d) scalars shared by
//    the G lanes of a channel;
//  * the partial C.s sums of a channel are reduced over its G lanes with xor
//    shuffles.
#include "common.cuh"
#include "launch.h"

namespace ssm {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 4;   // batch rows per thread

// NPL consecutive values widened to fp32: one 8- or 16-byte load when kVec (the
// host checked the alignment), element loads otherwise.
template <int NPL, bool kVec, typename T>
__device__ __forceinline__ void load_vec(const T* p, float* out) {
    if constexpr (kVec && NPL == 4 && sizeof(T) == 2) {
        const uint2 r = *reinterpret_cast<const uint2*>(p);
        out[0] = __uint_as_float(r.x << 16); out[1] = __uint_as_float(r.x & 0xffff0000u);
        out[2] = __uint_as_float(r.y << 16); out[3] = __uint_as_float(r.y & 0xffff0000u);
    } else if constexpr (kVec && NPL == 4 && sizeof(T) == 4) {
        const float4 r = *reinterpret_cast<const float4*>(p);
        out[0] = r.x; out[1] = r.y; out[2] = r.z; out[3] = r.w;
    } else {
#pragma unroll
        for (int i = 0; i < NPL; i++) out[i] = to_f32(p[i]);
    }
}

template <int N, typename Tin, typename Tout, bool kVec>
__global__ void __launch_bounds__(kThreads) state_update_kernel(DecodeArgs a) {
    constexpr int NPL = N < 4 ? N : 4;   // states per lane
    constexpr int G = N / NPL;           // lanes per channel (1, 2 or 4)
    using Dec = Decay<sizeof(Tin) == 4>;
    const Tin* xp = static_cast<const Tin*>(a.x);
    const Tin* dp = static_cast<const Tin*>(a.delta);
    const Tin* Bp = static_cast<const Tin*>(a.B);
    const Tin* Cp = static_cast<const Tin*>(a.C);
    const Tin* zp = static_cast<const Tin*>(a.z);
    Tout* y = static_cast<Tout*>(a.y);

    // every thread of the block runs every shuffle below (the row loop is uniform
    // across the block); threads past the last channel or row carry zeros
    const int64_t gid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t d = gid / G;
    const int j = (int)(gid % G);
    const bool dok = d < a.dim;
    float Al[NPL];
    const float bias = (dok && a.delta_bias) ? a.delta_bias[d] : 0.f;
    const float Dd = (dok && a.D) ? a.D[d] : 0.f;
    if (dok) load_vec<NPL, kVec>(a.A + d * N + j * NPL, Al);

    for (int64_t b0 = blockIdx.y; b0 < a.batch; b0 += (int64_t)gridDim.y * kRows) {
        float s[kRows][NPL];
        float xt[kRows], dv[kRows], zv[kRows];
        bool ok[kRows];
#pragma unroll
        for (int r = 0; r < kRows; r++) {
            const int64_t b = b0 + (int64_t)r * gridDim.y;
            ok[r] = dok && b < a.batch;
            if (ok[r]) {
                const float* sp = a.state + (b * a.dim + d) * N + j * NPL;
                if constexpr (NPL == 4) {
                    const float4 v = *reinterpret_cast<const float4*>(sp);
                    s[r][0] = v.x; s[r][1] = v.y; s[r][2] = v.z; s[r][3] = v.w;
                } else {
#pragma unroll
                    for (int i = 0; i < NPL; i++) s[r][i] = sp[i];
                }
                const int64_t ch = b * a.dim + d;
                xt[r] = to_f32(xp[ch]);
                dv[r] = to_f32(dp[ch]);
                zv[r] = zp ? to_f32(zp[ch]) : 0.f;
            } else {
#pragma unroll
                for (int i = 0; i < NPL; i++) s[r][i] = 0.f;
                xt[r] = dv[r] = zv[r] = 0.f;
            }
        }
#pragma unroll
        for (int r = 0; r < kRows; r++) {
            const int64_t b = b0 + (int64_t)r * gridDim.y;
            float acc = 0.f;
            if (ok[r]) {
                float Bv[NPL], Cv[NPL];
                load_vec<NPL, kVec>(Bp + b * N + j * NPL, Bv);
                load_vec<NPL, kVec>(Cp + b * N + j * NPL, Cv);
                const float v = dv[r] + bias;
                const float dt = a.softplus ? softplus(v) : v;
                const float dts = dt * Dec::scale;
                const float dtx = dt * xt[r];
#pragma unroll
                for (int i = 0; i < NPL; i++) {
                    s[r][i] = Dec::step(Dec::make(dts * Al[i]), s[r][i], dtx * Bv[i]);
                    acc = fmaf(Cv[i], s[r][i], acc);
                }
                float* sp = a.state + (b * a.dim + d) * N + j * NPL;
                if constexpr (NPL == 4) {
                    *reinterpret_cast<float4*>(sp) = make_float4(s[r][0], s[r][1], s[r][2], s[r][3]);
                } else {
#pragma unroll
                    for (int i = 0; i < NPL; i++) sp[i] = s[r][i];
                }
            }
#pragma unroll
            for (int off = 1; off < G; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (ok[r] && j == 0) {
                float yv = fmaf(Dd, xt[r], acc);
                if (zp) yv *= silu(zv[r]);
                y[b * a.dim + d] = from_f32<Tout>(yv);
            }
        }
    }
}

template <int N, typename Tin, typename Tout>
cudaError_t launch_n(const DecodeArgs& a, cudaStream_t s) {
    constexpr int G = N < 4 ? 1 : N / 4;
    if (a.batch == 0 || a.dim == 0) return cudaSuccess;
    const int64_t bx = (a.dim * G + kThreads - 1) / kThreads;
    // enough CTAs to fill the GPU several times over, each thread kRows rows deep
    int64_t by = (a.batch + kRows - 1) / kRows;
    if (by > 65535) by = 65535;
    if (bx > ((int64_t)1 << 31) - 1) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)bx, (unsigned)by);
    if (a.vec) state_update_kernel<N, Tin, Tout, true><<<grid, kThreads, 0, s>>>(a);
    else state_update_kernel<N, Tin, Tout, false><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
cudaError_t launch_t(const DecodeArgs& a, cudaStream_t s) {
    switch (a.dstate) {
        case 1: return launch_n<1, Tin, Tout>(a, s);
        case 2: return launch_n<2, Tin, Tout>(a, s);
        case 4: return launch_n<4, Tin, Tout>(a, s);
        case 8: return launch_n<8, Tin, Tout>(a, s);
        case 16: return launch_n<16, Tin, Tout>(a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_state_update(const DecodeArgs& a, cudaStream_t s) {
    if (a.in_dtype == kBF16) {
        return a.out_dtype == kBF16 ? launch_t<__nv_bfloat16, __nv_bfloat16>(a, s)
                                    : launch_t<__nv_bfloat16, float>(a, s);
    }
    return a.out_dtype == kBF16 ? launch_t<float, __nv_bfloat16>(a, s) : launch_t<float, float>(a, s);
}

}  // namespace ssm
