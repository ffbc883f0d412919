// kernels_decode.cu -- single-token state update (decode) for the selective scan.
//
// One token of the recurrence (Mamba SSM complete guide (youngju.dev), section 5,
// selective_scan loop body; applied once per token it is the O(1)-per-token
// recurrent inference of the Scalar Mamba1 page's section details):
//     s_n <- exp(dt*A_n) * s_n + dt*B_n*x ;  y = sum_n C_n s_n + D x ;  y *= silu(z)
// on a resident fp32 (batch, dim, dstate) state, in place.
//
// The kernel is HBM-bound (16 bytes of state traffic per (b, d, n) against one
// exp and four fp32 ops), so the layout is chosen for the state stream: each
// channel's dstate floats are split over G = dstate/4 lanes holding 4 states
// each, so a warp reads and writes one contiguous 512-byte run of state with
// 16-byte vector accesses. The per-channel scalars (x, delta, z) are loaded by
// every lane of the channel group (same address, one transaction), and the
// partial C.s sums are reduced across the group with xor shuffles.
#include "common.cuh"
#include "launch.h"

namespace ssm {
namespace {

template <int N, typename Tin, typename Tout>
__global__ void __launch_bounds__(256) state_update_kernel(DecodeArgs a) {
    constexpr int NPL = N < 4 ? N : 4;   // states per lane
    constexpr int G = N / NPL;           // lanes per channel (1, 2 or 4)
    const int64_t nch = a.batch * a.dim;
    const int64_t total = nch * G;
    const Tin* x = static_cast<const Tin*>(a.x);
    const Tin* dl = static_cast<const Tin*>(a.delta);
    const Tin* Bp = static_cast<const Tin*>(a.B);
    const Tin* Cp = static_cast<const Tin*>(a.C);
    const Tin* zp = static_cast<const Tin*>(a.z);
    Tout* y = static_cast<Tout*>(a.y);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    // the loop bound is warp-uniform (base is a multiple of the block size), so the
    // shuffles below always see the whole warp
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < total; base += stride) {
        const int64_t gid = base + threadIdx.x;
        const bool active = gid < total;
        const int64_t ch = active ? gid / G : 0;
        const int j = (int)(gid % G);
        const int64_t b = ch / a.dim, d = ch % a.dim;
        float acc = 0.f, xt = 0.f;
        if (active) {
            xt = to_f32(x[ch]);
            float v = to_f32(dl[ch]) + (a.delta_bias ? a.delta_bias[d] : 0.f);
            const float dt = a.softplus ? softplus(v) : v;
            const float dtl = dt * kLog2e;
            const float dtx = dt * xt;
            float s[NPL];
            float* sp = a.state + ch * N + j * NPL;
            if constexpr (NPL == 4) {
                float4 v4 = *reinterpret_cast<const float4*>(sp);
                s[0] = v4.x; s[1] = v4.y; s[2] = v4.z; s[3] = v4.w;
            } else {
#pragma unroll
                for (int i = 0; i < NPL; i++) s[i] = sp[i];
            }
#pragma unroll
            for (int i = 0; i < NPL; i++) {
                const int n = j * NPL + i;
                const float an = exp2_dec<sizeof(Tin) == 4>(dtl * a.A[d * N + n]);
                s[i] = fmaf(an, s[i], dtx * to_f32(Bp[b * N + n]));
                acc = fmaf(to_f32(Cp[b * N + n]), s[i], acc);
            }
            if constexpr (NPL == 4) {
                *reinterpret_cast<float4*>(sp) = make_float4(s[0], s[1], s[2], s[3]);
            } else {
#pragma unroll
                for (int i = 0; i < NPL; i++) sp[i] = s[i];
            }
        }
#pragma unroll
        for (int off = 1; off < G; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (active && j == 0) {
            float yv = acc + (a.D ? a.D[d] * xt : 0.f);
            if (zp) yv *= silu(to_f32(zp[ch]));
            y[ch] = from_f32<Tout>(yv);
        }
    }
}

template <int N, typename Tin, typename Tout>
cudaError_t launch_n(const DecodeArgs& a, cudaStream_t s) {
    constexpr int G = N < 4 ? 1 : N / 4;
    const int64_t total = a.batch * a.dim * G;
    if (total == 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > (1 << 30)) blocks = 1 << 30;
    state_update_kernel<N, Tin, Tout><<<(unsigned)blocks, 256, 0, s>>>(a);
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
