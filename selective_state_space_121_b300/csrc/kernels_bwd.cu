// kernels_bwd.cu -- backward of the selective scan (gradients for training).
//
// The forward (Mamba SSM complete guide (youngju.dev), section 5, "complete Mamba
// implementation": selective_scan, ssm, forward):
//     dt_t = softplus(delta_t + bias),  a_tn = exp(dt_t A_n),
//     h_tn = a_tn h_{t-1,n} + dt_t B_tn u_t,  y_t = sum_n C_tn h_tn + D u_t,
//     out_t = y_t silu(z_t).
// The pages print no backward; this is the chain rule through those steps in
// reverse time. With g_n = dl/dh_tn, carried from t = L-1 down to 0 (starting at
// dl/dh_last):
//     dy = dout silu(z),  dz = dout y silu'(z),  g_n += C_tn dy
//     dC_tn += dy h_tn,   dD += dy u,           du = D dy + sum_n g_n dt B_tn
//     d(dt) = sum_n g_n (h_{t-1,n} a_tn A_n + B_tn u),  dA_n += g_n h_{t-1,n} a_tn dt
//     dB_tn += g_n dt u,  ddelta = d(dt) softplus'(delta + bias),  dbias += ddelta
//     g_n *= a_tn;  finally dh0 = g.
// dB and dC sum over the channels of a batch row, dA, dD and dbias over batch rows
// (and time).
//
// Layout: as the forward's serial kernel, G lanes per channel (NPL = min(N, 4)
// states each), P = 32/G channels per warp, the lanes of one state group
// consecutive; a CTA holds 4 warps of one batch row. Two phases:
//   1. forward over the whole sequence, h only, writing the state at every
//      8-step chunk start to the workspace (B, D, ceil(L/8), N) fp32;
//   2. chunks in reverse: the chunk's 8 states are recomputed from its checkpoint
//      into registers, then the 8 steps run backwards. Per step, the per-channel
//      sums (y for dz, d(dt), du) are xor-shuffle reductions over the channel's G
//      lanes; dB and dC of the step are reduce-scattered over the warp's P
//      channels (each lane ends with one (n, B-or-C) total) and added to global
//      memory with one atomic per lane. B and C of a chunk are staged in shared
//      memory for the CTA's channels (one batch row).
// fp32 arithmetic; for fp32 inputs exp and softplus take the accurate forms.
#include "common.cuh"
#include "launch.h"

namespace ssm {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kT = 8;   // steps per chunk (checkpoint spacing)

template <int N> struct BwdCfg {
    static constexpr int NPL = N < 4 ? N : 4;   // states per lane
    static constexpr int G = N / NPL;           // lanes per channel
    static constexpr int P = 32 / G;            // channels per warp
    static constexpr int M = 2 * NPL;           // dB and dC values per lane-step
};

// kT values of row[t ..] as fp32 (zero past L or when !ok)
template <typename T, bool kVec>
__device__ __forceinline__ void load_run(const T* row, int64_t t, int64_t L, bool ok, float* out) {
    if (!ok) {
#pragma unroll
        for (int k = 0; k < kT; k++) out[k] = 0.f;
        return;
    }
    if (kVec && t + kT <= L) {
        constexpr int V = Vec16<T>::kN;
#pragma unroll
        for (int k = 0; k < kT; k += V) Vec16<T>::load(row + t + k, out + k);
        return;
    }
#pragma unroll
    for (int k = 0; k < kT; k++) out[k] = (t + k < L) ? to_f32(row[t + k]) : 0.f;
}

template <typename T, bool kVec>
__device__ __forceinline__ void store_run(T* row, int64_t t, int64_t L, const float* v) {
    if (kVec && t + kT <= L) {
        constexpr int V = Vec16<T>::kN;
#pragma unroll
        for (int k = 0; k < kT; k += V) Vec16<T>::store(row + t + k, v + k);
        return;
    }
#pragma unroll
    for (int k = 0; k < kT; k++)
        if (t + k < L) row[t + k] = from_f32<T>(v[k]);
}

template <bool kAcc> __device__ __forceinline__ float exp_f(float x) {
    if constexpr (kAcc) return exp_acc(x);
    else return ex2(x * kLog2e);
}

template <bool kAcc> __device__ __forceinline__ float sigmoid_f(float x) {
    // 1 / (1 + exp(-x)), argument capped so exp stays finite (sigmoid < 2e-35 there)
    const float e = exp_f<kAcc>(fminf(-x, 80.f));
    if constexpr (kAcc) {
        const float den = 1.f + e;
        float q = rcp(den);
        return fmaf(q, fmaf(-q, den, 1.f), q);
    } else {
        return rcp(1.f + e);
    }
}

// sum over the G lanes of a channel (lanes p, p + P, p + 2P, ...)
template <int G, int P>
__device__ __forceinline__ float chan_sum(float v) {
#pragma unroll
    for (int m = P; m < 32; m <<= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

template <int N, typename Tin, typename Tdo, bool kVec>
__global__ void __launch_bounds__(kThreads) scan_bwd_kernel(BwdArgs a) {
    using Cfg = BwdCfg<N>;
    constexpr int NPL = Cfg::NPL, G = Cfg::G, P = Cfg::P, M = Cfg::M;
    constexpr bool kAcc = sizeof(Tin) == 4;
    __shared__ __align__(16) float s_bc[kT][2][N];   // the chunk's B (0) and C (1)

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int p = lane % P, j = lane / P;
    const int64_t b = blockIdx.y;
    const int64_t d = ((int64_t)blockIdx.x * kWarps + warp) * P + p;
    const bool ok = d < a.dim;
    const int64_t L = a.seqlen, ch = b * a.dim + d;
    const int64_t nchunk = (L + kT - 1) / kT;
    const Tin* u_r = static_cast<const Tin*>(a.u) + ch * L;
    const Tin* dl_r = static_cast<const Tin*>(a.delta) + ch * L;
    const Tin* z_r = a.z ? static_cast<const Tin*>(a.z) + ch * L : nullptr;
    const Tdo* do_r = static_cast<const Tdo*>(a.dout) + ch * L;
    const Tin* B_b = static_cast<const Tin*>(a.B) + b * N * L;
    const Tin* C_b = static_cast<const Tin*>(a.C) + b * N * L;
    float* ws = static_cast<float*>(a.workspace) + ch * nchunk * N + j * NPL;

    float A[NPL], h[NPL], g[NPL], dA[NPL];
#pragma unroll
    for (int i = 0; i < NPL; i++) {
        A[i] = ok ? a.A[d * N + j * NPL + i] : 0.f;
        h[i] = (ok && a.h0) ? a.h0[ch * N + j * NPL + i] : 0.f;
        g[i] = (ok && a.dh_last) ? a.dh_last[ch * N + j * NPL + i] : 0.f;
        dA[i] = 0.f;
    }
    const float bias = (ok && a.delta_bias) ? a.delta_bias[d] : 0.f;
    const float Dd = (ok && a.D) ? a.D[d] : 0.f;

    // the chunk's B (and C) for the CTA's batch row, fp32 [t][which][n]
    auto stage = [&](int64_t t0, bool with_c) {
        __syncthreads();   // previous readers are done
        for (int v = threadIdx.x; v < (with_c ? 2 : 1) * N * kT; v += kThreads) {
            const int which = v / (N * kT), n = (v / kT) % N, k = v % kT;
            const int64_t t = t0 + k;
            const Tin* src = which ? C_b : B_b;
            s_bc[k][which][n] = t < L ? to_f32(src[(int64_t)n * L + t]) : 0.f;
        }
        __syncthreads();
    };
    auto dt_of = [&](float x) {
        if (!a.softplus) return x;
        return softplus_acc<kAcc>(x);
    };

    // 1. forward, checkpointing the state at every chunk start
    for (int64_t c = 0; c < nchunk; c++) {
        const int64_t t0 = c * kT;
        if (ok) {
            if constexpr (NPL == 4) {
                *reinterpret_cast<float4*>(ws + c * N) = make_float4(h[0], h[1], h[2], h[3]);
            } else {
#pragma unroll
                for (int i = 0; i < NPL; i++) ws[c * N + i] = h[i];
            }
        }
        float u[kT], dl[kT];
        load_run<Tin, kVec>(u_r, t0, L, ok, u);
        load_run<Tin, kVec>(dl_r, t0, L, ok, dl);
        stage(t0, false);
#pragma unroll
        for (int k = 0; k < kT; k++) {
            float dt = dt_of(dl[k] + bias);
            if (t0 + k >= L) dt = 0.f;
#pragma unroll
            for (int i = 0; i < NPL; i++)
                h[i] = fmaf(exp_f<kAcc>(dt * A[i]), h[i], dt * u[k] * s_bc[k][0][j * NPL + i]);
        }
    }

    // 2. chunks in reverse
    float dD = 0.f, dbias = 0.f;
    for (int64_t c = nchunk - 1; c >= 0; c--) {
        const int64_t t0 = c * kT;
        float u[kT], dl[kT], zz[kT], dout[kT];
        load_run<Tin, kVec>(u_r, t0, L, ok, u);
        load_run<Tin, kVec>(dl_r, t0, L, ok, dl);
        load_run<Tdo, kVec>(do_r, t0, L, ok, dout);
        if (z_r) load_run<Tin, kVec>(z_r, t0, L, ok, zz);
        float hs[kT + 1][NPL];   // hs[k] = state before step k; hs[kT] after the chunk
        if (ok) {
            if constexpr (NPL == 4) {
                const float4 v = *reinterpret_cast<const float4*>(ws + c * N);
                hs[0][0] = v.x; hs[0][1] = v.y; hs[0][2] = v.z; hs[0][3] = v.w;
            } else {
#pragma unroll
                for (int i = 0; i < NPL; i++) hs[0][i] = ws[c * N + i];
            }
        } else {
#pragma unroll
            for (int i = 0; i < NPL; i++) hs[0][i] = 0.f;
        }
        stage(t0, true);
        float dts[kT];
#pragma unroll
        for (int k = 0; k < kT; k++) {
            dts[k] = dt_of(dl[k] + bias);
            if (t0 + k >= L) dts[k] = 0.f;
#pragma unroll
            for (int i = 0; i < NPL; i++)
                hs[k + 1][i] = fmaf(exp_f<kAcc>(dts[k] * A[i]), hs[k][i], dts[k] * u[k] * s_bc[k][0][j * NPL + i]);
        }
        float du[kT], ddl[kT], dz[kT];
#pragma unroll
        for (int k = kT - 1; k >= 0; k--) {
            const bool live = t0 + k < L;
            const float* Bk = s_bc[k][0] + j * NPL;
            const float* Ck = s_bc[k][1] + j * NPL;
            float dy = live ? dout[k] : 0.f;
            if (z_r) {
                float part = 0.f;
#pragma unroll
                for (int i = 0; i < NPL; i++) part = fmaf(Ck[i], hs[k + 1][i], part);
                const float y = chan_sum<G, P>(part) + Dd * u[k];
                const float s = sigmoid_f<kAcc>(zz[k]);
                dz[k] = dy * y * s * fmaf(zz[k], 1.f - s, 1.f);
                dy *= zz[k] * s;
            }
            dD = fmaf(dy, u[k], dD);
            float vals[M];
            float ddt_p = 0.f, du_p = 0.f;
#pragma unroll
            for (int i = 0; i < NPL; i++) {
                g[i] = fmaf(Ck[i], dy, g[i]);
                vals[NPL + i] = dy * hs[k + 1][i];                    // dC
                const float an = exp_f<kAcc>(dts[k] * A[i]);
                const float ga = g[i] * hs[k][i] * an;                  // g h_{t-1} a
                ddt_p = fmaf(ga, A[i], ddt_p);
                ddt_p = fmaf(g[i] * Bk[i], u[k], ddt_p);
                dA[i] = fmaf(ga, dts[k], dA[i]);
                vals[i] = g[i] * dts[k] * u[k];                         // dB
                du_p = fmaf(g[i] * dts[k], Bk[i], du_p);
                g[i] *= an;
            }
            const float ddt = chan_sum<G, P>(ddt_p);
            du[k] = fmaf(Dd, dy, chan_sum<G, P>(du_p));
            float dx = ddt;
            if (a.softplus) dx = ddt * sigmoid_f<kAcc>(dl[k] + bias);
            if (!live) dx = 0.f;
            ddl[k] = dx;
            dbias += dx;
            // dB, dC of this step: reduce-scatter over the warp's P channels
            int idx = 0;
            int cnt = M;
#pragma unroll
            for (int m = 1; m < P; m <<= 1) {
                if (cnt > 1) {
                    const int half = cnt / 2;
                    const bool up = (lane & m) != 0;
#pragma unroll
                    for (int q = 0; q < M / 2; q++) {
                        if (q < half) {
                            const float send = up ? vals[q] : vals[half + q];
                            const float keep = up ? vals[half + q] : vals[q];
                            vals[q] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                        }
                    }
                    idx += up ? half : 0;
                    cnt = half;
                } else {
                    vals[0] += __shfl_xor_sync(0xffffffffu, vals[0], m);
                }
            }
            // lanes whose channel bits above the index bits are zero hold the totals
            if (live && (p / M) == 0) {
                const int which = idx / NPL, n = j * NPL + idx % NPL;
                atomicAdd((which ? a.dC : a.dB) + (b * N + n) * L + t0 + k, vals[0]);
            }
        }
        if (ok && j == 0) {
            store_run<Tin, kVec>(static_cast<Tin*>(a.du) + ch * L, t0, L, du);
            store_run<Tin, kVec>(static_cast<Tin*>(a.ddelta) + ch * L, t0, L, ddl);
            if (z_r) store_run<Tin, kVec>(static_cast<Tin*>(a.dz) + ch * L, t0, L, dz);
        }
    }
    if (ok) {
#pragma unroll
        for (int i = 0; i < NPL; i++) {
            atomicAdd(a.dA + d * N + j * NPL + i, dA[i]);
            if (a.dh0) a.dh0[ch * N + j * NPL + i] = g[i];
        }
        if (j == 0) {
            if (a.dD) atomicAdd(a.dD + d, dD);
            if (a.ddelta_bias) atomicAdd(a.ddelta_bias + d, dbias);
        }
    }
}

template <int N, typename Tin, typename Tdo>
cudaError_t launch_n(const BwdArgs& a, cudaStream_t s) {
    using Cfg = BwdCfg<N>;
    if (a.batch == 0 || a.dim == 0) return cudaSuccess;
    dim3 grid((unsigned)((a.dim + kWarps * Cfg::P - 1) / (kWarps * Cfg::P)), (unsigned)a.batch);
    if (a.vec) scan_bwd_kernel<N, Tin, Tdo, true><<<grid, kThreads, 0, s>>>(a);
    else scan_bwd_kernel<N, Tin, Tdo, false><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin, typename Tdo>
cudaError_t by_n(const BwdArgs& a, cudaStream_t s) {
    switch (a.dstate) {
        case 1: return launch_n<1, Tin, Tdo>(a, s);
        case 2: return launch_n<2, Tin, Tdo>(a, s);
        case 4: return launch_n<4, Tin, Tdo>(a, s);
        case 8: return launch_n<8, Tin, Tdo>(a, s);
        case 16: return launch_n<16, Tin, Tdo>(a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

size_t scan_bwd_workspace_bytes(int64_t batch, int64_t dim, int64_t seqlen, int dstate) {
    return (size_t)batch * dim * ((seqlen + kT - 1) / kT) * dstate * 4;
}

cudaError_t launch_scan_bwd(const BwdArgs& a, cudaStream_t s) {
    if (a.in_dtype == kBF16)
        return a.dout_dtype == kBF16 ? by_n<__nv_bfloat16, __nv_bfloat16>(a, s) : by_n<__nv_bfloat16, float>(a, s);
    return a.dout_dtype == kBF16 ? by_n<float, __nv_bfloat16>(a, s) : by_n<float, float>(a, s);
}

}  // namespace ssm
