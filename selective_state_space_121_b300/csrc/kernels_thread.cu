// kernels_thread.cu -- time-serial selective scan: each channel's N-wide state is
// split over G lanes (G = 1, 2 or 4) and every lane walks time step by step.
//
// Same operation as the warp-scan kernels (Mamba SSM complete guide
// (youngju.dev), section 5, selective_scan + softplus(dt) + silu(z) gate):
//     h_t = exp(dt_t A) h_{t-1} + dt_t B_t u_t,  y_t = C_t . h_t + D u_t,  y_t *= silu(z_t)
// Why a second algorithm: the recurrence for one (channel, state) pair is a chain
// of one FMA per step, and with many channels (batch * dim in the tens of
// thousands) there is enough independent work without splitting time. Walking
// time serially costs 4 FP32 ops + 1 ex2 per (t, n) element and nothing else --
// no shuffle scan, no second pass -- while the warp-shuffle scan pays ~2x in FP32
// ops and reads B/C per element. B300 executes 128 FP32 lanes and 32 ex2 per SM
// per clock, so the N = 16 bf16 scan is bound by these pipes, not by HBM, and the
// cheaper formulation wins whenever the channel count fills the GPU.
//
// Per warp: CPW = 32/G channels of one batch row, processed in chunks of
// T = 16*G time steps in three phases:
//   A. prologue, one lane per (channel, 16 bytes of consecutive steps): vector
//      loads of u and delta, dt = softplus(delta + bias), writes (dt*log2 e, dt*u)
//      to smem; keeps D*u and z in registers for phase C;
//   B. recurrence, lane (g, j) owns channel g, states [j*N/G, (j+1)*N/G): per step
//      it reads (dt*log2 e, dt*u) of its channel and the B, C values of its
//      states (fp32, [t][n] layout, identical across the warp's channels, so the
//      loads broadcast), updates its states and writes its partial C.h to smem;
//   C. epilogue, same lane mapping as A: sums the G partials, adds D*u, applies
//      silu(z), stores y with vector stores.
// The B/C tile of the chunk is staged once per CTA (4 warps share the batch row),
// double-buffered, and the next chunk's u/delta/z/B/C are loaded into registers
// while the current chunk computes.
#include <string.h>

#include "common.cuh"
#include "launch.h"

namespace ssm {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;

__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    float2 d;
    asm("mul.rn.f32x2 %0, %1, %2;"
        : "=l"(*reinterpret_cast<unsigned long long*>(&d))
        : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)));
    return d;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(*reinterpret_cast<unsigned long long*>(&d))
        : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)),
          "l"(*reinterpret_cast<unsigned long long*>(&c)));
    return d;
}

template <int N, int G, typename Tin>
struct TSConfig {
    static constexpr int NPL = N / G;               // states per lane
    static constexpr int CPW = 32 / G;              // channels per warp
    static constexpr int T = 16 * G;                // steps per chunk
    static constexpr int V = 16 / sizeof(Tin);      // steps per 16-byte vector
    static constexpr int PV = CPW * T / V / 32;     // vectors per lane per tensor (phase A/C)
    static constexpr int BCV = N * T / V;           // vectors per B (or C) tile
    static constexpr int BCPT = (BCV + kThreads - 1) / kThreads;
    static constexpr int DBS = T + 1;               // padded row (float2) of the (dtl, bu) tile
    static constexpr int PS = T + 4;                // padded row (float) of the partials tile
};

template <int N, int G, typename Tin>
struct TSSmem {
    using Cfg = TSConfig<N, G, Tin>;
    float BC[2][Cfg::T][2 * N];                     // [buf][t][B n.. | C n..]
    float2 DB[kWarps][Cfg::CPW][Cfg::DBS];          // (dt*log2 e, dt*u)
    float P[kWarps][Cfg::CPW * G][Cfg::PS];         // partial C.h per (channel, lane-in-group)
};

template <typename Tin>
__device__ __forceinline__ void unpack(const uint4& r, float* out) {
    if constexpr (sizeof(Tin) == 2) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            out[2 * i] = __uint_as_float(w[i] << 16);
            out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    } else {
        out[0] = __uint_as_float(r.x); out[1] = __uint_as_float(r.y);
        out[2] = __uint_as_float(r.z); out[3] = __uint_as_float(r.w);
    }
}

// 16 bytes at row[t .. t+V) with zero fill past L (vector load when the whole vector
// is in range and the path is aligned, element loads otherwise).
template <typename Tin, bool kVec>
__device__ __forceinline__ uint4 load_raw(const Tin* row, int64_t t, int64_t L, bool ok) {
    constexpr int V = 16 / sizeof(Tin);
    uint4 r = make_uint4(0, 0, 0, 0);
    if (!ok) return r;
    if (kVec && t + V <= L) return __ldg(reinterpret_cast<const uint4*>(row + t));
    Tin tmp[V];
#pragma unroll
    for (int k = 0; k < V; k++) tmp[k] = (t + k < L) ? row[t + k] : Tin(0.f);
    memcpy(&r, tmp, 16);
    return r;
}

// Store V consecutive steps of y (the aligned vector path).
template <typename Tout, int V>
__device__ __forceinline__ void store_steps(Tout* p, const float* v) {
    if constexpr (sizeof(Tout) == 2 && V == 8) {
        Vec16<Tout>::store(p, v);
    } else if constexpr (sizeof(Tout) == 2 && V == 4) {
        __nv_bfloat162 h0 = __floats2bfloat162_rn(v[0], v[1]), h1 = __floats2bfloat162_rn(v[2], v[3]);
        *reinterpret_cast<uint2*>(p) =
            make_uint2(*reinterpret_cast<uint32_t*>(&h0), *reinterpret_cast<uint32_t*>(&h1));
    } else {
#pragma unroll
        for (int k = 0; k < V; k += 4) Vec16<Tout>::store(p + k, v + k);
    }
}

template <int N, int G, typename Tin, typename Tout, bool kVec>
__global__ void __launch_bounds__(kThreads) thread_scan_kernel(ScanArgs a) {
    using Cfg = TSConfig<N, G, Tin>;
    constexpr int NPL = Cfg::NPL, CPW = Cfg::CPW, T = Cfg::T, V = Cfg::V, PV = Cfg::PV;
    constexpr bool kAcc = sizeof(Tin) == 4;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    TSSmem<N, G, Tin>& sm = *reinterpret_cast<TSSmem<N, G, Tin>*>(smem_raw);

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t b = blockIdx.y;
    const int64_t L = a.seqlen;
    const int64_t d_warp0 = ((int64_t)blockIdx.x * kWarps + warp) * CPW;   // first channel of this warp
    const Tin* u_base = static_cast<const Tin*>(a.u);
    const Tin* dl_base = static_cast<const Tin*>(a.delta);
    const Tin* z_base = static_cast<const Tin*>(a.z);
    const Tin* B_b = static_cast<const Tin*>(a.B) + b * N * L;
    const Tin* C_b = static_cast<const Tin*>(a.C) + b * N * L;
    Tout* y_base = static_cast<Tout*>(a.y);
    const bool has_z = a.z != nullptr;

    // phase A/C ownership: vector q of this lane covers channel ac[q], steps at[q] .. at[q]+V
    int ac[PV], at[PV];
#pragma unroll
    for (int q = 0; q < PV; q++) {
        const int v = q * 32 + lane;
        ac[q] = v / (T / V);
        at[q] = (v % (T / V)) * V;
    }
    float bias[PV], Dd[PV];
    bool chan_ok[PV];
#pragma unroll
    for (int q = 0; q < PV; q++) {
        const int64_t d = d_warp0 + ac[q];
        chan_ok[q] = d < a.dim;
        bias[q] = (chan_ok[q] && a.delta_bias) ? a.delta_bias[d] : 0.f;
        Dd[q] = (chan_ok[q] && a.D) ? a.D[d] : 0.f;
    }
    // phase B ownership
    const int g = lane / G, j = lane % G;
    const int64_t dB = d_warp0 + g;
    const bool okB = dB < a.dim;
    float Al[NPL], h[NPL];
#pragma unroll
    for (int i = 0; i < NPL; i++) {
        Al[i] = okB ? a.A[dB * N + j * NPL + i] : 0.f;
        h[i] = (okB && a.h0) ? a.h0[(b * a.dim + dB) * N + j * NPL + i] : 0.f;
    }

    // register prefetch of one chunk's raw inputs
    uint4 ru[PV], rd[PV], rz[PV], rbc[2][Cfg::BCPT];
    auto prefetch = [&](int64_t t0) {
#pragma unroll
        for (int q = 0; q < PV; q++) {
            const int64_t row = (b * a.dim + d_warp0 + ac[q]) * L;
            ru[q] = load_raw<Tin, kVec>(u_base + row, t0 + at[q], L, chan_ok[q]);
            rd[q] = load_raw<Tin, kVec>(dl_base + row, t0 + at[q], L, chan_ok[q]);
            rz[q] = load_raw<Tin, kVec>(has_z ? z_base + row : u_base, t0 + at[q], L, chan_ok[q] && has_z);
        }
#pragma unroll
        for (int r = 0; r < Cfg::BCPT; r++) {
            const int v = r * kThreads + threadIdx.x;
            const int n = v % N, tt = (v / N) * V;
            const bool ok = v < Cfg::BCV;
            rbc[0][r] = load_raw<Tin, kVec>(B_b + (int64_t)n * L, t0 + tt, L, ok);
            rbc[1][r] = load_raw<Tin, kVec>(C_b + (int64_t)n * L, t0 + tt, L, ok);
        }
    };

    const int64_t n_chunks = (L + T - 1) / T;
    if (n_chunks > 0) prefetch(0);
    for (int64_t c = 0; c < n_chunks; c++) {
        const int64_t t0 = c * T;
        const int buf = (int)(c & 1);
        // stage B/C (fp32, [t][n]) for this chunk
#pragma unroll
        for (int r = 0; r < Cfg::BCPT; r++) {
            const int v = r * kThreads + threadIdx.x;
            if (v < Cfg::BCV) {
                const int n = v % N, tt = (v / N) * V;
                float fb[V], fc[V];
                unpack<Tin>(rbc[0][r], fb);
                unpack<Tin>(rbc[1][r], fc);
#pragma unroll
                for (int k = 0; k < V; k++) {
                    sm.BC[buf][tt + k][n] = fb[k];
                    sm.BC[buf][tt + k][N + n] = fc[k];
                }
            }
        }
        // phase A: per (channel, step) prologue
        float du[PV][V];
        uint4 zc[PV];
#pragma unroll
        for (int q = 0; q < PV; q++) {
            float fu[V], fd[V];
            unpack<Tin>(ru[q], fu);
            unpack<Tin>(rd[q], fd);
            zc[q] = rz[q];
#pragma unroll
            for (int k = 0; k < V; k++) {
                const float x = fd[k] + bias[q];
                float dt = a.softplus ? softplus(x) : x;
                if (t0 + at[q] + k >= L || !chan_ok[q]) dt = 0.f;
                sm.DB[warp][ac[q]][at[q] + k] = make_float2(dt * kLog2e, dt * fu[k]);
                du[q][k] = Dd[q] * fu[k];
            }
        }
        // next chunk's loads fly while this one computes
        if (c + 1 < n_chunks) prefetch(t0 + T);
        __syncthreads();

        // phase B: the recurrence, step by step
        const float2* db = sm.DB[warp][g];
        float* prow = sm.P[warp][lane];
#pragma unroll 1
        for (int t = 0; t < T; t += 4) {
            float pv[4];
#pragma unroll
            for (int s = 0; s < 4; s++) {
                const float2 x = db[t + s];
                const float* bc = sm.BC[buf][t + s];
                float bq[NPL], cq[NPL];
                if constexpr (NPL >= 4) {
#pragma unroll
                    for (int i = 0; i < NPL; i += 4) {
                        const float4 vb = *reinterpret_cast<const float4*>(bc + j * NPL + i);
                        const float4 vc = *reinterpret_cast<const float4*>(bc + N + j * NPL + i);
                        bq[i] = vb.x; bq[i + 1] = vb.y; bq[i + 2] = vb.z; bq[i + 3] = vb.w;
                        cq[i] = vc.x; cq[i + 1] = vc.y; cq[i + 2] = vc.z; cq[i + 3] = vc.w;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < NPL; i++) { bq[i] = bc[j * NPL + i]; cq[i] = bc[N + j * NPL + i]; }
                }
                float acc = 0.f;
                if constexpr (NPL % 2 == 0) {
                    float2 acc2 = make_float2(0.f, 0.f);
                    const float2 dtl2 = make_float2(x.x, x.x), bu2 = make_float2(x.y, x.y);
#pragma unroll
                    for (int i = 0; i < NPL; i += 2) {
                        const float2 e = mul2(dtl2, make_float2(Al[i], Al[i + 1]));
                        const float2 an = make_float2(exp2_dec<kAcc>(e.x), exp2_dec<kAcc>(e.y));
                        const float2 bn = mul2(bu2, make_float2(bq[i], bq[i + 1]));
                        const float2 hh = fma2(an, make_float2(h[i], h[i + 1]), bn);
                        h[i] = hh.x; h[i + 1] = hh.y;
                        acc2 = fma2(make_float2(cq[i], cq[i + 1]), hh, acc2);
                    }
                    acc = acc2.x + acc2.y;
                } else {
#pragma unroll
                    for (int i = 0; i < NPL; i++) {
                        h[i] = fmaf(exp2_dec<kAcc>(x.x * Al[i]), h[i], x.y * bq[i]);
                        acc = fmaf(cq[i], h[i], acc);
                    }
                }
                pv[s] = acc;
            }
            *reinterpret_cast<float4*>(prow + t) = make_float4(pv[0], pv[1], pv[2], pv[3]);
        }
        __syncwarp();

        // phase C: reduce the G partials, D skip, gate, store
#pragma unroll
        for (int q = 0; q < PV; q++) {
            float yv[V];
#pragma unroll
            for (int k = 0; k < V; k++) yv[k] = du[q][k];
#pragma unroll
            for (int jj = 0; jj < G; jj++) {
                const float* pr = sm.P[warp][ac[q] * G + jj] + at[q];
#pragma unroll
                for (int k = 0; k < V; k += 4) {
                    const float4 p4 = *reinterpret_cast<const float4*>(pr + k);
                    yv[k] += p4.x; yv[k + 1] += p4.y; yv[k + 2] += p4.z; yv[k + 3] += p4.w;
                }
            }
            if (has_z) {
                float fz[V];
                unpack<Tin>(zc[q], fz);
#pragma unroll
                for (int k = 0; k < V; k++) yv[k] *= silu(fz[k]);
            }
            if (chan_ok[q]) {
                Tout* yrow = y_base + (b * a.dim + d_warp0 + ac[q]) * L;
                const int64_t tt = t0 + at[q];
                if (kVec && tt + V <= L) {
                    store_steps<Tout, V>(yrow + tt, yv);
                } else {
#pragma unroll
                    for (int k = 0; k < V; k++)
                        if (tt + k < L) yrow[tt + k] = from_f32<Tout>(yv[k]);
                }
            }
        }
        __syncwarp();
    }
    if (okB && a.h_last) {
#pragma unroll
        for (int i = 0; i < NPL; i++) a.h_last[(b * a.dim + dB) * N + j * NPL + i] = h[i];
    }
}

template <int N, int G, typename Tin, typename Tout>
cudaError_t launch_ts(const ScanArgs& a, cudaStream_t s) {
    using Cfg = TSConfig<N, G, Tin>;
    if (a.batch == 0 || a.dim == 0) return cudaSuccess;
    const int64_t ch_per_cta = (int64_t)kWarps * Cfg::CPW;
    dim3 grid((unsigned)((a.dim + ch_per_cta - 1) / ch_per_cta), (unsigned)a.batch);
    const size_t smem = sizeof(TSSmem<N, G, Tin>);
    cudaError_t e;
    if (a.vec) {
        auto k = thread_scan_kernel<N, G, Tin, Tout, true>;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        k<<<grid, kThreads, smem, s>>>(a);
    } else {
        auto k = thread_scan_kernel<N, G, Tin, Tout, false>;
        if ((e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        k<<<grid, kThreads, smem, s>>>(a);
    }
    return cudaGetLastError();
}

template <int N, typename Tin, typename Tout>
cudaError_t launch_g(const ScanArgs& a, int G, cudaStream_t s) {
    if constexpr (N >= 4) {
        if (G == 4) return launch_ts<N, 4, Tin, Tout>(a, s);
    }
    if constexpr (N >= 2) {
        if (G == 2) return launch_ts<N, 2, Tin, Tout>(a, s);
    }
    return launch_ts<N, 1, Tin, Tout>(a, s);
}

template <typename Tin, typename Tout>
cudaError_t launch_n(const ScanArgs& a, int G, cudaStream_t s) {
    switch (a.dstate) {
        case 1: return launch_g<1, Tin, Tout>(a, G, s);
        case 2: return launch_g<2, Tin, Tout>(a, G, s);
        case 4: return launch_g<4, Tin, Tout>(a, G, s);
        case 8: return launch_g<8, Tin, Tout>(a, G, s);
        case 16: return launch_g<16, Tin, Tout>(a, G, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_scan_thread(const ScanArgs& a, int lanes_per_channel, cudaStream_t s) {
    if (a.in_dtype == kBF16)
        return a.out_dtype == kBF16 ? launch_n<__nv_bfloat16, __nv_bfloat16>(a, lanes_per_channel, s)
                                    : launch_n<__nv_bfloat16, float>(a, lanes_per_channel, s);
    return a.out_dtype == kBF16 ? launch_n<float, __nv_bfloat16>(a, lanes_per_channel, s)
                                : launch_n<float, float>(a, lanes_per_channel, s);
}

}  // namespace ssm
