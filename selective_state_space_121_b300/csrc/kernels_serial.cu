// kernels_serial.cu -- time-serial selective scan for many channels: each channel's
// N-wide state is split over G lanes (G = 1, 2 or 4) and every lane walks time
// step by step.
//
// Operation (Mamba SSM complete guide (youngju.dev), section 5: selective_scan,
// with MambaBlock.ssm's softplus(dt_proj) and MambaBlock.forward's silu(z) gate):
//     h_t = exp(dt_t A) h_{t-1} + dt_t B_t u_t,  y_t = C_t . h_t + D u_t,  y_t *= silu(z_t)
//
// Why time-serial: on B300 the N = 16 bf16 scan is bound by the SFU (ex2, 32 per
// clock per SM) and by instruction issue (4 warp-instructions per clock per SM),
// not by HBM: every (t, n) element needs one exp and four FP32 operations, two
// bytes of HBM traffic per element feed it. With batch * dim in the tens of
// thousands there is enough independent work without splitting time, and walking
// time serially is the formulation with the fewest instructions per element:
//     e = dt*A (packed mul), a = ex2(e), bB = (dt*u)*B (packed mul),
//     h = a*h + bB (packed fma), acc += C*h (packed fma)
// -- 2 packed FP32 instructions, 1 SFU instruction and 1/2 shared-memory load per
// element, no shuffle scan, no second pass.
//
// Work layout. A CTA holds W = 4 warps; warp w owns CPW = 32/G consecutive
// channels of batch row b; lane (g, j) owns channel g's states
// [j*NPL, (j+1)*NPL), NPL = N/G. Time goes in chunks of T = 32 steps:
//   A. prologue, one lane per (channel, 16 bytes of consecutive steps): the
//      per-step scalars of the chunk (loaded one chunk ahead into registers) give
//      dt = softplus(delta + bias) and dt*u, written to shared memory DB[ch][t];
//   B. recurrence, lane (g, j): per step reads DB[g][t] (a broadcast within the
//      channel's lanes) and the B and C values of its states from the chunk's
//      B/C tile (fp32, [t][n], one tile per CTA: all warps share the batch row),
//      updates its states and writes its partial C.h to P[t][lane];
//   C. epilogue, same ownership as A: y = sum of the G partials + D*u, times
//      silu(z), stored with 16-byte stores.
// The B/C tile is double-buffered and filled from registers loaded one chunk
// ahead, so the only CTA-wide barrier is one per chunk.
//
// Precision. bf16 inputs (tolerance 2e-3): decay factors on the SFU (Decay<false>),
// dt via softplus(x) = ln2 * log2(1 + 2^(x*log2 e)) with SFU ex2/lg2 -- the kernel
// keeps dtl = dt*log2(e) (the ex2 argument scale) and folds ln2 into the staged B
// tile. fp32 inputs (tolerance 1e-5): accurate softplus (expf, log1pf), decays as
// expm1 (Decay<true>), and the state anchored at each chunk start: h = (hhi + hlo)
// + dlt, where the anchor is an unevaluated fp32 pair and dlt the change since the
// chunk start, so a slowly decaying large state is rounded once per output, not
// once per step.
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
struct SerialCfg {
    // time steps per chunk; with one lane per channel (G = 1) a warp owns 32
    // channels and a short chunk keeps the prologue's register footprint small
    static constexpr int kT = G == 1 ? 8 : 32;
    static constexpr int NPL = N / G;                 // states per lane
    static constexpr int CPW = 32 / G;                // channels per warp
    static constexpr int V = 16 / (int)sizeof(Tin);   // steps per 16-byte vector
    static constexpr int VPR = kT / V;                // vectors per (channel, chunk) row
    static constexpr int PV = CPW * VPR / 32;         // prologue vectors per lane per tensor
    static constexpr int BCV = 2 * N * VPR;           // vectors per B+C tile
    static constexpr int BCPT = (BCV + kThreads - 1) / kThreads;
    static constexpr int DBS = kT + 2;                // row (float2) of the DB tile: 16-byte rows
    static constexpr int PS = 32 + 1;                 // row (float4) of the partials tile
    static_assert(PV >= 1 && CPW * VPR % 32 == 0, "chunk must cover the warp's channels");
    static_assert(kT % V == 0, "chunk must be whole vectors");
};

// element i % 2 of a pair
__device__ __forceinline__ float lo_hi(const float2& v, int i) { return (i & 1) ? v.y : v.x; }
__device__ __forceinline__ float& lo_hi_ref(float2& v, int i) { return (i & 1) ? v.y : v.x; }

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

// 16 bytes at row[t .. t+V) with zero fill past L (one vector load when the whole
// vector is in range and rows are 16-byte aligned, element loads otherwise).
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
__global__ void __launch_bounds__(kThreads) serial_scan_kernel(ScanArgs a) {
    using Cfg = SerialCfg<N, G, Tin>;
    constexpr int NPL = Cfg::NPL, CPW = Cfg::CPW, V = Cfg::V, VPR = Cfg::VPR, PV = Cfg::PV, kT = Cfg::kT;
    constexpr bool kAcc = sizeof(Tin) == 4;
    using Dec = Decay<kAcc>;
    // separate arrays (not one struct) so the compiler sees that the partial-sum
    // stores cannot alias the operand loads of later steps
    __shared__ __align__(16) float s_bc[2][kT][2 * N];              // [buf][t][B n.. | C n..]
    __shared__ __align__(16) float2 s_db[kWarps][CPW][Cfg::DBS];    // (dt*scale, dt*scale*u)
    __shared__ __align__(16) float4 s_p[kWarps][kT / 4][Cfg::PS];   // partial C.h of 4 steps per lane

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t b = blockIdx.y;
    const int64_t L = a.seqlen;
    const int64_t d_warp0 = ((int64_t)blockIdx.x * kWarps + warp) * CPW;
    const Tin* u_base = static_cast<const Tin*>(a.u);
    const Tin* dl_base = static_cast<const Tin*>(a.delta);
    const Tin* z_base = static_cast<const Tin*>(a.z);
    const Tin* B_b = static_cast<const Tin*>(a.B) + b * N * L;
    const Tin* C_b = static_cast<const Tin*>(a.C) + b * N * L;
    Tout* y_base = static_cast<Tout*>(a.y);
    const bool has_z = a.z != nullptr;

    // prologue/epilogue ownership: vector q of this lane covers channel pc[q],
    // steps pt[q] .. pt[q]+V of the chunk
    int pc[PV], pt[PV];
    float bias[PV], Dd[PV];
    bool chan_ok[PV];
#pragma unroll
    for (int q = 0; q < PV; q++) {
        const int v = q * 32 + lane;
        pc[q] = v / VPR;
        pt[q] = (v % VPR) * V;
        const int64_t d = d_warp0 + pc[q];
        chan_ok[q] = d < a.dim;
        bias[q] = (chan_ok[q] && a.delta_bias) ? a.delta_bias[d] : 0.f;
        if constexpr (!kAcc) bias[q] *= kLog2e;
        Dd[q] = (chan_ok[q] && a.D) ? a.D[d] : 0.f;
    }
    // recurrence ownership
    const int g = lane / G, j = lane % G;
    const int64_t dR = d_warp0 + g;
    const bool okR = dR < a.dim;
    // A and the state in pairs (the packed f32x2 operands); the anchored form of
    // the fp32 path also keeps (hhi, hlo, dlt) per state
    constexpr int NP2 = (NPL + 1) / 2;
    float2 A2[NP2], h2[NP2];
    float hhi[NPL], hlo[NPL], dlt[NPL];
#pragma unroll
    for (int i = 0; i < NP2; i++) { A2[i] = make_float2(0.f, 0.f); h2[i] = make_float2(0.f, 0.f); }
#pragma unroll
    for (int i = 0; i < NPL; i++) {
        lo_hi_ref(A2[i / 2], i) = okR ? a.A[dR * N + j * NPL + i] : 0.f;
        const float h0 = (okR && a.h0) ? a.h0[(b * a.dim + dR) * N + j * NPL + i] : 0.f;
        lo_hi_ref(h2[i / 2], i) = h0;
        hhi[i] = h0;
        hlo[i] = 0.f;
        dlt[i] = 0.f;
    }

    // one chunk of raw inputs, loaded a chunk ahead
    uint4 ru[PV], rd[PV], rz[PV], rbc[Cfg::BCPT];
    auto prefetch = [&](int64_t t0) {
#pragma unroll
        for (int q = 0; q < PV; q++) {
            const int64_t row = (b * a.dim + d_warp0 + pc[q]) * L;
            ru[q] = load_raw<Tin, kVec>(u_base + row, t0 + pt[q], L, chan_ok[q]);
            rd[q] = load_raw<Tin, kVec>(dl_base + row, t0 + pt[q], L, chan_ok[q]);
            rz[q] = load_raw<Tin, kVec>(has_z ? z_base + row : u_base, t0 + pt[q], L, chan_ok[q] && has_z);
        }
#pragma unroll
        for (int r = 0; r < Cfg::BCPT; r++) {
            const int v = r * kThreads + threadIdx.x;
            const int which = v / (N * VPR), rem = v % (N * VPR);
            const int n = rem / VPR, tt = (rem % VPR) * V;
            rbc[r] = load_raw<Tin, kVec>((which ? C_b : B_b) + (int64_t)n * L, t0 + tt, L, v < Cfg::BCV);
        }
    };

    const int64_t n_chunks = (L + kT - 1) / kT;
    if (n_chunks > 0) prefetch(0);
    for (int64_t c = 0; c < n_chunks; c++) {
        const int64_t t0 = c * kT;
        const int buf = (int)(c & 1);
        // B/C tile of this chunk: fp32, [t][n]; B carries ln2 on the bf16 path
#pragma unroll
        for (int r = 0; r < Cfg::BCPT; r++) {
            const int v = r * kThreads + threadIdx.x;
            if (v < Cfg::BCV) {
                const int which = v / (N * VPR), rem = v % (N * VPR);
                const int n = rem / VPR, tt = (rem % VPR) * V;
                float f[V];
                unpack<Tin>(rbc[r], f);
                const float s = (!kAcc && which == 0) ? kLn2 : 1.f;
#pragma unroll
                for (int k = 0; k < V; k++) s_bc[buf][tt + k][which * N + n] = f[k] * s;
            }
        }
        // A. prologue
        uint4 ku[PV], kz[PV];
#pragma unroll
        for (int q = 0; q < PV; q++) {
            float fu[V], fd[V];
            unpack<Tin>(ru[q], fu);
            unpack<Tin>(rd[q], fd);
            ku[q] = ru[q];
            kz[q] = rz[q];
#pragma unroll
            for (int k = 0; k < V; k++) {
                float dts;   // dt * Dec::scale
                if constexpr (kAcc) {
                    const float x = fd[k] + bias[q];
                    dts = a.softplus ? softplus_acc<true>(x) : x;
                } else {
                    // x*log2(e); log2(1 + 2^xl) equals xl in fp32 once xl > 24
                    const float xl = fmaf(fd[k], kLog2e, bias[q]);
                    dts = a.softplus ? (xl > 24.f ? xl : lg2(1.f + ex2(xl))) : xl;
                }
                if (t0 + pt[q] + k >= L || !chan_ok[q]) dts = 0.f;   // identity step past the end
                s_db[warp][pc[q]][pt[q] + k] = make_float2(dts, dts * fu[k]);
            }
        }
        if (c + 1 < n_chunks) prefetch(t0 + kT);
        __syncthreads();

        // B. recurrence, in groups of 4 steps. Only the chained state updates of a
        // group depend on the state; its loads and exps do not. The bf16 path is
        // software-pipelined by hand: the loads and exps of group g+1 are issued
        // before the chained updates of group g, so an in-order warp has the
        // SFU/shared-memory latency of one group covered by the other's FMAs.
        const float4* db = reinterpret_cast<const float4*>(s_db[warp][g]);   // 2 steps per load
        // B and C of this lane's states at step t, in pairs
        auto load_bc = [&](int t, float2* bq, float2* cq) {
            const float* bc = s_bc[buf][t];
            if constexpr (NPL % 4 == 0) {
#pragma unroll
                for (int i = 0; i < NPL; i += 4) {
                    const float4 vb = *reinterpret_cast<const float4*>(bc + j * NPL + i);
                    const float4 vc = *reinterpret_cast<const float4*>(bc + N + j * NPL + i);
                    bq[i / 2] = make_float2(vb.x, vb.y); bq[i / 2 + 1] = make_float2(vb.z, vb.w);
                    cq[i / 2] = make_float2(vc.x, vc.y); cq[i / 2 + 1] = make_float2(vc.z, vc.w);
                }
            } else if constexpr (NPL == 2) {
                bq[0] = *reinterpret_cast<const float2*>(bc + j * 2);
                cq[0] = *reinterpret_cast<const float2*>(bc + N + j * 2);
            } else {
                bq[0] = make_float2(bc[j], 0.f);
                cq[0] = make_float2(bc[N + j], 0.f);
            }
        };
        auto load_x = [&](int tg, float2* x) {
            const float4 x01 = db[tg / 2], x23 = db[tg / 2 + 1];
            x[0] = make_float2(x01.x, x01.y); x[1] = make_float2(x01.z, x01.w);
            x[2] = make_float2(x23.x, x23.y); x[3] = make_float2(x23.z, x23.w);
        };
        if constexpr (!kAcc && NPL % 2 == 0) {
            // operands of one group, ready for its chained updates
            struct Stage {
                float2 an[4][NP2], bn[4][NP2], cq[4][NP2];
            };
            auto stage = [&](int tg, Stage& S) {
                float2 x[4];
                load_x(tg, x);
#pragma unroll
                for (int st = 0; st < 4; st++) {
                    float2 bq[NP2];
                    load_bc(tg + st, bq, S.cq[st]);
                    const float2 dtl2 = make_float2(x[st].x, x[st].x), bu2 = make_float2(x[st].y, x[st].y);
#pragma unroll
                    for (int i = 0; i < NP2; i++) {
                        const float2 e = mul2(dtl2, A2[i]);
                        S.an[st][i] = make_float2(ex2(e.x), ex2(e.y));
                        S.bn[st][i] = mul2(bu2, bq[i]);
                    }
                }
            };
            Stage cur, nxt;
            stage(0, cur);
#pragma unroll
            for (int tg = 0; tg < kT; tg += 4) {
                if (tg + 4 < kT) stage(tg + 4, nxt);
                float acc[4];
#pragma unroll
                for (int st = 0; st < 4; st++) {
                    float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int i = 0; i < NP2; i++) {
                        h2[i] = fma2(cur.an[st][i], h2[i], cur.bn[st][i]);
                        acc2 = fma2(cur.cq[st][i], h2[i], acc2);
                    }
                    acc[st] = acc2.x + acc2.y;
                }
                s_p[warp][tg / 4][lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                if (tg + 4 < kT) cur = nxt;
            }
        } else {
#pragma unroll
            for (int tg = 0; tg < kT; tg += 4) {
                float2 x[4];
                load_x(tg, x);
                float2 bq[4][NP2], cq[4][NP2];
#pragma unroll
                for (int st = 0; st < 4; st++) load_bc(tg + st, bq[st], cq[st]);
                float an[4][NPL];
#pragma unroll
                for (int st = 0; st < 4; st++)
#pragma unroll
                    for (int i = 0; i < NPL; i++) an[st][i] = Dec::make(x[st].x * lo_hi(A2[i / 2], i));
                float acc[4];
#pragma unroll
                for (int st = 0; st < 4; st++) {
                    acc[st] = 0.f;
#pragma unroll
                    for (int i = 0; i < NPL; i++) {
                        const float bv = x[st].y * lo_hi(bq[st][i / 2], i);
                        float& hi = lo_hi_ref(h2[i / 2], i);
                        if constexpr (kAcc) {
                            dlt[i] += fmaf(an[st][i], hi, bv);
                            hi = hhi[i] + (dlt[i] + hlo[i]);
                        } else {
                            hi = Dec::step(an[st][i], hi, bv);
                        }
                        acc[st] = fmaf(lo_hi(cq[st][i / 2], i), hi, acc[st]);
                    }
                }
                s_p[warp][tg / 4][lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            }
        }
        if constexpr (kAcc) {
            // re-anchor: (hhi, hlo) <- the exact sum of the pair and dlt
#pragma unroll
            for (int i = 0; i < NPL; i++) {
                two_sum(hhi[i], dlt[i] + hlo[i], hhi[i], hlo[i]);
                dlt[i] = 0.f;
            }
        }
        __syncwarp();

        // C. epilogue: y = (sum of the G partials + D*u) * silu(z)
#pragma unroll
        for (int q = 0; q < PV; q++) {
            float fu[V], yv[V];
            unpack<Tin>(ku[q], fu);
#pragma unroll
            for (int k = 0; k < V; k++) yv[k] = fu[k] * Dd[q];
#pragma unroll
            for (int jj = 0; jj < G; jj++) {
#pragma unroll
                for (int k = 0; k < V; k += 4) {
                    const float4 p4 = s_p[warp][(pt[q] + k) / 4][pc[q] * G + jj];
                    yv[k] += p4.x; yv[k + 1] += p4.y; yv[k + 2] += p4.z; yv[k + 3] += p4.w;
                }
            }
            if (has_z) {
                float fz[V];
                unpack<Tin>(kz[q], fz);
#pragma unroll
                for (int k = 0; k < V; k++) yv[k] *= silu_acc<kAcc>(fz[k]);
            }
            if (chan_ok[q]) {
                Tout* yrow = y_base + (b * a.dim + d_warp0 + pc[q]) * L;
                const int64_t tt = t0 + pt[q];
                if (kVec && tt + V <= L) {
                    store_steps<Tout, V>(yrow + tt, yv);
                } else {
#pragma unroll
                    for (int k = 0; k < V; k++)
                        if (tt + k < L) yrow[tt + k] = from_f32<Tout>(yv[k]);
                }
            }
        }
    }
    if (okR && a.h_last) {
#pragma unroll
        for (int i = 0; i < NPL; i++)
            a.h_last[(b * a.dim + dR) * N + j * NPL + i] = kAcc ? hhi[i] + hlo[i] : lo_hi(h2[i / 2], i);
    }
}

template <int N, int G, typename Tin, typename Tout>
cudaError_t launch_serial(const ScanArgs& a, cudaStream_t s) {
    using Cfg = SerialCfg<N, G, Tin>;
    if (a.batch == 0 || a.dim == 0) return cudaSuccess;
    const int64_t ch_per_cta = (int64_t)kWarps * Cfg::CPW;
    dim3 grid((unsigned)((a.dim + ch_per_cta - 1) / ch_per_cta), (unsigned)a.batch);
    if (a.vec) serial_scan_kernel<N, G, Tin, Tout, true><<<grid, kThreads, 0, s>>>(a);
    else serial_scan_kernel<N, G, Tin, Tout, false><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

// lanes per channel: 4 for N >= 4 (2 also built for N = 16), else N
template <int N, typename Tin, typename Tout>
cudaError_t launch_g(const ScanArgs& a, int G, cudaStream_t s) {
    if constexpr (N >= 4) {
        if constexpr (N == 16) {
            if (G == 2) return launch_serial<N, 2, Tin, Tout>(a, s);
        }
        return launch_serial<N, 4, Tin, Tout>(a, s);
    } else {
        return launch_serial<N, N, Tin, Tout>(a, s);
    }
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
