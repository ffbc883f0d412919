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
// consecutive; a CTA holds 4 warps of one batch row. Time goes in tiles of
// 8-32 steps; each tile's inputs are loaded into registers one tile ahead, then
// staged in shared memory: B and C for the CTA's batch row, and per (channel,
// step) {dt, u, dout silu(z), dout silu'(z)} and softplus', computed once (one
// lane per 16-byte vector of a channel) rather than by each of a channel's G
// lanes. Two phases:
//   1. forward over the whole sequence, h only, writing the state at every
//      8-step chunk start to the workspace (B, D, ceil(L/8), N) fp32;
//   2. tiles in reverse, and the tile's 8-step chunks in reverse: the chunk's
//      states are recomputed from its checkpoint into registers, then its steps
//      run backwards. Per step, the per-channel sums (y for dz, d(dt), du) are
//      xor-shuffle reductions over the channel's G lanes; dB and dC of the step
//      are reduce-scattered over the warp's P channels (each lane ends with one
//      (n, B-or-C) total), the 4 warps' totals meet in shared memory, and one
//      atomic add per (step, n, B-or-C) per CTA goes to global memory.
// fp32 arithmetic; for fp32 inputs exp and softplus take the accurate forms.
#include <string.h>

#include "common.cuh"
#include "launch.h"

namespace ssm {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kC = 8;   // steps per checkpoint chunk

template <int N, typename Tin> struct BwdCfg {
    static constexpr int NPL = N < 4 ? N : 4;   // states per lane
    static constexpr int G = N / NPL;           // lanes per channel
    static constexpr int P = 32 / G;            // channels per warp
    static constexpr int M = 2 * NPL;           // dB and dC values per lane-step
    static constexpr int V = 16 / (int)sizeof(Tin);                    // steps per 16-byte vector
    static constexpr int kTile = 32 * V / P > kC ? 32 * V / P : kC;    // steps per tile
    static constexpr int VPT = kTile / V;                              // vectors per (channel, tile)
    static constexpr int PV = P * VPT / 32;                            // prologue vectors per lane
    static constexpr int BCV = 2 * N * VPT;                            // B/C vectors per tile
    static_assert(PV >= 1 && P * VPT % 32 == 0 && kTile % kC == 0, "tile shape");
    static_assert(BCV <= kThreads, "one B/C vector per thread");
};

// 16 bytes at row[t .. t+V) with zero fill past L (one vector load when whole)
template <typename T, bool kVec>
__device__ __forceinline__ uint4 load_raw(const T* row, int64_t t, int64_t L, bool ok) {
    constexpr int V = 16 / sizeof(T);
    uint4 r = make_uint4(0, 0, 0, 0);
    if (!ok) return r;
    if (kVec && t + V <= L) return __ldg(reinterpret_cast<const uint4*>(row + t));
    T tmp[V];
#pragma unroll
    for (int k = 0; k < V; k++) tmp[k] = (t + k < L) ? row[t + k] : T(0.f);
    memcpy(&r, tmp, 16);
    return r;
}

template <typename T>
__device__ __forceinline__ void unpack(const uint4& r, float* out) {
    if constexpr (sizeof(T) == 2) {
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

// V consecutive values of a T row held raw (32-bit words): V * sizeof(T) bytes,
// loaded with 16- or 8-byte vectors when whole and aligned. (dout may be wider or
// narrower than the inputs whose 16-byte vectors set V.)
template <typename T, int V>
struct RawRun {
    static constexpr int W = V * (int)sizeof(T) / 4;
    uint32_t w[W];
    template <bool kVec>
    __device__ __forceinline__ void load(const T* row, int64_t t, int64_t L, bool ok) {
#pragma unroll
        for (int i = 0; i < W; i++) w[i] = 0;
        if (!ok) return;
        if (kVec && t + V <= L) {
            if constexpr (W % 4 == 0) {
#pragma unroll
                for (int i = 0; i < W; i += 4) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + t) + i / 4);
                    w[i] = v.x; w[i + 1] = v.y; w[i + 2] = v.z; w[i + 3] = v.w;
                }
            } else {
                static_assert(W == 2, "8-byte runs");
                const uint2 v = __ldg(reinterpret_cast<const uint2*>(row + t));
                w[0] = v.x; w[1] = v.y;
            }
            return;
        }
        T tmp[V];
#pragma unroll
        for (int k = 0; k < V; k++) tmp[k] = (t + k < L) ? row[t + k] : T(0.f);
        memcpy(w, tmp, sizeof(tmp));
    }
    __device__ __forceinline__ void unpack(float* out) const {
        if constexpr (sizeof(T) == 2) {
#pragma unroll
            for (int i = 0; i < W; i++) {
                out[2 * i] = __uint_as_float(w[i] << 16);
                out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
            }
        } else {
#pragma unroll
            for (int i = 0; i < W; i++) out[i] = __uint_as_float(w[i]);
        }
    }
};

// V values at row[t ..] (a 16-byte vector of T), those before L only
template <typename T, int V, bool kVec>
__device__ __forceinline__ void store_vec(T* row, int64_t t, int64_t L, const float* v) {
    static_assert(V == Vec16<T>::kN, "one 16-byte vector");
    if (kVec && t + V <= L) {
        Vec16<T>::store(row + t, v);
        return;
    }
#pragma unroll
    for (int k = 0; k < V; k++)
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
template <int P>
__device__ __forceinline__ float chan_sum(float v) {
#pragma unroll
    for (int m = P; m < 32; m <<= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

template <int N, typename Tin, typename Tdo, bool kVec>
// three CTAs per SM: the Mamba-130M-shaped layer's 384 CTAs then run in one wave
__global__ void __launch_bounds__(kThreads, 3) scan_bwd_kernel(BwdArgs a) {
    using Cfg = BwdCfg<N, Tin>;
    constexpr int NPL = Cfg::NPL, P = Cfg::P, M = Cfg::M, V = Cfg::V, kTile = Cfg::kTile;
    constexpr int VPT = Cfg::VPT, PV = Cfg::PV, BCV = Cfg::BCV;
    constexpr bool kAcc = sizeof(Tin) == 4;
    // per tile: B and C (fp32 [t][which][n]); per (channel, step) {dt, u, dy, dz factor}
    // and softplus'; the dB/dC totals of each warp per step, summed over warps after
    __shared__ __align__(16) float s_bc[kTile][2][N];
    // rows padded by one entry: the 8 lanes of a quarter-warp read 8 channels' rows
    // at the same step, which unpadded (a power-of-two stride) share one bank group
    __shared__ __align__(16) float4 s_ch[kWarps][P][kTile + 1];
    __shared__ float s_sig[kWarps][P][kTile + 1];
    __shared__ float s_dbc[kWarps][kTile][2 * N];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int p = lane % P, j = lane / P;
    const int64_t b = blockIdx.y;
    const int64_t d_w = ((int64_t)blockIdx.x * kWarps + warp) * P;   // the warp's first channel
    const int64_t d = d_w + p;
    const bool ok = d < a.dim;
    const int64_t L = a.seqlen, ch = b * a.dim + d;
    const int64_t nchunk = (L + kC - 1) / kC;
    const int64_t ntile = (L + kTile - 1) / kTile;
    const bool has_z = a.z != nullptr;
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
    const float Dd = (ok && a.D) ? a.D[d] : 0.f;
    // exp(dt A_i): on the bf16 path the SFU's 2^x with A pre-scaled by log2(e)
    float Al[NPL];
#pragma unroll
    for (int i = 0; i < NPL; i++) Al[i] = kAcc ? A[i] : A[i] * kLog2e;
    auto exp_a = [&](float dt, int i) {
        if constexpr (kAcc) return exp_acc(dt * A[i]);
        else return ex2(dt * Al[i]);
    };

    // prologue ownership: vector q of this lane covers channel pc[q] of the warp,
    // steps pt[q] .. pt[q] + V of the tile
    int pc[PV], pt[PV];
    bool pok[PV];
    float pbias[PV];
    const Tin *pu[PV], *pdl[PV], *pz[PV];
    const Tdo* pdo[PV];
#pragma unroll
    for (int q = 0; q < PV; q++) {
        const int v = q * 32 + lane;
        pc[q] = v % P;
        pt[q] = (v / P) * V;
        const int64_t dq = d_w + pc[q];
        pok[q] = dq < a.dim;
        const int64_t cq = b * a.dim + (pok[q] ? dq : 0);
        pbias[q] = (pok[q] && a.delta_bias) ? a.delta_bias[dq] : 0.f;
        pu[q] = static_cast<const Tin*>(a.u) + cq * L;
        pdl[q] = static_cast<const Tin*>(a.delta) + cq * L;
        pz[q] = has_z ? static_cast<const Tin*>(a.z) + cq * L : nullptr;
        pdo[q] = static_cast<const Tdo*>(a.dout) + cq * L;
    }
    // the B/C vector this thread stages
    const int bv = threadIdx.x;
    const int bwhich = bv / (N * VPT), bn = (bv / VPT) % N, btt = (bv % VPT) * V;

    uint4 ru[PV], rd[PV], rz[PV], rbc;
    RawRun<Tdo, V> rdo[PV];
    auto prefetch = [&](int64_t t0, bool bwd) {
#pragma unroll
        for (int q = 0; q < PV; q++) {
            ru[q] = load_raw<Tin, kVec>(pu[q], t0 + pt[q], L, pok[q]);
            rd[q] = load_raw<Tin, kVec>(pdl[q], t0 + pt[q], L, pok[q]);
            if (bwd) {
                rdo[q].template load<kVec>(pdo[q], t0 + pt[q], L, pok[q]);
                rz[q] = load_raw<Tin, kVec>(has_z ? pz[q] : pu[q], t0 + pt[q], L, pok[q] && has_z);
            }
        }
        rbc = load_raw<Tin, kVec>((bwhich ? C_b : B_b) + (int64_t)bn * L, t0 + btt, L,
                                  bv < BCV && (bwd || bwhich == 0));
    };
    // the tile's shared data from the prefetched registers
    auto stage = [&](int64_t t0, bool bwd) {
        if (bv < BCV && (bwd || bwhich == 0)) {
            float f[V];
            unpack<Tin>(rbc, f);
#pragma unroll
            for (int k = 0; k < V; k++) s_bc[btt + k][bwhich][bn] = f[k];
        }
#pragma unroll
        for (int q = 0; q < PV; q++) {
            float fu[V], fd[V], fz[V], fo[V];
            unpack<Tin>(ru[q], fu);
            unpack<Tin>(rd[q], fd);
            if (bwd) {
                rdo[q].unpack(fo);
                unpack<Tin>(rz[q], fz);
            }
#pragma unroll
            for (int k = 0; k < V; k++) {
                const bool live = pok[q] && t0 + pt[q] + k < L;
                const float x = fd[k] + pbias[q];
                float dt = a.softplus ? softplus_acc<kAcc>(x) : x;
                float4 e = make_float4(live ? dt : 0.f, fu[k], 0.f, 0.f);
                if (bwd) {
                    float dy = live ? fo[k] : 0.f, dzf = 0.f;
                    if (has_z) {
                        const float sg = sigmoid_f<kAcc>(fz[k]);
                        dzf = dy * sg * fmaf(fz[k], 1.f - sg, 1.f);   // dout silu'(z)
                        dy *= fz[k] * sg;                               // dout silu(z)
                    }
                    e.z = dy;
                    e.w = dzf;
                    s_sig[warp][pc[q]][pt[q] + k] = live ? (a.softplus ? sigmoid_f<kAcc>(x) : 1.f) : 0.f;
                }
                s_ch[warp][pc[q]][pt[q] + k] = e;
            }
        }
    };

    // 1. forward, checkpointing the state at every chunk start
    if (ntile > 0) prefetch(0, false);
    for (int64_t tile = 0; tile < ntile; tile++) {
        const int64_t t0 = tile * kTile;
        __syncthreads();   // the previous tile's readers are done
        stage(t0, false);
        if (tile + 1 < ntile) prefetch(t0 + kTile, false);
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kTile; k++) {
            if (k % kC == 0 && ok && t0 + k < L) {
                float* w = ws + ((t0 + k) / kC) * N;
                if constexpr (NPL == 4) *reinterpret_cast<float4*>(w) = make_float4(h[0], h[1], h[2], h[3]);
                else {
#pragma unroll
                    for (int i = 0; i < NPL; i++) w[i] = h[i];
                }
            }
            const float4 e = s_ch[warp][p][k];
            const float dtu = e.x * e.y;
#pragma unroll
            for (int i = 0; i < NPL; i++)
                h[i] = fmaf(exp_a(e.x, i), h[i], dtu * s_bc[k][0][j * NPL + i]);
        }
    }

    // 2. tiles in reverse; inside a tile, chunks in reverse
    float dD = 0.f, dbias = 0.f;
    if (ntile > 0) prefetch((ntile - 1) * kTile, true);
    for (int64_t tile = ntile - 1; tile >= 0; tile--) {
        const int64_t t0 = tile * kTile;
        __syncthreads();   // the previous tile's readers (and the flush) are done
        stage(t0, true);
        if (tile > 0) prefetch(t0 - kTile, true);
        __syncthreads();
#pragma unroll 1
        for (int cc = kTile / kC - 1; cc >= 0; cc--) {
            const int64_t tc = t0 + cc * kC;
            if (tc >= L) continue;   // warp-uniform (chunks past the end of the last tile)
            float hs[kC + 1][NPL];   // hs[k] = state before step k of the chunk
            if (ok) {
                const float* w = ws + (tc / kC) * N;
                if constexpr (NPL == 4) {
                    const float4 v = *reinterpret_cast<const float4*>(w);
                    hs[0][0] = v.x; hs[0][1] = v.y; hs[0][2] = v.z; hs[0][3] = v.w;
                } else {
#pragma unroll
                    for (int i = 0; i < NPL; i++) hs[0][i] = w[i];
                }
            } else {
#pragma unroll
                for (int i = 0; i < NPL; i++) hs[0][i] = 0.f;
            }
#pragma unroll
            for (int k = 0; k < kC; k++) {
                const int kk = cc * kC + k;
                const float4 e = s_ch[warp][p][kk];
                const float dtu = e.x * e.y;
#pragma unroll
                for (int i = 0; i < NPL; i++)
                    hs[k + 1][i] = fmaf(exp_a(e.x, i), hs[k][i], dtu * s_bc[kk][0][j * NPL + i]);
            }
            // steps in pairs: the dB/dC values of two steps share one reduce-scatter
            // (same shuffle count, half the dependent rounds per step)
#pragma unroll
            for (int k2 = kC - 1; k2 >= 1; k2 -= 2) {
                float vals[2 * M];   // [step k2: dB, dC | step k2-1: dB, dC]
#pragma unroll
                for (int sidx = 0; sidx < 2; sidx++) {
                    const int k = k2 - sidx;
                    const int kk = cc * kC + k;
                    const float4 e = s_ch[warp][p][kk];
                    const float dt = e.x, u = e.y, dy = e.z;
                    const float* Bk = s_bc[kk][0] + j * NPL;
                    const float* Ck = s_bc[kk][1] + j * NPL;
                    float dz = 0.f;
                    if (has_z) {
                        float part = 0.f;
#pragma unroll
                        for (int i = 0; i < NPL; i++) part = fmaf(Ck[i], hs[k + 1][i], part);
                        dz = e.w * (chan_sum<P>(part) + Dd * u);
                    }
                    dD = fmaf(dy, u, dD);
                    float ddt_p = 0.f, du_p = 0.f;
                    const float dtu = dt * u;
#pragma unroll
                    for (int i = 0; i < NPL; i++) {
                        g[i] = fmaf(Ck[i], dy, g[i]);
                        vals[sidx * M + NPL + i] = dy * hs[k + 1][i];         // dC
                        const float an = exp_a(dt, i);
                        const float ga = g[i] * hs[k][i] * an;                  // g h_{t-1} a
                        ddt_p = fmaf(ga, A[i], ddt_p);
                        ddt_p = fmaf(g[i] * Bk[i], u, ddt_p);
                        dA[i] = fmaf(ga, dt, dA[i]);
                        vals[sidx * M + i] = g[i] * dtu;                        // dB
                        du_p = fmaf(g[i] * dt, Bk[i], du_p);
                        g[i] *= an;
                    }
                    const float du = fmaf(Dd, dy, chan_sum<P>(du_p));
                    const float dx = chan_sum<P>(ddt_p) * s_sig[warp][p][kk];
                    dbias += dx;
                    // every lane of the channel has read this step's entry (the shuffles
                    // above sync the warp): lane j = 0 puts the step's outputs there
                    if (j == 0) s_ch[warp][p][kk] = make_float4(du, dx, dz, 0.f);
                }
                // reduce-scatter over the warp's P channels: each round a lane keeps one
                // half of its block of values and adds the partner's copy of that half;
                // once a lane holds a single value the remaining rounds all-reduce it
                constexpr int MV = 2 * M;
                int idx = 0, cnt = MV;
#pragma unroll
                for (int m = 1; m < P; m <<= 1) {
                    if (cnt > 1) {
                        const int half = cnt / 2;
                        const bool up = (lane & m) != 0;
#pragma unroll
                        for (int q = 0; q < MV / 2; q++) {
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
                // the lane holds values idx .. idx + cnt - 1 (one step, contiguous); with
                // cnt == 1 only the lanes p < MV hold distinct ones
                if (cnt > 1 || p < MV) {
#pragma unroll
                    for (int c = 0; c < (MV > P ? MV / P : 1); c++) {
                        const int v = idx + c;
                        const int kk = cc * kC + k2 - v / M;
                        s_dbc[warp][kk][j * M + v % M] = vals[c];
                    }
                }
            }
        }
        __syncthreads();
        // the tile's du, ddelta, dz, with the prologue's ownership (16-byte stores)
#pragma unroll
        for (int q = 0; q < PV; q++) {
            if (!pok[q]) continue;
            float o0[V], o1[V], o2[V];
#pragma unroll
            for (int k = 0; k < V; k++) {
                const float4 e = s_ch[warp][pc[q]][pt[q] + k];
                o0[k] = e.x; o1[k] = e.y; o2[k] = e.z;
            }
            const int64_t cq = b * a.dim + d_w + pc[q], tq = t0 + pt[q];
            store_vec<Tin, V, kVec>(static_cast<Tin*>(a.du) + cq * L, tq, L, o0);
            store_vec<Tin, V, kVec>(static_cast<Tin*>(a.ddelta) + cq * L, tq, L, o1);
            if (has_z) store_vec<Tin, V, kVec>(static_cast<Tin*>(a.dz) + cq * L, tq, L, o2);
        }
        // the tile's dB, dC: the warps' totals summed, one atomic per (step, B/C, n)
        for (int e = threadIdx.x; e < kTile * 2 * N; e += kThreads) {
            const int kk = e / (2 * N), slot = e % (2 * N);
            if (t0 + kk >= L) continue;
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; w++) v += s_dbc[w][kk][slot];
            const int jj = slot / M, idx = slot % M;
            const int which = idx / NPL, n = jj * NPL + idx % NPL;
            atomicAdd((which ? a.dC : a.dB) + (b * N + n) * L + t0 + kk, v);
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
    using Cfg = BwdCfg<N, Tin>;
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
    return (size_t)batch * dim * ((seqlen + kC - 1) / kC) * dstate * 4;
}

cudaError_t launch_scan_bwd(const BwdArgs& a, cudaStream_t s) {
    if (a.in_dtype == kBF16)
        return a.dout_dtype == kBF16 ? by_n<__nv_bfloat16, __nv_bfloat16>(a, s) : by_n<__nv_bfloat16, float>(a, s);
    return a.dout_dtype == kBF16 ? by_n<float, __nv_bfloat16>(a, s) : by_n<float, float>(a, s);
}

}  // namespace ssm
