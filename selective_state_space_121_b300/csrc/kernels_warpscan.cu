// kernels_warpscan.cu -- chunked selective scan with a warp-shuffle associative
// scan inside each chunk and a serial carry across chunks (lanes split time, so
// it keeps a whole warp busy per channel: the algorithm for few channels and
// short sequences).
//
// What is computed (Mamba SSM complete guide (youngju.dev), section 5,
// selective_scan, with MambaBlock.ssm's softplus(dt_proj) and forward's silu(z)
// gate fused): per (b, d, n)
//     h_t = a_t h_{t-1} + b_t,   a_t = exp(dt_t A_dn),   b_t = dt_t B_tn u_t
//     y_t = sum_n C_tn h_t + D_d u_t, then y_t *= silu(z_t).
// Each step is an affine map h -> a h + b. Maps compose associatively,
//     (a2, b2) o (a1, b1) = (a2 a1, a2 b1 + b2),
// which is what lets the time axis be split across lanes and blocks (the
// parallel scan of the guide's "Hardware-Aware Algorithm" section; the page's
// printed up-sweep is garbled, this is the composition it stands for).
//
// Layout of the work (B300, sm_103a):
//  * A CTA holds W = 8 warps; warp w owns channel d = 8*blockIdx.x + w of batch
//    row b. All 8 channels share b, so the B and C tiles of a chunk are staged
//    once per CTA in shared memory (fp32, [n][t]) and read by all 8 warps.
//  * A chunk is 256 time steps: lane l owns steps 8l .. 8l+7 of the chunk and
//    loads its u, delta, z with one 16-byte vector load each (bf16) -- a warp
//    reads 512 contiguous bytes per tensor, fully coalesced.
//  * For each state n: the lane computes its 8 (a, b) pairs in registers, folds
//    them into one lane map (the product of the a's is exp(A * sum dt), one ex2),
//    the warp composes the 32 lane maps with a 5-step shuffle scan, the lane
//    takes its exclusive prefix, applies the carry from earlier chunks, and
//    re-runs its 8 steps to produce h_t and accumulate C_tn h_t into y_t.
//    Every a_t = exp(dt A) is evaluated exactly once.
//  * The N-wide carry (state at the chunk boundary) lives in registers; across
//    chunks it is carried serially by the warp.
//
// Directional form (launch_scan_dir, kDir): the same scan along another
// traversal of the sequence -- the four scans of an image of rows x cols patches
// stored in raster order (Mamba SSM complete guide, section 9, VMamba): raster,
// reversed, column-major, reversed columns. Traversal step k reads every input
// at position pos(k) and writes y there, so each direction's output is already
// in raster order; the lanes still own consecutive traversal steps, with the
// loads gathered by position. Optionally the input matrix is the exact
// zero-order hold of section 2 ("Discretization"), (exp(dt A) - 1) / A * B
// (dt * B where A = 0), from the decay already computed for the step.
#include "common.cuh"
#include "launch.h"

namespace ssm {
namespace {

constexpr int K = kWarpScanItems;     // 8 steps per lane
constexpr int T = kWarpScanChunk;     // 256 steps per chunk
constexpr int W = 8;                  // warps (channels) per CTA
constexpr int kThreads = 32 * W;

// Sequence position of traversal step k (see the directional form above);
// seqlen < 2^31 for the directional form, so 32-bit arithmetic.
__device__ __forceinline__ int64_t pos_of(const ScanArgs& a, int64_t k) {
    uint32_t kk = (uint32_t)k;
    if (a.order == 1 || a.order == 3) kk = (uint32_t)a.seqlen - 1u - kk;
    if (a.order >= 2) {
        const uint32_t rows = (uint32_t)a.rows, q = kk / rows;
        return (int64_t)(kk - q * rows) * a.cols + q;
    }
    return kk;
}
// Positions of K consecutive traversal steps k0 .. k0+K-1 (-1 past the end): one
// division, then the column walk steps row by row.
__device__ __forceinline__ void positions(const ScanArgs& a, int64_t k0, int64_t* pos) {
    const uint32_t L = (uint32_t)a.seqlen;
    if (a.order < 2) {
#pragma unroll
        for (int k = 0; k < K; k++) {
            const uint32_t kk = (uint32_t)k0 + k;
            pos[k] = kk < L ? (a.order == 1 ? (int64_t)(L - 1u - kk) : (int64_t)kk) : -1;
        }
        return;
    }
    const uint32_t rows = (uint32_t)a.rows;
    const bool rev = a.order == 3;
    uint32_t kk = (uint32_t)k0 < L ? (uint32_t)k0 : 0u;
    if (rev) kk = L - 1u - kk;
    uint32_t q = kk / rows, r = kk - q * rows;   // column q, row r
#pragma unroll
    for (int k = 0; k < K; k++) {
        pos[k] = (uint32_t)k0 + k < L ? (int64_t)r * a.cols + q : -1;
        if (!rev) {
            if (++r == rows) { r = 0; ++q; }
        } else {
            if (r == 0) { r = rows - 1u; --q; } else { --r; }
        }
    }
}

template <int N>
struct Smem {
    float B[N][T];
    float C[N][T];
};

// Stage B (and C) of batch row b, steps t0 .. t0+T-1, into shared memory as fp32.
template <int N, typename Tin, bool kVec, bool kWithC, bool kDir = false>
__device__ __forceinline__ void stage_bc(const ScanArgs& a, int64_t b, int64_t t0, Smem<N>& sm) {
    const Tin* Bp = static_cast<const Tin*>(a.B) + b * N * a.seqlen;
    const Tin* Cp = static_cast<const Tin*>(a.C) + b * N * a.seqlen;
    const int64_t L = a.seqlen;
    if (kDir && a.vec && a.order == 1) {
        // reversed raster: steps t0+i0 .. t0+i0+V-1 are the V positions ending at
        // L-1-(t0+i0), one aligned 16-byte block (L is a multiple of V when rows
        // are 16-byte aligned), stored reversed
        constexpr int V = Vec16<Tin>::kN;
        for (int idx = threadIdx.x; idx < N * T / V; idx += kThreads) {
            const int n = idx / (T / V);
            const int i0 = (idx % (T / V)) * V;
            const int64_t kk = t0 + i0;
            float vb[V], vc[V];
            if (kk + V <= L) {
                Vec16<Tin>::load(Bp + n * L + (L - V - kk), vb);
                if constexpr (kWithC) Vec16<Tin>::load(Cp + n * L + (L - V - kk), vc);
            } else {
#pragma unroll
                for (int j = 0; j < V; j++) {   // reversed below, so index by V-1-j
                    vb[V - 1 - j] = kk + j < L ? to_f32(Bp[n * L + (L - 1 - kk - j)]) : 0.f;
                    if constexpr (kWithC) vc[V - 1 - j] = kk + j < L ? to_f32(Cp[n * L + (L - 1 - kk - j)]) : 0.f;
                }
            }
#pragma unroll
            for (int j = 0; j < V; j++) {
                sm.B[n][i0 + j] = vb[V - 1 - j];
                if constexpr (kWithC) sm.C[n][i0 + j] = vc[V - 1 - j];
            }
        }
    } else if (kDir && !(a.vec && a.order == 0)) {
        // traversal steps t0 .. t0+T-1, gathered from their positions
        for (int i = threadIdx.x; i < T; i += kThreads) {
            const bool in = t0 + i < L;
            const int64_t t = in ? pos_of(a, t0 + i) : 0;
#pragma unroll
            for (int n = 0; n < N; n++) {
                sm.B[n][i] = in ? to_f32(Bp[n * L + t]) : 0.f;
                if constexpr (kWithC) sm.C[n][i] = in ? to_f32(Cp[n * L + t]) : 0.f;
            }
        }
    } else if (kVec || (kDir && a.vec)) {
        constexpr int V = Vec16<Tin>::kN;
        constexpr int kVecs = N * T / V;
        for (int idx = threadIdx.x; idx < kVecs; idx += kThreads) {
            const int n = idx / (T / V);
            const int i = (idx % (T / V)) * V;
            const int64_t t = t0 + i;
            float vb[V], vc[V];
            if (t + V <= L) {
                Vec16<Tin>::load(Bp + n * L + t, vb);
                if constexpr (kWithC) Vec16<Tin>::load(Cp + n * L + t, vc);
            } else {
#pragma unroll
                for (int k = 0; k < V; k++) {
                    vb[k] = (t + k < L) ? to_f32(Bp[n * L + t + k]) : 0.f;
                    if constexpr (kWithC) vc[k] = (t + k < L) ? to_f32(Cp[n * L + t + k]) : 0.f;
                }
            }
#pragma unroll
            for (int k = 0; k < V; k += 4) {
                *reinterpret_cast<float4*>(&sm.B[n][i + k]) = make_float4(vb[k], vb[k + 1], vb[k + 2], vb[k + 3]);
                if constexpr (kWithC)
                    *reinterpret_cast<float4*>(&sm.C[n][i + k]) = make_float4(vc[k], vc[k + 1], vc[k + 2], vc[k + 3]);
            }
        }
    } else {
        for (int idx = threadIdx.x; idx < N * T; idx += kThreads) {
            const int n = idx / T, i = idx % T;
            const int64_t t = t0 + i;
            sm.B[n][i] = t < L ? to_f32(Bp[n * L + t]) : 0.f;
            if constexpr (kWithC) sm.C[n][i] = t < L ? to_f32(Cp[n * L + t]) : 0.f;
        }
    }
}

// Load this lane's K steps of one (b, d) row starting at step t (may run past L).
template <typename Tin, bool kVec>
__device__ __forceinline__ void load_items(const Tin* row, int64_t t, int64_t L, float* out) {
    if constexpr (kVec) {
        constexpr int V = Vec16<Tin>::kN;
#pragma unroll
        for (int k = 0; k < K; k += V) {
            if (t + k + V <= L) {
                Vec16<Tin>::load(row + t + k, out + k);
            } else {
#pragma unroll
                for (int j = 0; j < V; j++) out[k + j] = (t + k + j < L) ? to_f32(row[t + k + j]) : 0.f;
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < K; k++) out[k] = (t + k < L) ? to_f32(row[t + k]) : 0.f;
    }
}

template <typename Tout, bool kVec>
__device__ __forceinline__ void store_items(Tout* row, int64_t t, int64_t L, const float* v) {
    if constexpr (kVec) {
        constexpr int V = Vec16<Tout>::kN;
#pragma unroll
        for (int k = 0; k < K; k += V) {
            if (t + k + V <= L) {
                Vec16<Tout>::store(row + t + k, v + k);
            } else {
#pragma unroll
                for (int j = 0; j < V; j++)
                    if (t + k + j < L) row[t + k + j] = from_f32<Tout>(v[k + j]);
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < K; k++)
            if (t + k < L) row[t + k] = from_f32<Tout>(v[k]);
    }
}

// The lane's K items at sequence positions pos[k] (-1: past the end, reads 0).
template <typename Tin>
__device__ __forceinline__ void load_at(const Tin* row, const int64_t* pos, float* out) {
#pragma unroll
    for (int k = 0; k < K; k++) out[k] = pos[k] >= 0 ? to_f32(row[pos[k]]) : 0.f;
}
template <typename Tout>
__device__ __forceinline__ void store_at(Tout* row, const int64_t* pos, const float* v) {
#pragma unroll
    for (int k = 0; k < K; k++)
        if (pos[k] >= 0) row[pos[k]] = from_f32<Tout>(v[k]);
}

// Directional loads and stores of the lane's K items (steps t .. t+K-1): with
// 16-byte aligned rows the raster order reads them as consecutive positions and
// the reversed order as the block ending at L-1-t, reversed in registers; any
// other case gathers by position.
template <typename Tin>
__device__ __forceinline__ void load_dir(const ScanArgs& a, const Tin* row, int64_t t, const int64_t* pos,
                                         float* out) {
    const int64_t L = a.seqlen;
    if (a.vec && a.order == 0) {
        load_items<Tin, true>(row, t, L, out);
    } else if (a.vec && a.order == 1 && t + K <= L) {
        float tmp[K];
        load_items<Tin, true>(row, L - K - t, L, tmp);
#pragma unroll
        for (int k = 0; k < K; k++) out[k] = tmp[K - 1 - k];
    } else {
        load_at<Tin>(row, pos, out);
    }
}
template <typename Tout>
__device__ __forceinline__ void store_dir(const ScanArgs& a, Tout* row, int64_t t, const int64_t* pos,
                                          const float* v) {
    const int64_t L = a.seqlen;
    if (a.vec && a.order == 0) {
        store_items<Tout, true>(row, t, L, v);
    } else if (a.vec && a.order == 1 && t + K <= L) {
        float tmp[K];
#pragma unroll
        for (int k = 0; k < K; k++) tmp[k] = v[K - 1 - k];
        store_items<Tout, true>(row, L - K - t, L, tmp);
    } else {
        store_at<Tout>(row, pos, v);
    }
}

// Per-lane step inputs of one chunk: dtl = dt*log2(e), bu = dt*u (zero past L).
// kDir: items of the traversal (load_dir) instead of steps t .. t+K-1.
template <typename Tin, bool kVec, bool kDir = false>
__device__ __forceinline__ float prepare_items(const ScanArgs& a, int64_t row_off, int64_t d,
                                               int64_t t, float* dtl, float* bu, float* u,
                                               const int64_t* pos = nullptr) {
    const Tin* up = static_cast<const Tin*>(a.u) + row_off;
    const Tin* dp = static_cast<const Tin*>(a.delta) + row_off;
    float dl[K];
    if constexpr (kDir) {
        load_dir<Tin>(a, up, t, pos, u);
        load_dir<Tin>(a, dp, t, pos, dl);
    } else {
        load_items<Tin, kVec>(up, t, a.seqlen, u);
        load_items<Tin, kVec>(dp, t, a.seqlen, dl);
    }
    const float bias = a.delta_bias ? a.delta_bias[d] : 0.f;
    float sdtl = 0.f;
#pragma unroll
    for (int k = 0; k < K; k++) {
        const float x = dl[k] + bias;
        float dt = a.softplus ? softplus(x) : x;
        if (t + k >= a.seqlen) dt = 0.f;   // identity map past the end: a = 1, b = 0
        dtl[k] = dt * Decay<sizeof(Tin) == 4>::scale;
        bu[k] = dt * u[k];
        sdtl += dtl[k];
    }
    return sdtl;
}

// Inclusive warp scan of lane maps (P, H): lane l ends with the composition of the
// maps of lanes 0..l.
template <class Dec>
__device__ __forceinline__ void warp_scan_maps(float& P, float& H, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float Pp = __shfl_up_sync(0xffffffffu, P, off);
        const float Hp = __shfl_up_sync(0xffffffffu, H, off);
        if (lane >= off) {
            H = Dec::step(P, Hp, H);
            P = Dec::mul(P, Pp);
        }
    }
}

// Full pass over one chunk: y for the lane's steps from the N-wide carry; carry
// is advanced to the state at the end of the chunk.
// With fp32 inputs (Decay<true>) the carry is an unevaluated pair (carry, carry_lo)
// and every state inside the chunk is formed as carry + delta, where delta (the
// change since the chunk start) is accumulated on its own: a slowly decaying
// large state is then rounded once per output instead of once per step, which
// keeps the fp32 result within ~1e-6 of its scale over thousands of steps. With
// bf16 inputs carry_lo stays zero and the plain recurrence runs.
template <int N, typename Tin, typename Tout, bool kVec, bool kDir = false, bool kZoh = false>
__device__ __forceinline__ void chunk_full(const ScanArgs& a, int64_t b, int64_t d, int64_t t0,
                                           const Smem<N>& sm, const float* Ad, float* carry,
                                           float* carry_lo, int lane) {
    constexpr bool kAnchored = sizeof(Tin) == 4;
    using Dec = Decay<kAnchored>;
    const int64_t row_off = (b * a.dim + d) * a.seqlen;
    const int64_t t = t0 + lane * K;
    int64_t pos[K];
    if constexpr (kDir) positions(a, t, pos);
    float dtl[K], bu[K], u[K], y[K];
    const float sdtl = prepare_items<Tin, kVec, kDir>(a, row_off, d, t, dtl, bu, u, pos);

#pragma unroll
    for (int k = 0; k < K; k++) y[k] = 0.f;
#pragma unroll
    for (int n = 0; n < N; n++) {
        const float* sb = &sm.B[n][lane * K];
        const float* sc = &sm.C[n][lane * K];
        float an[K], bn[K];
        float H = 0.f;
        // zero-order hold: (a - 1) / A replaces dt (a - 1 is what the fp32 form carries)
        const bool hold = kZoh && Ad[n] != 0.f;
        const float inv_a = hold ? 1.f / Ad[n] : 0.f;
#pragma unroll
        for (int k = 0; k < K; k++) {
            an[k] = Dec::make(dtl[k] * Ad[n]);
            if (hold) bn[k] = (kAnchored ? an[k] : an[k] - 1.f) * inv_a * u[k] * sb[k];
            else bn[k] = bu[k] * sb[k];
            H = Dec::step(an[k], H, bn[k]);
        }
        float P = Dec::make(sdtl * Ad[n]);
        warp_scan_maps<Dec>(P, H, lane);
        float Pe = __shfl_up_sync(0xffffffffu, P, 1);
        float He = __shfl_up_sync(0xffffffffu, H, 1);
        if (lane == 0) { Pe = Dec::one(); He = 0.f; }
        const float Pt = __shfl_sync(0xffffffffu, P, 31);
        const float Ht = __shfl_sync(0xffffffffu, H, 31);
        if constexpr (kAnchored) {
            float dlt = fmaf(Pe, carry[n], He) + carry_lo[n];
            float h = carry[n] + dlt;
#pragma unroll
            for (int k = 0; k < K; k++) {
                dlt += fmaf(an[k], h, bn[k]);
                h = carry[n] + dlt;
                y[k] = fmaf(sc[k], h, y[k]);
            }
            two_sum(carry[n], fmaf(Pt, carry[n], Ht) + carry_lo[n], carry[n], carry_lo[n]);
        } else {
            float h = Dec::step(Pe, carry[n], He);
#pragma unroll
            for (int k = 0; k < K; k++) {
                h = Dec::step(an[k], h, bn[k]);
                y[k] = fmaf(sc[k], h, y[k]);
            }
            carry[n] = Dec::step(Pt, carry[n], Ht);
        }
    }
    const float Dd = a.D ? a.D[d] : 0.f;
    if (a.z) {
        float zz[K];
        if constexpr (kDir) load_dir<Tin>(a, static_cast<const Tin*>(a.z) + row_off, t, pos, zz);
        else load_items<Tin, kVec>(static_cast<const Tin*>(a.z) + row_off, t, a.seqlen, zz);
#pragma unroll
        for (int k = 0; k < K; k++) y[k] = fmaf(Dd, u[k], y[k]) * silu(zz[k]);
    } else {
#pragma unroll
        for (int k = 0; k < K; k++) y[k] = fmaf(Dd, u[k], y[k]);
    }
    if constexpr (kDir) store_dir<Tout>(a, static_cast<Tout*>(a.y) + row_off, t, pos, y);
    else store_items<Tout, kVec>(static_cast<Tout*>(a.y) + row_off, t, a.seqlen, y);
}

template <int N>
__device__ __forceinline__ void load_A(const ScanArgs& a, int64_t d, float* Ad) {
#pragma unroll
    for (int n = 0; n < N; n++) Ad[n] = a.A[d * N + n];
}

template <int N>
__device__ __forceinline__ void load_h0(const ScanArgs& a, int64_t b, int64_t d, float* carry, float* carry_lo) {
#pragma unroll
    for (int n = 0; n < N; n++) {
        carry[n] = a.h0 ? a.h0[(b * a.dim + d) * N + n] : 0.f;
        carry_lo[n] = 0.f;
    }
}

template <int N>
__device__ __forceinline__ void store_hlast(const ScanArgs& a, int64_t b, int64_t d, const float* carry,
                                            const float* carry_lo, int lane) {
    if (!a.h_last) return;
#pragma unroll
    for (int n = 0; n < N; n++)
        if (lane == (n & 31)) a.h_last[(b * a.dim + d) * N + n] = carry[n] + carry_lo[n];
}

// ---------------------------------------------------------------------------
// Serial-carry kernel: grid (ceil(dim / 8), batch); each warp walks its
// channel's whole sequence chunk by chunk.
// ---------------------------------------------------------------------------
// Two CTAs per SM (128 registers): at the few-channel shapes this algorithm serves,
// latency is hidden by warps, and the grid then fits one round more often.
template <int N, typename Tin, typename Tout, bool kVec, bool kDir = false, bool kZoh = false>
__global__ void __launch_bounds__(kThreads, 2) warp_scan_kernel(ScanArgs a) {
    __shared__ __align__(16) Smem<N> sm;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t b = blockIdx.y;
    const int64_t d = (int64_t)blockIdx.x * W + warp;
    const bool active = d < a.dim;
    float Ad[N], carry[N], carry_lo[N];
    if (active) {
        load_A<N>(a, d, Ad);
        load_h0<N>(a, b, d, carry, carry_lo);
    }
    for (int64_t t0 = 0; t0 < a.seqlen; t0 += T) {
        stage_bc<N, Tin, kVec, true, kDir>(a, b, t0, sm);
        __syncthreads();
        if (active) chunk_full<N, Tin, Tout, kVec, kDir, kZoh>(a, b, d, t0, sm, Ad, carry, carry_lo, lane);
        __syncthreads();
    }
    if (active) store_hlast<N>(a, b, d, carry, carry_lo, lane);
}

template <int N, typename Tin, typename Tout, bool kDir>
cudaError_t launch_ws_n(const ScanArgs& a, cudaStream_t s) {
    if (a.batch == 0 || a.dim == 0) return cudaSuccess;
    dim3 grid((unsigned)((a.dim + W - 1) / W), (unsigned)a.batch);
    // the raster order with dt * B is the plain scan: its vectorised form
    if (kDir && a.zoh) warp_scan_kernel<N, Tin, Tout, false, true, true><<<grid, kThreads, 0, s>>>(a);
    else if (kDir && a.order != 0) warp_scan_kernel<N, Tin, Tout, false, true, false><<<grid, kThreads, 0, s>>>(a);
    else if (a.vec) warp_scan_kernel<N, Tin, Tout, true><<<grid, kThreads, 0, s>>>(a);
    else warp_scan_kernel<N, Tin, Tout, false><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin, typename Tout, bool kDir = false>
cudaError_t dispatch_n(const ScanArgs& a, cudaStream_t s) {
    switch (a.dstate) {
        case 1: return launch_ws_n<1, Tin, Tout, kDir>(a, s);
        case 2: return launch_ws_n<2, Tin, Tout, kDir>(a, s);
        case 4: return launch_ws_n<4, Tin, Tout, kDir>(a, s);
        case 8: return launch_ws_n<8, Tin, Tout, kDir>(a, s);
        case 16: return launch_ws_n<16, Tin, Tout, kDir>(a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_scan_warp(const ScanArgs& a, cudaStream_t s) {
    if (a.in_dtype == kBF16)
        return a.out_dtype == kBF16 ? dispatch_n<__nv_bfloat16, __nv_bfloat16>(a, s)
                                    : dispatch_n<__nv_bfloat16, float>(a, s);
    return a.out_dtype == kBF16 ? dispatch_n<float, __nv_bfloat16>(a, s) : dispatch_n<float, float>(a, s);
}

cudaError_t launch_scan_dir(const ScanArgs& a, cudaStream_t s) {
    if (a.in_dtype == kBF16)
        return a.out_dtype == kBF16 ? dispatch_n<__nv_bfloat16, __nv_bfloat16, true>(a, s)
                                    : dispatch_n<__nv_bfloat16, float, true>(a, s);
    return a.out_dtype == kBF16 ? dispatch_n<float, __nv_bfloat16, true>(a, s) : dispatch_n<float, float, true>(a, s);
}

}  // namespace ssm
