// kernels_scalar.cu -- the d_state = 1 scan (SM1, "Scalar Mamba1").
//
// What is computed (SM1 (Scalar Mamba1) page, section details: with one state per
// channel the selective scan has the closed form h = L * (h0 + cumsum(dBx / L)),
// L = cumprod(dA); the kernel evaluates the same recurrence without dividing by the
// cumulative product):
//     h_t = exp(dt_t A_d) h_{t-1} + dt_t B_t u_t,   y_t = C_t h_t (+ D_d u_t) (* silu(z_t))
// with dt_t = softplus(delta_t + bias_d).
//
// The scan moves 12 bytes (fp32 u, delta, y) per token*channel against one exp,
// one softplus and a handful of FP32 ops: it is HBM-bound, and the design goal is
// enough independent work in flight. With one state per channel a lane holding a
// whole channel would leave the GPU nearly idle (batch*dim lanes), so time is
// split inside the warp:
//  * a warp holds 4 channels (consecutive rows of the flattened (batch, dim)),
//    8 lanes per channel; time goes in chunks of 64 steps, lane s of a channel
//    owns steps 8s .. 8s+7 of the chunk and loads them with 16-byte vectors (a
//    warp reads 4 x 256 contiguous bytes per tensor); the next chunk's inputs
//    are loaded while the current one computes;
//  * each lane folds its 8 steps into one affine map (a, b) (the associative
//    composition (a2, b2) o (a1, b1) = (a2 a1, a2 b1 + b2), the parallel scan idea
//    of the Mamba SSM complete guide's "Hardware-Aware Algorithm" section), a
//    3-round shuffle scan over the channel's 8 lanes gives each lane the map of
//    the steps before it, and the lane re-runs its 8 steps from the carry;
//  * the carry (the state at the chunk boundary) comes from the channel's last
//    lane. The decay factors and the state follow the same precision scheme as
//    the N-state kernels: for fp32 inputs decays are carried as expm1 and the
//    state as an anchored pair, so a slowly decaying large state is rounded once
//    per output; for bf16 inputs the plain SFU form.
#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace ssm {
namespace {

// one warp per CTA: the finest unit of residency, so that the register budget
// below, not the CTA shape, sets how many warps an SM holds
constexpr int kWarps = 1;
constexpr int kThreads = 32 * kWarps;
constexpr int kSeg = 8;             // lanes per channel
constexpr int kK = 8;               // steps per lane per chunk
constexpr int kChunk = kSeg * kK;   // 64 steps
constexpr int kChPerWarp = 32 / kSeg;

// kK consecutive values of row[t ..] widened to fp32 (zero past L or when !ok).
template <typename T, bool kVec>
__device__ __forceinline__ void load_k(const T* row, int64_t t, int64_t L, bool ok, float* out) {
    if (!ok) {
#pragma unroll
        for (int k = 0; k < kK; k++) out[k] = 0.f;
        return;
    }
    if constexpr (kVec) {
        constexpr int V = Vec16<T>::kN;
        if (t + kK <= L) {
#pragma unroll
            for (int k = 0; k < kK; k += V) Vec16<T>::load(row + t + k, out + k);
            return;
        }
    }
#pragma unroll
    for (int k = 0; k < kK; k++) out[k] = (t + k < L) ? to_f32(row[t + k]) : 0.f;
}

template <typename T, bool kVec>
__device__ __forceinline__ void store_k(T* row, int64_t t, int64_t L, const float* v) {
    if constexpr (kVec) {
        constexpr int V = Vec16<T>::kN;
        if (t + kK <= L) {
#pragma unroll
            for (int k = 0; k < kK; k += V) Vec16<T>::store(row + t + k, v + k);
            return;
        }
    }
#pragma unroll
    for (int k = 0; k < kK; k++)
        if (t + k < L) row[t + k] = from_f32<T>(v[k]);
}

// Register budget: 96 per thread without z and D lets an SM hold 21 warps, so the
// Mamba-shaped SM1 workload (12,288 channels, 3,072 warps) runs in one wave; at
// the unconstrained ~110 it needs 1.3 waves, and each warp walks the whole
// sequence, so the partial second wave costs nearly a full one. With z or D the
// kernel takes up to 128.
#ifndef SSM_SCALAR_MAXNREG
#define SSM_SCALAR_MAXNREG 96
#endif
template <typename Tin, typename Tout, bool kVec, bool kZ, bool kD>
__global__ void __maxnreg__((kZ || kD) ? 128 : SSM_SCALAR_MAXNREG) scalar_scan_kernel(ScanArgs a) {
    constexpr bool kAcc = sizeof(Tin) == 4;
    using Dec = Decay<kAcc>;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c = lane / kSeg, s = lane % kSeg;
    const int64_t rows = a.batch * a.dim;
    const int64_t row = ((int64_t)blockIdx.x * kWarps + warp) * kChPerWarp + c;
    const bool ok = row < rows;
    const int64_t b = ok ? row / a.dim : 0, d = ok ? row % a.dim : 0;
    const int64_t L = a.seqlen;
    const Tin* up = static_cast<const Tin*>(a.u) + row * L;
    const Tin* dp = static_cast<const Tin*>(a.delta) + row * L;
    const Tin* zp = kZ ? static_cast<const Tin*>(a.z) + row * L : nullptr;
    const Tin* Bp = static_cast<const Tin*>(a.B) + b * L;
    const Tin* Cp = static_cast<const Tin*>(a.C) + b * L;
    Tout* yp = static_cast<Tout*>(a.y) + row * L;
    const float Ad = ok ? a.A[d] * Dec::scale : 0.f;
    const float bias = (ok && a.delta_bias) ? a.delta_bias[d] : 0.f;
    const float Dd = (kD && ok) ? a.D[d] : 0.f;
    float carry = (ok && a.h0) ? a.h0[row] : 0.f, carry_lo = 0.f;

    // The next chunk's inputs are loaded while the current one computes: u, delta
    // and B once the current ones are consumed (after the first pass), C and z
    // after the last use of the current ones (after the second pass), so no
    // register copies are needed. Whole chunks (all but the last) skip every
    // bounds check: one warp-uniform test per chunk.
    float nu[kK], nd[kK], nB[kK], nC[kK], nz[kK];
    const int64_t t_l = (int64_t)s * kK;   // the lane's first step within a chunk
    auto load_run = [&](const Tin* row, int64_t t, bool full, float* out) {
        if (kVec && full && ok) {
            constexpr int V = Vec16<Tin>::kN;
#pragma unroll
            for (int k = 0; k < kK; k += V) Vec16<Tin>::load(row + t + k, out + k);
        } else {
            load_k<Tin, kVec>(row, t, L, ok, out);
        }
    };
    if (L > 0) {
        const bool full = kChunk <= L;
        load_run(up, t_l, full, nu);
        load_run(dp, t_l, full, nd);
        load_run(Bp, t_l, full, nB);
        load_run(Cp, t_l, full, nC);
        if constexpr (kZ) load_run(zp, t_l, full, nz);
    }
    for (int64_t t0 = 0; t0 < L; t0 += kChunk) {
        const int64_t t = t0 + t_l;
        const bool full = t0 + kChunk <= L;            // warp-uniform
        const bool next_full = t0 + 2 * kChunk <= L;
        const bool has_next = t0 + kChunk < L;
        float du[kK], p[kK], bb[kK];
        // steps of this lane's run inside the sequence
        const int nvalid = full ? kK : (int)max((int64_t)0, min((int64_t)kK, L - t));
        auto first = [&](auto check) {
#pragma unroll
            for (int k = 0; k < kK; k++) {
                const float x = nd[k] + bias;
                float dt = a.softplus ? softplus_acc<kAcc>(x) : x;
                if constexpr (decltype(check)::value) {
                    if (k >= nvalid) dt = 0.f;         // identity step past the end
                }
                if constexpr (kD) du[k] = Dd * nu[k];
                p[k] = Dec::make(dt * Ad);
                bb[k] = dt * nu[k] * nB[k];
            }
        };
        if (full) first(std::false_type{});
        else first(std::true_type{});
        if (has_next) {
            load_run(up, t + kChunk, next_full, nu);
            load_run(dp, t + kChunk, next_full, nd);
            load_run(Bp, t + kChunk, next_full, nB);
        }
        // fold the lane's steps into one map (P, H), then scan the 8 lane maps
        float P = Dec::one(), H = 0.f;
#pragma unroll
        for (int k = 0; k < kK; k++) {
            H = Dec::step(p[k], H, bb[k]);
            P = Dec::mul(p[k], P);
        }
#pragma unroll
        for (int off = 1; off < kSeg; off <<= 1) {
            const float Pp = __shfl_up_sync(0xffffffffu, P, off, kSeg);
            const float Hp = __shfl_up_sync(0xffffffffu, H, off, kSeg);
            if (s >= off) {
                H = Dec::step(P, Hp, H);
                P = Dec::mul(P, Pp);
            }
        }
        float Pe = __shfl_up_sync(0xffffffffu, P, 1, kSeg);
        float He = __shfl_up_sync(0xffffffffu, H, 1, kSeg);
        if (s == 0) { Pe = Dec::one(); He = 0.f; }
        const float Pt = __shfl_sync(0xffffffffu, P, kSeg - 1, kSeg);
        const float Ht = __shfl_sync(0xffffffffu, H, kSeg - 1, kSeg);
        float y[kK], C[kK], zz[kK];
#pragma unroll
        for (int k = 0; k < kK; k++) {
            C[k] = nC[k];
            if constexpr (kZ) zz[k] = nz[k];
        }
        if constexpr (kAcc) {
            float dlt = fmaf(Pe, carry, He) + carry_lo;
            float h = carry + dlt;
#pragma unroll
            for (int k = 0; k < kK; k++) {
                dlt += fmaf(p[k], h, bb[k]);
                h = carry + dlt;
                y[k] = C[k] * h;
            }
            two_sum(carry, fmaf(Pt, carry, Ht) + carry_lo, carry, carry_lo);
        } else {
            float h = Dec::step(Pe, carry, He);
#pragma unroll
            for (int k = 0; k < kK; k++) {
                h = Dec::step(p[k], h, bb[k]);
                y[k] = C[k] * h;
            }
            carry = Dec::step(Pt, carry, Ht);
        }
        if (has_next) {
            load_run(Cp, t + kChunk, next_full, nC);
            if constexpr (kZ) load_run(zp, t + kChunk, next_full, nz);
        }
#pragma unroll
        for (int k = 0; k < kK; k++) {
            if constexpr (kD) y[k] += du[k];
            if constexpr (kZ) y[k] *= silu_acc<kAcc>(zz[k]);
        }
        if (ok) store_k<Tout, kVec>(yp, t, L, y);
    }
    if (ok && s == 0 && a.h_last) a.h_last[row] = carry + carry_lo;
}


// ---------------------------------------------------------------------------
// Streaming form of the same kernel for 16-byte aligned rows with dim % 4 == 0
// (a warp's 4 channels then share one batch row, hence one B and one C row): the
// inputs of each 64-step chunk arrive by bulk asynchronous copies
// (cp.async.bulk: 4 rows of u and of delta, one row of B and of C, 4 rows of z)
// in a kRing-deep shared-memory ring per warp, completion counted on an mbarrier,
// so kRing chunks are in flight per warp without holding registers; the lanes
// read their 8 steps from shared memory. The arithmetic is the kernel above's.
// Every mbarrier wait is bounded; on expiry the warp records the failure in
// g_scalar_status, waits (again bounded) for its copies in flight and returns.
// ---------------------------------------------------------------------------
#ifndef SSM_SCALAR_RING
#define SSM_SCALAR_RING 3
#endif
constexpr int kRing = SSM_SCALAR_RING;
constexpr uint32_t kRingWaitLimit = 1u << 24;
__device__ int g_scalar_status;   // 0, or the line of a wait that ran out of budget

__device__ __forceinline__ uint32_t sm_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void ring_bar_init(uint64_t* bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(sm_u32(bar)) : "memory");
}
__device__ __forceinline__ void ring_expect(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sm_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool ring_wait(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < kRingWaitLimit; i++) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(sm_u32(bar)), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}
__device__ __forceinline__ void ring_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     sm_u32(dst)),
                 "l"(src), "r"(bytes), "r"(sm_u32(bar))
                 : "memory");
}

template <typename Tin, bool kZ>
struct RingStage {
    Tin u[kChPerWarp][kChunk], dl[kChPerWarp][kChunk];
    Tin B[kChunk], C[kChunk];
    Tin z[kZ ? kChPerWarp : 1][kZ ? kChunk : 8];
};

template <typename Tin, typename Tout, bool kZ, bool kD>
__global__ void __launch_bounds__(32) __maxnreg__((kZ || kD) ? 128 : SSM_SCALAR_MAXNREG)
    scalar_scan_ring_kernel(ScanArgs a) {
    constexpr bool kAcc = sizeof(Tin) == 4;
    using Dec = Decay<kAcc>;
    __shared__ __align__(128) RingStage<Tin, kZ> s_st[kRing];
    __shared__ __align__(8) uint64_t s_full[kRing];
    const int lane = threadIdx.x & 31;
    const int c = lane / kSeg, s = lane % kSeg;
    const int64_t rows = a.batch * a.dim;
    const int64_t row0 = (int64_t)blockIdx.x * kChPerWarp;    // dim % 4 == 0: rows share b
    const int64_t row = row0 + c;
    const bool ok = row < rows;
    const int nrow = (int)min((int64_t)kChPerWarp, rows - row0);
    const int64_t b = row0 / a.dim, d = ok ? row % a.dim : 0;
    const int64_t L = a.seqlen;
    const int64_t n_chunks = (L + kChunk - 1) / kChunk;
    const Tin* ub = static_cast<const Tin*>(a.u) + row0 * L;
    const Tin* db = static_cast<const Tin*>(a.delta) + row0 * L;
    const Tin* zb = kZ ? static_cast<const Tin*>(a.z) + row0 * L : nullptr;
    const Tin* Bb = static_cast<const Tin*>(a.B) + b * L;
    const Tin* Cb = static_cast<const Tin*>(a.C) + b * L;
    Tout* yp = static_cast<Tout*>(a.y) + row * L;
    const float Ad = ok ? a.A[d] * Dec::scale : 0.f;
    const float bias = (ok && a.delta_bias) ? a.delta_bias[d] : 0.f;
    const float Dd = (kD && ok) ? a.D[d] : 0.f;
    float carry = (ok && a.h0) ? a.h0[row] : 0.f, carry_lo = 0.f;

    // lanes 0 .. nrow-1 copy the u rows, nrow .. 2 nrow-1 the delta rows, then B,
    // C and (z) the z rows: one bulk copy per lane, lane 0 first posts the bytes
    auto issue = [&](int64_t k) {
        const int st = (int)(k % kRing);
        const int64_t t0 = k * kChunk;
        const uint32_t n = (uint32_t)min((int64_t)kChunk, L - t0) * (uint32_t)sizeof(Tin);
        const uint32_t copies = (uint32_t)(2 * nrow + 2 + (kZ ? nrow : 0));
        if (lane == 0) ring_expect(&s_full[st], copies * n);
        __syncwarp();
        RingStage<Tin, kZ>& S = s_st[st];
        if (lane < nrow) ring_copy(S.u[lane], ub + lane * L + t0, n, &s_full[st]);
        else if (lane < 2 * nrow) ring_copy(S.dl[lane - nrow], db + (lane - nrow) * L + t0, n, &s_full[st]);
        else if (lane == 2 * nrow) ring_copy(S.B, Bb + t0, n, &s_full[st]);
        else if (lane == 2 * nrow + 1) ring_copy(S.C, Cb + t0, n, &s_full[st]);
        else if constexpr (kZ) {
            if (lane < 3 * nrow + 2) ring_copy(S.z[lane - 2 * nrow - 2], zb + (lane - 2 * nrow - 2) * L + t0, n, &s_full[st]);
        }
    };
    if (lane == 0) {
        for (int st = 0; st < kRing; st++) ring_bar_init(&s_full[st]);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    for (int64_t k = 0; k < kRing && k < n_chunks; k++) issue(k);

    bool failed = false;
    int64_t k = 0;
    for (; k < n_chunks; k++) {
        const int st = (int)(k % kRing);
        const bool got = ring_wait(&s_full[st], (uint32_t)((k / kRing) & 1));
        if (__any_sync(0xffffffffu, !got)) { failed = true; break; }
        const RingStage<Tin, kZ>& S = s_st[st];
        const int64_t t0 = k * kChunk;
        const int64_t t = t0 + (int64_t)s * kK;
        const bool full = t0 + kChunk <= L;                       // warp-uniform
        const int nvalid = full ? kK : (int)max((int64_t)0, min((int64_t)kK, L - t));
        float nu[kK], nd[kK], nB[kK], nC[kK], nz[kK];
        {
            constexpr int V = Vec16<Tin>::kN;
#pragma unroll
            for (int q = 0; q < kK; q += V) {
                Vec16<Tin>::load_shared(&S.u[c][s * kK + q], nu + q);
                Vec16<Tin>::load_shared(&S.dl[c][s * kK + q], nd + q);
                Vec16<Tin>::load_shared(&S.B[s * kK + q], nB + q);
                Vec16<Tin>::load_shared(&S.C[s * kK + q], nC + q);
                if constexpr (kZ) Vec16<Tin>::load_shared(&S.z[c][s * kK + q], nz + q);
            }
        }
        if (!full) {
            // steps past the end hold stale shared memory: make them identity steps
#pragma unroll
            for (int q = 0; q < kK; q++)
                if (q >= nvalid) { nu[q] = 0.f; nd[q] = 0.f; nB[q] = 0.f; nC[q] = 0.f; nz[q] = 0.f; }
        }
        // this lane's reads of the stage (generic proxy) precede the refill's bulk
        // writes (async proxy)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (k + kRing < n_chunks) issue(k + kRing);

        float du[kK], p[kK], bb[kK];
        // whole chunks (all but the last) take no per-step bounds test
        auto first = [&](auto check) {
#pragma unroll
            for (int q = 0; q < kK; q++) {
                const float x = nd[q] + bias;
                float dt = a.softplus ? softplus_acc<kAcc>(x) : x;
                if constexpr (decltype(check)::value) {
                    if (q >= nvalid) dt = 0.f;                     // identity step past the end
                }
                if constexpr (kD) du[q] = Dd * nu[q];
                p[q] = Dec::make(dt * Ad);
                bb[q] = dt * nu[q] * nB[q];
            }
        };
        if (full) first(std::false_type{});
        else first(std::true_type{});
        float P = Dec::one(), H = 0.f;
#pragma unroll
        for (int q = 0; q < kK; q++) {
            H = Dec::step(p[q], H, bb[q]);
            P = Dec::mul(p[q], P);
        }
#pragma unroll
        for (int off = 1; off < kSeg; off <<= 1) {
            const float Pp = __shfl_up_sync(0xffffffffu, P, off, kSeg);
            const float Hp = __shfl_up_sync(0xffffffffu, H, off, kSeg);
            if (s >= off) {
                H = Dec::step(P, Hp, H);
                P = Dec::mul(P, Pp);
            }
        }
        float Pe = __shfl_up_sync(0xffffffffu, P, 1, kSeg);
        float He = __shfl_up_sync(0xffffffffu, H, 1, kSeg);
        if (s == 0) { Pe = Dec::one(); He = 0.f; }
        const float Pt = __shfl_sync(0xffffffffu, P, kSeg - 1, kSeg);
        const float Ht = __shfl_sync(0xffffffffu, H, kSeg - 1, kSeg);
        float y[kK];
        if constexpr (kAcc) {
            float dlt = fmaf(Pe, carry, He) + carry_lo;
            float h = carry + dlt;
#pragma unroll
            for (int q = 0; q < kK; q++) {
                dlt += fmaf(p[q], h, bb[q]);
                h = carry + dlt;
                y[q] = nC[q] * h;
            }
            two_sum(carry, fmaf(Pt, carry, Ht) + carry_lo, carry, carry_lo);
        } else {
            float h = Dec::step(Pe, carry, He);
#pragma unroll
            for (int q = 0; q < kK; q++) {
                h = Dec::step(p[q], h, bb[q]);
                y[q] = nC[q] * h;
            }
            carry = Dec::step(Pt, carry, Ht);
        }
#pragma unroll
        for (int q = 0; q < kK; q++) {
            if constexpr (kD) y[q] += du[q];
            if constexpr (kZ) y[q] *= silu_acc<kAcc>(nz[q]);
        }
        if (ok) store_k<Tout, true>(yp, t, L, y);
    }
    if (failed) {
        if (lane == 0) atomicExch(&g_scalar_status, __LINE__);
        for (int64_t kk = k; kk < k + kRing && kk < n_chunks; kk++)
            (void)ring_wait(&s_full[kk % kRing], (uint32_t)((kk / kRing) & 1));
        return;
    }
    if (ok && s == 0 && a.h_last) a.h_last[row] = carry + carry_lo;
}

template <typename Tin, typename Tout>
cudaError_t launch(const ScanArgs& a, cudaStream_t s) {
    const int64_t rows = a.batch * a.dim;
    if (rows == 0) return cudaSuccess;
    const int64_t per_cta = (int64_t)kWarps * kChPerWarp;
    const int64_t ctas = (rows + per_cta - 1) / per_cta;
    if (ctas > ((int64_t)1 << 31) - 1) return cudaErrorInvalidValue;
    // z (the gate) and D (the skip) are template switches: without them the kernel
    // holds no registers for them
    const unsigned g = (unsigned)ctas;
    if (a.vec && a.dim % kChPerWarp == 0 && a.seqlen > 0) {
        switch ((a.z ? 2 : 0) | (a.D ? 1 : 0)) {
            case 0: scalar_scan_ring_kernel<Tin, Tout, false, false><<<g, 32, 0, s>>>(a); break;
            case 1: scalar_scan_ring_kernel<Tin, Tout, false, true><<<g, 32, 0, s>>>(a); break;
            case 2: scalar_scan_ring_kernel<Tin, Tout, true, false><<<g, 32, 0, s>>>(a); break;
            default: scalar_scan_ring_kernel<Tin, Tout, true, true><<<g, 32, 0, s>>>(a); break;
        }
        return cudaGetLastError();
    }
    const int sel = (a.vec ? 4 : 0) | (a.z ? 2 : 0) | (a.D ? 1 : 0);
    switch (sel) {
        case 0: scalar_scan_kernel<Tin, Tout, false, false, false><<<g, kThreads, 0, s>>>(a); break;
        case 1: scalar_scan_kernel<Tin, Tout, false, false, true><<<g, kThreads, 0, s>>>(a); break;
        case 2: scalar_scan_kernel<Tin, Tout, false, true, false><<<g, kThreads, 0, s>>>(a); break;
        case 3: scalar_scan_kernel<Tin, Tout, false, true, true><<<g, kThreads, 0, s>>>(a); break;
        case 4: scalar_scan_kernel<Tin, Tout, true, false, false><<<g, kThreads, 0, s>>>(a); break;
        case 5: scalar_scan_kernel<Tin, Tout, true, false, true><<<g, kThreads, 0, s>>>(a); break;
        case 6: scalar_scan_kernel<Tin, Tout, true, true, false><<<g, kThreads, 0, s>>>(a); break;
        default: scalar_scan_kernel<Tin, Tout, true, true, true><<<g, kThreads, 0, s>>>(a); break;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t scalar_status(int* line, bool clear, cudaStream_t s) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(line, g_scalar_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && clear && *line != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_scalar_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

cudaError_t launch_scan_scalar(const ScanArgs& a, cudaStream_t s) {
    if (a.in_dtype == kBF16)
        return a.out_dtype == kBF16 ? launch<__nv_bfloat16, __nv_bfloat16>(a, s) : launch<__nv_bfloat16, float>(a, s);
    return a.out_dtype == kBF16 ? launch<float, __nv_bfloat16>(a, s) : launch<float, float>(a, s);
}

}  // namespace ssm
