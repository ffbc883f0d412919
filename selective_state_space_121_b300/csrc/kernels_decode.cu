// kernels_decode.cu -- single-token state update (decode) for the selective scan.
//
// One token of the recurrence (Mamba SSM complete guide (youngju.dev), section 5,
// the selective_scan loop body; applied once per token it is the O(1)-per-token
// recurrent inference of the SM1 (Scalar Mamba1) page's section details):
//     s_n <- exp(dt*A_n) * s_n + dt*B_n*x ;  y = sum_n C_n s_n + D x ;  y *= silu(z)
// on a resident fp32 (batch, dim, dstate) state, in place.
//
// The kernel is HBM-bound: 8 bytes of state traffic per (b, d, n) (read + write)
// against one exp and four FP32 operations, provided the per-element instruction
// count stays small (the streaming form below measured issue-bound at ~60
// instructions per element with a library log1p softplus). Precision as in the
// scan kernels: bf16 inputs take softplus and silu through the SFU (ex2, lg2,
// rcp), fp32 inputs the accurate forms of common.cuh. Layout of the work:
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
                // bf16 inputs: SFU softplus in the log2 domain, its argument formed as
                // the prefill scan forms it; fp32 inputs: accurate
                float dts, dtx;
                const float v = dv[r] + bias;
                if constexpr (sizeof(Tin) == 2) {
                    const float xl = fmaf(dv[r], kLog2e, bias * kLog2e);
                    dts = a.softplus ? softplus_log2(xl) : xl;
                    dtx = dts * (kLn2 * xt[r]);
                } else {
                    const float dt = a.softplus ? softplus_acc<true>(v) : v;
                    dts = dt * Dec::scale;
                    dtx = dt * xt[r];
                }
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
                if (zp) yv *= silu_acc<sizeof(Tin) == 4>(zv[r]);
                y[b * a.dim + d] = from_f32<Tout>(yv);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Streaming variant (dstate 8 or 16, bf16/fp32 inputs with 16-byte aligned rows):
// a persistent CTA owns kTileCh channels and walks batch rows (its A, bias and D
// stay in registers); per row, the tile's
// state (kTileCh x N fp32, contiguous), its x, delta, z (kTileCh values each) and
// the row's B and C are fetched into a kStages-deep shared-memory ring with bulk
// asynchronous copies (cp.async.bulk, completion counted on an mbarrier), so the
// bytes in flight are set by the ring, not by registers: with 4 stages and ~4 CTAs
// per SM about 70 KB per SM are outstanding, enough to cover HBM latency.
// Threads read their 4 states from shared memory, update them and store them
// straight back to global memory with 16-byte stores. Every mbarrier wait is
// bounded; on expiry the CTA records the failure in g_decode_status, waits (again
// bounded) for its own copies in flight and returns.
// ---------------------------------------------------------------------------
// threads per CTA (a build option): 4 per channel at d_state 16, so a CTA's tile
// is kTmaThreads / 4 channels of one batch row
#ifndef SSM_DECODE_THREADS
#define SSM_DECODE_THREADS 256
#endif
constexpr int kTmaThreads = SSM_DECODE_THREADS;
// ring depth (a build option; static shared memory keeps it under 48 KB per CTA)
#ifndef SSM_DECODE_STAGES
#define SSM_DECODE_STAGES 4
#endif
constexpr int kStages = SSM_DECODE_STAGES;
constexpr uint32_t kWaitLimit = 1u << 24;


__device__ int g_decode_status;   // 0, or the line of a wait that ran out of budget

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}
// true once the phase with this parity has completed
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < kWaitLimit; i++)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
// global -> shared bulk copy of `bytes` (a multiple of 16, both addresses 16-byte
// aligned), completion counted on `bar`
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

template <int N, typename Tin>
struct TmaTile {
    static constexpr int G = N / 4;                    // lanes per channel (4 states each)
    static constexpr int kTileCh = kTmaThreads / G;    // channels per tile
    float state[kTileCh * N];
    Tin x[kTileCh], dl[kTileCh], z[kTileCh];
    Tin B[N], C[N];
};

template <int N, typename Tin, typename Tout>
__global__ void __launch_bounds__(kTmaThreads) state_update_tma_kernel(DecodeArgs a) {
    using Tile = TmaTile<N, Tin>;
    constexpr int G = Tile::G, kTileCh = Tile::kTileCh;
    using Dec = Decay<sizeof(Tin) == 4>;
    __shared__ __align__(128) Tile s_tile[kStages];
    __shared__ __align__(8) uint64_t s_full[kStages];

    // CTA (range r, row offset q) owns channels [r*kTileCh, (r+1)*kTileCh) of batch
    // rows q, q + R, q + 2R, ... (gridDim.x = ranges * R): its A, bias and D stay in
    // registers for the whole walk
    const int64_t ranges = (a.dim + kTileCh - 1) / kTileCh;
    const int64_t R = gridDim.x / ranges;
    const int64_t r = blockIdx.x % ranges, q = blockIdx.x / ranges;
    const int64_t d0 = r * kTileCh;
    const int64_t nch = min((int64_t)kTileCh, a.dim - d0);
    const int64_t n_rows = q < a.batch ? (a.batch - 1 - q) / R + 1 : 0;   // rows of this CTA
    const int c = threadIdx.x / G, j = threadIdx.x % G;
    const int64_t d = d0 + c;
    const bool ok = c < nch;
    const Tin* zp = static_cast<const Tin*>(a.z);
    Tout* y = static_cast<Tout*>(a.y);
    float Av[4] = {0.f, 0.f, 0.f, 0.f};
    float bias = 0.f, Dd = 0.f;
    if (ok) {
        const float4 A4 = *reinterpret_cast<const float4*>(a.A + d * N + j * 4);
        Av[0] = A4.x; Av[1] = A4.y; Av[2] = A4.z; Av[3] = A4.w;
        bias = a.delta_bias ? a.delta_bias[d] : 0.f;
        Dd = a.D ? a.D[d] : 0.f;
    }

    // the copies of this CTA's k-th row (thread 0 only)
    auto issue = [&](int64_t k) {
        if (k >= n_rows) return;
        const int st = (int)(k % kStages);
        const int64_t b = q + k * R;
        const uint32_t sb = (uint32_t)(nch * N * 4), xb = (uint32_t)(nch * sizeof(Tin)),
                       bb = (uint32_t)(N * sizeof(Tin));
        const uint32_t total = sb + xb * (zp ? 3u : 2u) + 2u * bb;
        Tile& t = s_tile[st];
        mbar_expect_tx(&s_full[st], total);
        bulk_g2s(t.state, a.state + (b * a.dim + d0) * N, sb, &s_full[st]);
        bulk_g2s(t.x, static_cast<const Tin*>(a.x) + b * a.dim + d0, xb, &s_full[st]);
        bulk_g2s(t.dl, static_cast<const Tin*>(a.delta) + b * a.dim + d0, xb, &s_full[st]);
        if (zp) bulk_g2s(t.z, zp + b * a.dim + d0, xb, &s_full[st]);
        bulk_g2s(t.B, static_cast<const Tin*>(a.B) + b * N, bb, &s_full[st]);
        bulk_g2s(t.C, static_cast<const Tin*>(a.C) + b * N, bb, &s_full[st]);
    };

    if (threadIdx.x == 0) {
        for (int st = 0; st < kStages; st++) mbar_init(&s_full[st], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0)
        for (int k = 0; k < kStages; k++) issue(k);

    // this lane's 4 states of channel d in batch row b: sp0 + b * row_stride
    float* const sp0 = a.state + d * N + j * 4;
    const int64_t row_stride = a.dim * N;
    bool failed = false;
    int64_t k = 0;
    for (; k < n_rows; k++) {
        const int st = (int)(k % kStages);
        const uint32_t parity = (uint32_t)((k / kStages) & 1);
        // a wait that runs out of budget skips this thread's work; the end-of-row
        // barrier then stops the whole CTA (the decision has to be uniform)
        const bool got = mbar_wait(&s_full[st], parity);
        const Tile& t = s_tile[st];
        const int64_t b = q + k * R;
        float acc = 0.f, xt = 0.f, zt = 0.f;
        if (ok && got) {
            const float4 s4 = *reinterpret_cast<const float4*>(&t.state[c * N + j * 4]);
            float sv[4] = {s4.x, s4.y, s4.z, s4.w}, Bv[4], Cv[4];
            if constexpr (sizeof(Tin) == 2) {
                // the lane's 4 B and 4 C values: one 8-byte shared load each
                const uint2 bw = *reinterpret_cast<const uint2*>(&t.B[j * 4]);
                const uint2 cw = *reinterpret_cast<const uint2*>(&t.C[j * 4]);
                Bv[0] = __uint_as_float(bw.x << 16); Bv[1] = __uint_as_float(bw.x & 0xffff0000u);
                Bv[2] = __uint_as_float(bw.y << 16); Bv[3] = __uint_as_float(bw.y & 0xffff0000u);
                Cv[0] = __uint_as_float(cw.x << 16); Cv[1] = __uint_as_float(cw.x & 0xffff0000u);
                Cv[2] = __uint_as_float(cw.y << 16); Cv[3] = __uint_as_float(cw.y & 0xffff0000u);
            } else {
                const float4 b4 = *reinterpret_cast<const float4*>(&t.B[j * 4]);
                const float4 c4 = *reinterpret_cast<const float4*>(&t.C[j * 4]);
                Bv[0] = b4.x; Bv[1] = b4.y; Bv[2] = b4.z; Bv[3] = b4.w;
                Cv[0] = c4.x; Cv[1] = c4.y; Cv[2] = c4.z; Cv[3] = c4.w;
            }
            xt = to_f32(t.x[c]);
            const float dlv = to_f32(t.dl[c]);
            // bf16 inputs: softplus through the SFU in the log2 domain (dtl = dt
            // log2 e, the ex2 argument scale), its argument formed as the prefill
            // scan forms it; fp32 inputs: the accurate form
            float dts, dtx;
            if constexpr (sizeof(Tin) == 2) {
                const float xl = fmaf(dlv, kLog2e, bias * kLog2e);
                dts = a.softplus ? softplus_log2(xl) : xl;
                dtx = dts * (kLn2 * xt);
            } else {
                const float v = dlv + bias;
                const float dt = a.softplus ? softplus_acc<true>(v) : v;
                dts = dt * Dec::scale;
                dtx = dt * xt;
            }
#pragma unroll
            for (int i = 0; i < 4; i++) {
                sv[i] = Dec::step(Dec::make(dts * Av[i]), sv[i], dtx * Bv[i]);
                acc = fmaf(Cv[i], sv[i], acc);
            }
            *reinterpret_cast<float4*>(sp0 + b * row_stride) = make_float4(sv[0], sv[1], sv[2], sv[3]);
            if (zp) zt = to_f32(t.z[c]);
        }
#pragma unroll
        for (int off = 1; off < G; off <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (ok && got && j == 0) {
            float yv = fmaf(Dd, xt, acc);
            if (zp) yv *= silu_acc<sizeof(Tin) == 4>(zt);
            y[b * a.dim + d] = from_f32<Tout>(yv);
        }
        // every thread is done with stage st (its reads, generic proxy, ordered
        // before the refill's bulk writes, async proxy); a failed wait anywhere
        // stops the CTA here
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (__syncthreads_or(!got)) {
            failed = true;
            break;
        }
        if (threadIdx.x == 0) issue(k + kStages);
    }
    if (failed) {
        // record, then drain this CTA's copies still in flight before leaving
        if (threadIdx.x == 0) atomicExch(&g_decode_status, __LINE__);
        for (int64_t kk = k; kk < k + kStages && kk < n_rows; kk++)
            (void)mbar_wait(&s_full[kk % kStages], (uint32_t)((kk / kStages) & 1));
    }
}


template <int N, typename Tin, typename Tout>
cudaError_t launch_n(const DecodeArgs& a, cudaStream_t s) {
    constexpr int G = N < 4 ? 1 : N / 4;
    if (a.batch == 0 || a.dim == 0) return cudaSuccess;
    if constexpr (N >= 8) {
        if (a.tma) {
            // persistent: one wave of CTAs
            static const int64_t wave = [] {
                int dev = 0, sms = 148, per_sm = 1;
                if (cudaGetDevice(&dev) == cudaSuccess)
                    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, state_update_tma_kernel<N, Tin, Tout>,
                                                              kTmaThreads, 0);
                return (int64_t)(sms > 0 ? sms : 148) * (per_sm > 0 ? per_sm : 1);
            }();
            // ranges x R CTAs: R row offsets per channel range, about one wave in all
            const int64_t ranges = (a.dim + TmaTile<N, Tin>::kTileCh - 1) / TmaTile<N, Tin>::kTileCh;
            int64_t R = wave / ranges;
            if (R < 1) R = 1;
            if (R > a.batch) R = a.batch;
            const int64_t grid = ranges * R;
            if (grid > ((int64_t)1 << 31) - 1) return cudaErrorInvalidValue;
            state_update_tma_kernel<N, Tin, Tout><<<(unsigned)grid, kTmaThreads, 0, s>>>(a);
            return cudaGetLastError();
        }
    }
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
