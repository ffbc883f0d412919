// kernels_serial.cu -- time-serial selective scan for many channels: each lane owns
// a few states of K channels (K = 1 or 2) and walks time step by step; plus the
// look-back variant that splits time into segments for long sequences.
//
// Operation (Mamba SSM complete guide (youngju.dev), section 5: selective_scan,
// with MambaBlock.ssm's softplus(dt_proj) and MambaBlock.forward's silu(z) gate):
//     h_t = exp(dt_t A) h_{t-1} + dt_t B_t u_t,  y_t = C_t . h_t + D u_t,  y_t *= silu(z_t)
//
// Why time-serial: on B300 the N = 16 bf16 scan is bound by the SM, not by HBM:
// every (t, n) element needs one exp (SFU ex2, 32 per clock per SM) and four FP32
// operations, and two bytes of HBM traffic feed it. With batch * dim in the tens of
// thousands there is enough independent work without splitting time, and walking
// time serially is the formulation with the fewest instructions per element:
//     e = dt*A (packed mul), a = ex2(e), bB = (dt*u)*B (packed mul),
//     h = a*h + bB (packed fma), acc += C*h (packed fma)
// -- 2 packed FP32 instructions and 1 SFU instruction per element, no shuffle
// scan, no second pass.
//
// The operands B_tn and C_tn are the same for every channel of a batch row and
// come from shared memory, and that bandwidth first limited the scan (measured:
// removing the B/C loads made the kernel 1.5x faster while removing every exp
// changed nothing). Three things cut the traffic: in the serial kernel the lanes
// reading one state group form a quarter-warp, so a 16-byte B/C load is a
// broadcast within each quarter (2 passes instead of 4), and on the bf16 path
// B and C stay bf16 there (one 16-byte load gives a lane-step its 4 B and 4 C);
// the look-back kernel gives each lane the same states of K = 2 channels, so one
// load feeds 2K elements. What is left bounding the serial kernel at Mamba-130M
// sizes is issue and latency: about 10 warps per SM.
//
// Work layout. A CTA holds W = 4 warps; warp w owns CPW = 32 K / G consecutive
// channels of batch row b; lane (p, j) (see lane_grp) owns states
// [j*NPL, (j+1)*NPL), NPL = N/G, of channels K*p .. K*p + K-1. Time goes in
// chunks of T steps:
//   A. prologue, one lane per (channel, 16 bytes of consecutive steps): the
//      per-step scalars of the chunk (loaded one chunk ahead into registers) give
//      dt = softplus(delta + bias) and dt*u, written to shared memory; the K
//      channels of a lane are adjacent there, so one load gives a step for all K;
//   B. recurrence, lane (p, j): per step the (dt, dt*u) of its K channels and the
//      B and C values of its states ([t][...] tile, one per CTA: all warps
//      share the batch row); writes its partial C.h sums, 4 steps per store;
//   C. epilogue, same ownership as A: y = sum of the G partials + D*u, times
//      silu(z), stored with 16-byte stores.
// The B/C tile is double-buffered and filled from registers loaded one chunk
// ahead, so the only CTA-wide barrier is one per chunk.
//
// Precision. bf16 inputs (tolerance 2e-3): decay factors on the SFU (Decay<false>),
// dt via softplus(x) = ln2 * log2(1 + 2^(x*log2 e)) with SFU ex2/lg2 -- the kernel
// keeps dtl = dt*log2(e) (the ex2 argument scale) and folds ln2 into the staged B
// tile. fp32 inputs (tolerance 1e-5): accurate softplus, decays as expm1
// (Decay<true>), and the state anchored at each chunk start: h = (hhi + hlo) +
// dlt, where the anchor is an unevaluated fp32 pair and dlt the change since the
// chunk start, so a slowly decaying large state is rounded once per output, not
// once per step.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <string.h>

#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace ssm {
namespace {

// warps per CTA (a build option; all warps of a CTA share one batch row's B/C tile)
#ifndef SSM_SERIAL_WARPS
#define SSM_SERIAL_WARPS 4
#endif
constexpr int kWarps = SSM_SERIAL_WARPS;
// software-pipelined shared-memory operands in the recurrence (a build option;
// measured 2-3% faster at Mamba-130M and Mamba-2.8B sizes)
#ifndef SSM_SERIAL_PIPE
#define SSM_SERIAL_PIPE 1
#endif
constexpr int kThreads = 32 * kWarps;

// Channels per lane a kernel may use: 2 on the bf16 path when a lane holds 2 to 4
// states (more would not fit the registers), else 1. The serial kernel keeps 1: at
// Mamba-130M sizes (12,288 channels) it needs every warp it can get to hide
// latency, and 2 channels per lane halves the warps (measured slower); the
// look-back kernel, whose segments supply the parallelism, takes 2.
template <int N, int G, typename Tin>
constexpr int max_k() { return (sizeof(Tin) == 2 && N / G >= 2 && N / G <= 4) ? 2 : 1; }

template <int N, int G, typename Tin, int K_>
struct SerialCfg {
    static constexpr int K = K_;
    static_assert(K == 1 || K == max_k<N, G, Tin>(), "unsupported channels per lane");
    // time steps per chunk: short enough that the prologue's registers and the
    // tiles (static shared memory, at most 48 KB) stay small -- a warp owns 32
    // channels at G = 1 and 32 K / G at G >= 2
    static constexpr int kT = G == 1 ? 8 : (K == 2 ? 16 : 32);
    static constexpr int NPL = N / G;                 // states per lane
    static constexpr int CPW = 32 * K / G;            // channels per warp
    static constexpr int V = 16 / (int)sizeof(Tin);   // steps per 16-byte vector
    static constexpr int VPR = kT / V;                // vectors per (channel, chunk) row
    static constexpr int PV = CPW * VPR / 32;         // prologue vectors per lane per tensor
    static constexpr int BCV = 2 * N * VPR;           // vectors per B+C tile
    // row of the (dt, dt*u) tile in floats: kT steps x K channels x 2, padded by
    // 16 bytes to keep rows 16-byte aligned and spread a warp's rows over the banks
    static constexpr int DBS = 2 * K * kT + 4;
    static constexpr int PS = 32 + 1;                 // row (float4) of the partials tile
    static_assert(PV >= 1 && CPW * VPR % 32 == 0, "chunk must cover the warp's channels");
    static_assert(kT % V == 0 && kT % 4 == 0, "chunk must be whole vectors and step groups");
};

// Lane (p, j) of a warp: lane group p (channels K p .. K p + K - 1 of the warp)
// and state group j (states j NPL .. j NPL + NPL - 1). At K = 1 the 32/G lanes of
// one state group are consecutive -- at G = 4 a quarter-warp -- so the 8 lanes of
// a quarter read the same B/C address and a 16-byte shared load takes 2 passes
// instead of 4 (measured on B300: 2.2 against 4.0 cycles per warp load; the
// Mamba-130M scan runs 7% faster). At K = 2 the G lanes of a channel group are
// adjacent instead: there each step's (dt, dt*u) load is a 16-byte one too, and
// this order measured 7% faster in the look-back. A channel's partial C.h sums
// meet in shared memory, so its G lanes need not be adjacent.
template <int G, int K> __device__ __forceinline__ int lane_grp(int lane) {
    return K == 1 ? lane % (32 / G) : lane / G;
}
template <int G, int K> __device__ __forceinline__ int lane_sgrp(int lane) {
    return K == 1 ? lane / (32 / G) : lane % G;
}
template <int G, int K> __device__ __forceinline__ int lane_of(int p, int j) {
    return K == 1 ? j * (32 / G) + p : p * G + j;
}

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

// 8 bf16 values of a 16-byte vector in reverse order
__device__ __forceinline__ uint4 rev8(uint4 v) {
    return make_uint4(__byte_perm(v.w, 0, 0x1032), __byte_perm(v.z, 0, 0x1032), __byte_perm(v.y, 0, 0x1032),
                      __byte_perm(v.x, 0, 0x1032));
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

// Per-lane recurrence state of the serial kernels, for K channels: the lane's NPL
// states in pairs (the packed f32x2 operands); on the fp32 path also the chunk
// anchor (hhi, hlo) and dlt, the change since the chunk start; for the aggregate
// pass the sum of dt*scale over the pass (Kahan-compensated on the fp32 path).
template <int K, int NPL>
struct LaneState {
    static constexpr int NP2 = (NPL + 1) / 2;
    float2 h2[K][NP2];
    float hhi[K][NPL], hlo[K][NPL], dlt[K][NPL];
    float sdt[K], sdt_c[K];
};

// Tensor maps of the bulk-copy (TMA) input path: u, delta, z as (L, dim, batch)
// and B, C as (L, N, batch), bf16, boxes of one chunk of the CTA's channels (the
// B and C boxes hold all N states).
struct ScanMaps {
    CUtensorMap u, d, z, B, C;
};

__device__ int g_prefill_status;   // 0, or the line of a bulk-copy wait that ran out of budget
constexpr uint32_t kTmaWaitLimit = 1u << 24;

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// The chunk tiles of a CTA (separate arrays, not one struct, so the compiler sees
// that the partial-sum stores cannot alias the operand loads of later steps), and
// for the bulk-copy path the one-chunk input stage, its mbarrier, the tensor maps
// and the CTA's first channel.
template <int N, int G, typename Tin, int K>
struct Tiles {
    using Cfg = SerialCfg<N, G, Tin, K>;
    float (*bc)[Cfg::kT][2 * N];                  // [buf][t][B n.. | C n..]
    float (*db)[Cfg::CPW / Cfg::K][Cfg::DBS];     // [warp][lane group][t][K][dt, dt*u]
    float4 (*p)[Cfg::K][Cfg::kT / 4][Cfg::PS];    // [warp][k][t/4][lane]: partial C.h
    unsigned char* stage;                         // u, delta, z tiles, then B, C (bulk-copy path)
    uint64_t* full;                               // its mbarrier
    const ScanMaps* maps;
    int64_t cta_d0;
};

// Bytes of the bulk-copy stage: u, delta, z tiles of the CTA's channels for one
// chunk, then the B and C tiles.
template <int N, int G, typename Tin, int K>
struct StageGeom {
    using Cfg = SerialCfg<N, G, Tin, K>;
    static constexpr int CPC = kWarps * Cfg::CPW;                              // channels per CTA
    static constexpr int XB = CPC * Cfg::kT * (int)sizeof(Tin);
    static constexpr int BB = N * Cfg::kT * (int)sizeof(Tin);
    static constexpr int BYTES = 3 * XB + 2 * BB;
    // 64-byte tile rows (the time-serial kernel's 32-step bf16 chunks) take the
    // 64-byte TMA swizzle: a quarter-warp reads one 16-byte chunk of 8 consecutive
    // rows, which unswizzled puts 4 lanes on each bank group (16 wavefronts per
    // warp load instead of 4); the swizzle stores chunk j of row r at chunk
    // j ^ ((r >> 1) & 3) of the row
    static constexpr bool kSw64 = Cfg::kT * (int)sizeof(Tin) == 64;
    // byte offset of elements [t, t + 8) of tile row r (t a multiple of 8)
    static __device__ __forceinline__ int off(int r, int t) {
        const int j = t * (int)sizeof(Tin) / 16;
        return r * Cfg::kT * (int)sizeof(Tin) + ((kSw64 ? (j ^ ((r >> 1) & 3)) : j) << 4);
    }
};

template <int N, int G, int K>
using A2Arr = float2[K][LaneState<1, N / G>::NP2];
template <int N, int G, int K>
using LaneStateT = LaneState<K, N / G>;

// One pass of the serial scan over steps [tb, te) of batch row b, for the warp's
// channels d_warp0 .. d_warp0 + CPW - 1, continuing the lane state S.
//   kFull:  the whole operation; y is written for steps [tb, te).
//   !kFull: the aggregate pass of the look-back: the state recurrence only (B
//           staged, no C, no y) plus the sum of dt*scale, so the caller can form
//           the map of the segment: decay exp(A * sum dt), offset = S.
// Every thread of the CTA must call it with the same (tb, te).
//   kTma:   the chunk inputs arrive by bulk tensor copies (TMA) into the CTA's
//           stage, one chunk ahead, instead of per-lane global loads into
//           registers; `phase` counts the stage mbarrier's completed phases across
//           passes. Returns false when a copy wait ran out of budget (recorded in
//           g_prefill_status; the outputs are then unspecified).
template <int N, int G, int K, typename Tin, typename Tout, bool kVec, bool kFull, bool kTma = false,
          bool kRev = false>
__device__ __forceinline__ bool serial_pass(const ScanArgs& a, int64_t b, int64_t d_warp0, int64_t tb,
                                            int64_t te, const A2Arr<N, G, K>& A2, LaneStateT<N, G, K>& S,
                                            const Tiles<N, G, Tin, K>& tl, uint32_t* phase = nullptr) {
    using Cfg = SerialCfg<N, G, Tin, K>;
    constexpr int NPL = Cfg::NPL, V = Cfg::V, VPR = Cfg::VPR, PV = Cfg::PV, kT = Cfg::kT, CPW = Cfg::CPW;
    constexpr int NP2 = LaneState<K, NPL>::NP2;
    constexpr bool kAcc = sizeof(Tin) == 4;
    constexpr int BCV = kFull ? Cfg::BCV : Cfg::BCV / 2;   // the aggregate pass stages B only
    constexpr int BCPT = (BCV + kThreads - 1) / kThreads;
    // Serial kernel, bf16 inputs, 4 states per lane: B and C stay bf16 in shared
    // memory, a lane's 4 B and 4 C values of a step side by side in one 16-byte
    // slot, so one quarter-warp broadcast load serves a lane-step: half the
    // shared-memory wavefronts of fp32 operands for one integer unpacking op per
    // value. Measured: 10% faster at Mamba-2.8B sizes (4-5 CTAs per SM, where
    // shared memory is the limit), 1% slower at Mamba-130M sizes (2.6 CTAs per
    // SM, latency-bound), slower in the look-back (K = 2 reads each slot for two
    // channels already), where it is off.
    constexpr bool kRawBC = !kAcc && NPL == 4 && K == 1;
    // A raw tile row (one step) has N/2 16-byte slots, state group g in slot
    // g ^ ((2 (t / 8)) mod N/2): the lanes staging 8-step vectors of one tensor
    // then write to 16 different banks (unswizzled, the rows t, t+8, t+16, t+24
    // they fill at once share banks); reads stay one slot per quarter-warp.
    auto raw_slot = [](int g, int t) { return g ^ ((2 * (t / 8)) & (N / 2 - 1)); };
    using Dec = Decay<kAcc>;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t L = a.seqlen;
    const Tin* u_base = static_cast<const Tin*>(a.u);
    const Tin* dl_base = static_cast<const Tin*>(a.delta);
    const Tin* z_base = static_cast<const Tin*>(a.z);
    const Tin* B_b = static_cast<const Tin*>(a.B) + b * N * L;
    const Tin* C_b = static_cast<const Tin*>(a.C) + b * N * L;
    Tout* y_base = static_cast<Tout*>(a.y);
    const bool has_z = kFull && a.z != nullptr;
    constexpr bool rev = kTma && kRev;   // reversed walk (built for the bulk-copy path only)
    const int p = lane_grp<G, K>(lane), j = lane_sgrp<G, K>(lane);

    // prologue/epilogue ownership: vector q of this lane covers channel pc[q],
    // steps pt[q] .. pt[q]+V of the chunk
    int pc[PV], pt[PV];
    float bias[PV], Dd[PV];
    bool chan_ok[PV];
#pragma unroll
    for (int q = 0; q < PV; q++) {
        const int v = q * 32 + lane;
        // K = 1: a quarter-warp's lanes take 8 channels at the same steps (their
        // (dt, dt*u) stores and partial-sum reads are conflict-free). K = 2: a lane's
        // neighbours take the next vector of the same channel (with the K = 2
        // partial-sum layout the K = 1 order makes the epilogue's reads 4-way
        // bank conflicts; measured 23% slower in the look-back).
        pc[q] = K == 1 ? v % CPW : v / VPR;
        pt[q] = K == 1 ? (v / CPW) * V : (v % VPR) * V;
        const int64_t d = d_warp0 + pc[q];
        chan_ok[q] = d < a.dim;
        bias[q] = (chan_ok[q] && a.delta_bias) ? a.delta_bias[d] : 0.f;
        if constexpr (!kAcc) bias[q] *= kLog2e;
        Dd[q] = (kFull && chan_ok[q] && a.D) ? a.D[d] : 0.f;
    }

    // one chunk of raw inputs, loaded a chunk ahead
    uint4 ru[PV], rd[PV], rz[PV], rbc[BCPT];
    auto prefetch = [&](int64_t t0) {
#pragma unroll
        for (int q = 0; q < PV; q++) {
            const int64_t row = (b * a.dim + d_warp0 + pc[q]) * L;
            ru[q] = load_raw<Tin, kVec>(u_base + row, t0 + pt[q], L, chan_ok[q]);
            rd[q] = load_raw<Tin, kVec>(dl_base + row, t0 + pt[q], L, chan_ok[q]);
            rz[q] = load_raw<Tin, kVec>(has_z ? z_base + row : u_base, t0 + pt[q], L, chan_ok[q] && has_z);
        }
#pragma unroll
        for (int r = 0; r < BCPT; r++) {
            const int v = r * kThreads + threadIdx.x;
            const int which = v / (N * VPR), rem = v % (N * VPR);
            const int n = rem / VPR, tt = (rem % VPR) * V;
            rbc[r] = load_raw<Tin, kVec>((which ? C_b : B_b) + (int64_t)n * L, t0 + tt, L, v < BCV);
        }
    };

    // bulk-copy path: thread 0 posts the chunk's bytes and issues its tile copies;
    // every thread later reads the same vectors the global loads above would have
    using SG = StageGeom<N, G, Tin, K>;
    auto issue = [&](int64_t t0) {
        const uint32_t bytes = (uint32_t)(2 * SG::XB + (has_z ? SG::XB : 0) + (kFull ? 2 : 1) * SG::BB);
        tc::mbar_expect_tx(tl.full, bytes);
        // reversed walk: the chunk's steps t0 .. t0+kT-1 are positions L-1-t0 down to
        // L-t0-kT, one box starting at L-t0-kT (a multiple of 8: L is, on this path;
        // a negative start reads zeros)
        const int x = rev ? (int)(L - t0 - kT) : (int)t0, y0 = (int)tl.cta_d0, zb = (int)b;
        tc::tma_load_3d(tl.stage, &tl.maps->u, x, y0, zb, tl.full);
        tc::tma_load_3d(tl.stage + SG::XB, &tl.maps->d, x, y0, zb, tl.full);
        if (has_z) tc::tma_load_3d(tl.stage + 2 * SG::XB, &tl.maps->z, x, y0, zb, tl.full);
        tc::tma_load_3d(tl.stage + 3 * SG::XB, &tl.maps->B, x, 0, zb, tl.full);
        if (kFull) tc::tma_load_3d(tl.stage + 3 * SG::XB + SG::BB, &tl.maps->C, x, 0, zb, tl.full);
    };
    // (reversed walk: steps s .. s+V-1 of the chunk sit, in reverse order, at tile
    // columns kT-s-V .. kT-s-1)
    auto read_stage = [&]() {
        const unsigned char* st = tl.stage;
#pragma unroll
        for (int q = 0; q < PV; q++) {
            const int row = warp * CPW + pc[q];
            const int col = rev ? kT - pt[q] - V : pt[q];
            ru[q] = *reinterpret_cast<const uint4*>(st + SG::off(row, col));
            rd[q] = *reinterpret_cast<const uint4*>(st + SG::off(SG::CPC + row, col));
            rz[q] = has_z ? *reinterpret_cast<const uint4*>(st + SG::off(2 * SG::CPC + row, col))
                          : make_uint4(0, 0, 0, 0);
            if (rev) { ru[q] = rev8(ru[q]); rd[q] = rev8(rd[q]); rz[q] = rev8(rz[q]); }
        }
#pragma unroll
        for (int r = 0; r < BCPT; r++) {
            const int v = r * kThreads + threadIdx.x;
            const int which = v / (N * VPR), rem = v % (N * VPR);
            const int n = rem / VPR, tt = (rem % VPR) * V;
            rbc[r] = v < BCV ? *reinterpret_cast<const uint4*>(st + SG::off(3 * SG::CPC + which * N + n,
                                                                            rev ? kT - tt - V : tt))
                             : make_uint4(0, 0, 0, 0);
            if (rev) rbc[r] = rev8(rbc[r]);
        }
    };

    const int64_t n_chunks = te > tb ? (te - tb + kT - 1) / kT : 0;
    bool ok = true;
    if constexpr (kTma) {
        if (n_chunks > 0 && threadIdx.x == 0) issue(tb);
    } else {
        if (n_chunks > 0) prefetch(tb);
    }
    for (int64_t c = 0; c < n_chunks; c++) {
        const int64_t t0 = tb + c * kT;
        const int buf = (int)(c & 1);
        bool got = true;
        if constexpr (kTma) {
            got = tc::mbar_wait(tl.full, *phase & 1u, kTmaWaitLimit);
            if (got) read_stage();
            // these reads of the stage (generic proxy) precede the refill's bulk
            // writes (async proxy) issued after the barrier below
            tc::fence_proxy_async();
        }
        // B/C tile of this chunk, [t][...]: fp32 [n], B then C (B carries ln2 on
        // the bf16 path), or the raw bf16 slots above (ln2 then goes into dt*u)
#pragma unroll
        for (int r = 0; r < BCPT; r++) {
            const int v = r * kThreads + threadIdx.x;
            if (v < BCV) {
                const int which = v / (N * VPR), rem = v % (N * VPR);
                const int n = rem / VPR, tt = (rem % VPR) * V;
                if constexpr (kRawBC) {
                    const uint16_t* raw = reinterpret_cast<const uint16_t*>(&rbc[r]);
                    const int slot = raw_slot(n / NPL, tt) * 2 * NPL + which * NPL + n % NPL;
#pragma unroll
                    for (int k = 0; k < V; k++)
                        reinterpret_cast<uint16_t*>(tl.bc[buf][tt + k])[slot] = raw[k];
                } else {
                    float f[V];
                    unpack<Tin>(rbc[r], f);
                    const float sc = (!kAcc && which == 0) ? kLn2 : 1.f;
#pragma unroll
                    for (int k = 0; k < V; k++) tl.bc[buf][tt + k][which * N + n] = f[k] * sc;
                }
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
            float* dbrow = tl.db[warp][pc[q] / K] + (pc[q] % K) * 2;
            float dts[V];   // dt * Dec::scale
            if constexpr (kAcc) {
#pragma unroll
                for (int k = 0; k < V; k++) {
                    const float x = fd[k] + bias[q];
                    dts[k] = a.softplus ? softplus_acc<true>(x) : x;
                }
            } else {
                // x*log2(e) in pairs; log2(1 + 2^xl) equals xl in fp32 once xl > 24
#pragma unroll
                for (int k = 0; k < V; k += 2) {
                    const float2 xl = fma2(make_float2(fd[k], fd[k + 1]), make_float2(kLog2e, kLog2e),
                                           make_float2(bias[q], bias[q]));
                    dts[k] = a.softplus ? softplus_log2(xl.x) : xl.x;
                    dts[k + 1] = a.softplus ? softplus_log2(xl.y) : xl.y;
                }
            }
            // identity steps past the end (and for channels past dim)
            if (!chan_ok[q] || t0 + pt[q] + V > te) {
#pragma unroll
                for (int k = 0; k < V; k++)
                    if (t0 + pt[q] + k >= te || !chan_ok[q]) dts[k] = 0.f;
            }
            // (dt, dt*u) pairs, two steps per 16-byte store where the K = 1 layout
            // puts consecutive steps side by side
#pragma unroll
            for (int k = 0; k < V; k += 2) {
                float2 u2 = make_float2(fu[k], fu[k + 1]);
                if constexpr (kRawBC) u2 = mul2(u2, make_float2(kLn2, kLn2));
                const float2 bu = mul2(make_float2(dts[k], dts[k + 1]), u2);
                if constexpr (K == 1) {
                    *reinterpret_cast<float4*>(dbrow + (pt[q] + k) * 2) = make_float4(dts[k], bu.x, dts[k + 1], bu.y);
                } else {
                    *reinterpret_cast<float2*>(dbrow + (pt[q] + k) * 2 * K) = make_float2(dts[k], bu.x);
                    *reinterpret_cast<float2*>(dbrow + (pt[q] + k + 1) * 2 * K) = make_float2(dts[k + 1], bu.y);
                }
            }
        }
        if constexpr (kTma) {
            if (__syncthreads_or(!got)) {
                ok = false;
                break;
            }
            ++*phase;
            if (threadIdx.x == 0 && c + 1 < n_chunks) issue(t0 + kT);   // the stage was read by all
        } else {
            if (c + 1 < n_chunks) prefetch(t0 + kT);
            __syncthreads();
        }

        // B. recurrence, in groups of 4 steps: the loads and exps of a group do not
        // depend on the state, only its chained state updates do
        const float* dbg = tl.db[warp][p];
        // (dt*scale, dt*scale*u) of the lane's K channels for 4 steps
        auto load_x = [&](int tg, float2 (&x)[4][K]) {
            if constexpr (K == 2) {
#pragma unroll
                for (int st = 0; st < 4; st++) {
                    const float4 v = *reinterpret_cast<const float4*>(dbg + (tg + st) * 4);
                    x[st][0] = make_float2(v.x, v.y);
                    x[st][K - 1] = make_float2(v.z, v.w);
                }
            } else {
                const float4 x01 = *reinterpret_cast<const float4*>(dbg + tg * 2);
                const float4 x23 = *reinterpret_cast<const float4*>(dbg + tg * 2 + 4);
                x[0][0] = make_float2(x01.x, x01.y); x[1][0] = make_float2(x01.z, x01.w);
                x[2][0] = make_float2(x23.x, x23.y); x[3][0] = make_float2(x23.z, x23.w);
            }
        };
        // B and C of this lane's states at step t, in pairs
        auto load_bc = [&](int t, float2* bq, float2* cq) {
            const float* bc = tl.bc[buf][t];
            if constexpr (kRawBC) {
                const uint4 w = reinterpret_cast<const uint4*>(bc)[raw_slot(j, t)];
                bq[0] = make_float2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u));
                bq[1] = make_float2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
                if constexpr (kFull) {
                    cq[0] = make_float2(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u));
                    cq[1] = make_float2(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u));
                }
            } else if constexpr (NPL % 4 == 0) {
#pragma unroll
                for (int i = 0; i < NPL; i += 4) {
                    const float4 vb = *reinterpret_cast<const float4*>(bc + j * NPL + i);
                    bq[i / 2] = make_float2(vb.x, vb.y); bq[i / 2 + 1] = make_float2(vb.z, vb.w);
                    if constexpr (kFull) {
                        const float4 vc = *reinterpret_cast<const float4*>(bc + N + j * NPL + i);
                        cq[i / 2] = make_float2(vc.x, vc.y); cq[i / 2 + 1] = make_float2(vc.z, vc.w);
                    }
                }
            } else if constexpr (NPL == 2) {
                bq[0] = *reinterpret_cast<const float2*>(bc + j * 2);
                if constexpr (kFull) cq[0] = *reinterpret_cast<const float2*>(bc + N + j * 2);
            } else {
                bq[0] = make_float2(bc[j], 0.f);
                if constexpr (kFull) cq[0] = make_float2(bc[N + j], 0.f);
            }
        };
        // sum of dt*scale for the aggregate decay (Kahan on the fp32 path)
        auto add_dt = [&](int k, float v) {
            if constexpr (kAcc) {
                const float yk = v - S.sdt_c[k];
                const float tk = S.sdt[k] + yk;
                S.sdt_c[k] = (tk - S.sdt[k]) - yk;
                S.sdt[k] = tk;
            } else {
                S.sdt[k] += v;
            }
        };
        // (optionally) the next group's shared-memory operands are read while this
        // group computes: x and the raw B/C words of 4 steps
        constexpr bool kPipe = SSM_SERIAL_PIPE && kRawBC && kFull;
        float2 xn[4][K];
        uint4 wn[4];
        if constexpr (kPipe) {
            load_x(0, xn);
#pragma unroll
            for (int st = 0; st < 4; st++) wn[st] = reinterpret_cast<const uint4*>(tl.bc[buf][st])[raw_slot(j, st)];
        }
#pragma unroll
        for (int tg = 0; tg < kT; tg += 4) {
            float2 x[4][K];
            float2 bq[4][NP2], cq[4][NP2];
            if constexpr (kPipe) {
                uint4 w[4];
#pragma unroll
                for (int st = 0; st < 4; st++) {
                    w[st] = wn[st];
#pragma unroll
                    for (int k = 0; k < K; k++) x[st][k] = xn[st][k];
                }
                if (tg + 4 < kT) {
                    load_x(tg + 4, xn);
#pragma unroll
                    for (int st = 0; st < 4; st++)
                        wn[st] = reinterpret_cast<const uint4*>(tl.bc[buf][tg + 4 + st])[raw_slot(j, tg + 4 + st)];
                }
#pragma unroll
                for (int st = 0; st < 4; st++) {
                    bq[st][0] = make_float2(__uint_as_float(w[st].x << 16), __uint_as_float(w[st].x & 0xffff0000u));
                    bq[st][1] = make_float2(__uint_as_float(w[st].y << 16), __uint_as_float(w[st].y & 0xffff0000u));
                    cq[st][0] = make_float2(__uint_as_float(w[st].z << 16), __uint_as_float(w[st].z & 0xffff0000u));
                    cq[st][1] = make_float2(__uint_as_float(w[st].w << 16), __uint_as_float(w[st].w & 0xffff0000u));
                }
            } else {
                load_x(tg, x);
#pragma unroll
                for (int st = 0; st < 4; st++) load_bc(tg + st, bq[st], cq[st]);
            }
            if constexpr (!kFull) {
#pragma unroll
                for (int st = 0; st < 4; st++)
#pragma unroll
                    for (int k = 0; k < K; k++) add_dt(k, x[st][k].x);
            }
            float acc[K][4];
            if constexpr (!kAcc && NPL % 2 == 0) {
                float2 an[4][K][NP2], bn[4][K][NP2];
#pragma unroll
                for (int st = 0; st < 4; st++)
#pragma unroll
                    for (int k = 0; k < K; k++) {
                        const float2 dtl2 = make_float2(x[st][k].x, x[st][k].x);
                        const float2 bu2 = make_float2(x[st][k].y, x[st][k].y);
#pragma unroll
                        for (int i = 0; i < NP2; i++) {
                            const float2 e = mul2(dtl2, A2[k][i]);
                            an[st][k][i] = make_float2(ex2(e.x), ex2(e.y));
                            bn[st][k][i] = mul2(bu2, bq[st][i]);
                        }
                    }
#pragma unroll
                for (int st = 0; st < 4; st++)
#pragma unroll
                    for (int k = 0; k < K; k++) {
                        float2 acc2 = make_float2(0.f, 0.f);
#pragma unroll
                        for (int i = 0; i < NP2; i++) {
                            S.h2[k][i] = fma2(an[st][k][i], S.h2[k][i], bn[st][k][i]);
                            if constexpr (kFull) acc2 = fma2(cq[st][i], S.h2[k][i], acc2);
                        }
                        acc[k][st] = acc2.x + acc2.y;
                    }
            } else {
#pragma unroll
                for (int st = 0; st < 4; st++)
#pragma unroll
                    for (int k = 0; k < K; k++) {
                        acc[k][st] = 0.f;
#pragma unroll
                        for (int i = 0; i < NPL; i++) {
                            const float an = Dec::make(x[st][k].x * lo_hi(A2[k][i / 2], i));
                            const float bv = x[st][k].y * lo_hi(bq[st][i / 2], i);
                            float& hi = lo_hi_ref(S.h2[k][i / 2], i);
                            if constexpr (kAcc) {
                                S.dlt[k][i] += fmaf(an, hi, bv);
                                hi = S.hhi[k][i] + (S.dlt[k][i] + S.hlo[k][i]);
                            } else {
                                hi = Dec::step(an, hi, bv);
                            }
                            if constexpr (kFull) acc[k][st] = fmaf(lo_hi(cq[st][i / 2], i), hi, acc[k][st]);
                        }
                    }
            }
            if constexpr (kFull) {
#pragma unroll
                for (int k = 0; k < K; k++)
                    tl.p[warp][k][tg / 4][lane] = make_float4(acc[k][0], acc[k][1], acc[k][2], acc[k][3]);
            }
        }
        if constexpr (kAcc) {
            // re-anchor: (hhi, hlo) <- the exact sum of the pair and dlt
#pragma unroll
            for (int k = 0; k < K; k++)
#pragma unroll
                for (int i = 0; i < NPL; i++) {
                    two_sum(S.hhi[k][i], S.dlt[k][i] + S.hlo[k][i], S.hhi[k][i], S.hlo[k][i]);
                    S.dlt[k][i] = 0.f;
                }
        }
        if constexpr (kFull) {
            __syncwarp();
            // C. epilogue: y = (sum of the G partials + D*u) * silu(z)
#pragma unroll
            for (int q = 0; q < PV; q++) {
                // in pairs of steps: y = D*u + the G partials, then times silu(z)
                float fu[V], yv[V];
                unpack<Tin>(ku[q], fu);
                float2 y2[V / 2];
#pragma unroll
                for (int k = 0; k < V; k += 2)
                    y2[k / 2] = mul2(make_float2(fu[k], fu[k + 1]), make_float2(Dd[q], Dd[q]));
                const int pk = pc[q] % K, pg = pc[q] / K;
#pragma unroll
                for (int jj = 0; jj < G; jj++) {
#pragma unroll
                    for (int k = 0; k < V; k += 4) {
                        const float4 p4 = tl.p[warp][pk][(pt[q] + k) / 4][lane_of<G, K>(pg, jj)];
                        y2[k / 2] = add2(y2[k / 2], make_float2(p4.x, p4.y));
                        y2[k / 2 + 1] = add2(y2[k / 2 + 1], make_float2(p4.z, p4.w));
                    }
                }
                if (has_z) {
                    float fz[V];
                    unpack<Tin>(kz[q], fz);
#pragma unroll
                    for (int k = 0; k < V; k += 2) {
                        float2 s;
                        if constexpr (kAcc) {
                            s = make_float2(silu_acc<true>(fz[k]), silu_acc<true>(fz[k + 1]));
                        } else {
                            // z * rcp(1 + 2^(-z log2 e)), the SFU form
                            const float2 e = mul2(make_float2(fz[k], fz[k + 1]), make_float2(-kLog2e, -kLog2e));
                            const float2 den = add2(make_float2(ex2(e.x), ex2(e.y)), make_float2(1.f, 1.f));
                            s = mul2(make_float2(fz[k], fz[k + 1]), make_float2(rcp(den.x), rcp(den.y)));
                        }
                        y2[k / 2] = mul2(y2[k / 2], s);
                    }
                }
#pragma unroll
                for (int k = 0; k < V; k += 2) {
                    yv[k] = y2[k / 2].x;
                    yv[k + 1] = y2[k / 2].y;
                }
                if (chan_ok[q]) {
                    Tout* yrow = y_base + (b * a.dim + d_warp0 + pc[q]) * L;
                    const int64_t tt = t0 + pt[q];
                    if (rev) {
                        // steps tt .. tt+V-1 are positions L-1-tt down to L-tt-V
                        if (tt + V <= te) {
                            float yr[V];
#pragma unroll
                            for (int k = 0; k < V; k++) yr[k] = yv[V - 1 - k];
                            store_steps<Tout, V>(yrow + (L - tt - V), yr);
                        } else {
#pragma unroll
                            for (int k = 0; k < V; k++)
                                if (tt + k < te) yrow[L - 1 - (tt + k)] = from_f32<Tout>(yv[k]);
                        }
                    } else if (kVec && tt + V <= te) {
                        store_steps<Tout, V>(yrow + tt, yv);
                    } else {
#pragma unroll
                        for (int k = 0; k < V; k++)
                            if (tt + k < te) yrow[tt + k] = from_f32<Tout>(yv[k]);
                    }
                }
            }
        }
        (void)ku; (void)kz;
    }
    if constexpr (kTma) {
        if (!ok && threadIdx.x == 0) {
            // record, then let the copy still in flight land before leaving
            atomicExch(&g_prefill_status, __LINE__);
            (void)tc::mbar_wait(tl.full, *phase & 1u, kTmaWaitLimit);
        }
    }
    // the next pass (or caller) reuses the tiles: all warps must be done with them
    __syncthreads();
    return ok;
}

// The lane's A values (pairs) and states initialised to h[k] (anchor h, nothing
// since), for its K channels dR[k] (valid while okR[k]).
template <int N, int G, int K>
__device__ __forceinline__ void lane_init(const ScanArgs& a, const int64_t* dR, const bool* okR, int j,
                                          A2Arr<N, G, K>& A2, LaneStateT<N, G, K>& S, const float (*h)[N / G]) {
    constexpr int NPL = N / G;
#pragma unroll
    for (int k = 0; k < K; k++) {
#pragma unroll
        for (int i = 0; i < LaneState<K, NPL>::NP2; i++) {
            A2[k][i] = make_float2(0.f, 0.f);
            S.h2[k][i] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < NPL; i++) {
            lo_hi_ref(A2[k][i / 2], i) = okR[k] ? a.A[dR[k] * N + j * NPL + i] : 0.f;
            const float h0 = h ? h[k][i] : 0.f;
            lo_hi_ref(S.h2[k][i / 2], i) = h0;
            S.hhi[k][i] = h0;
            S.hlo[k][i] = 0.f;
            S.dlt[k][i] = 0.f;
        }
        S.sdt[k] = 0.f;
        S.sdt_c[k] = 0.f;
    }
}

// State i of channel k of the lane (the anchored pair's sum on the fp32 path).
template <int N, int G, int K, typename Tin>
__device__ __forceinline__ float lane_state(const LaneStateT<N, G, K>& S, int k, int i) {
    if constexpr (sizeof(Tin) == 4) return S.hhi[k][i] + S.hlo[k][i];
    else return lo_hi(S.h2[k][i / 2], i);
}

// Two launch forms of the time-serial kernel.
//   Plain (bal_ctas == 0): CTA (x, y) walks channel group x of batch row y over all
//     L steps. Every CTA does the same work, so the kernel takes as long as the SM
//     holding the most CTAs: at (4, 5120, 4096) 640 CTAs leave 48 SMs with five and
//     100 with four, and the kernel ran as long as with five on every SM.
//   Work-balanced (bal_ctas = P > 0, a multiple of the SM count, at most the number
//     of channel groups U): the U (channel group, batch row) units, each of
//     nch = ceil(L / T) chunks, are laid end to end and cut into P equal runs at
//     chunk boundaries. A run of at least nch chunks is the tail of one unit (from
//     chunk kF), any whole units, and the head of the last (to chunk kLe). The CTA
//     takes its run by an atomic ticket, walks the head first (from h0) and
//     publishes the state at its end in its workspace slot, then the whole units,
//     then the tail, whose starting state is the previous ticket's published slot.
//     That CTA published after kF chunks of work and this one reaches its tail after
//     kLe + (whole units) nch >= kF chunks, so at equal speed the wait is free; a
//     CTA only waits on an earlier ticket, whose CTA is running, so the wait always
//     ends. Each wait is bounded; on expiry the kernel records the line in
//     g_prefill_status and continues from a zero state (y is then unspecified).
//   Workspace: [4] ticket counter (zeroed by the host), flags[P] at 16, then P state
//   slots of (channels per CTA) x N floats.
template <int N, int G, typename Tin, typename Tout, bool kVec, bool kTma, bool kRev = false>
// at most 128 registers (4 CTAs per SM): measured ~1% faster than unbounded
__global__ void __launch_bounds__(kThreads, 4) serial_scan_kernel(ScanArgs a, const __grid_constant__ ScanMaps maps) {
    constexpr int K = 1;
    using Cfg = SerialCfg<N, G, Tin, K>;
    constexpr int NPL = Cfg::NPL, CPW = Cfg::CPW, kT = Cfg::kT;
    constexpr int CPC = kWarps * CPW;
    __shared__ __align__(16) float s_bc[2][kT][2 * N];
    __shared__ __align__(16) float s_db[kWarps][CPW / K][Cfg::DBS];
    __shared__ __align__(16) float4 s_p[kWarps][K][kT / 4][Cfg::PS];
    __shared__ __align__(1024) unsigned char s_stage[kTma ? StageGeom<N, G, Tin, K>::BYTES : 16];
    __shared__ __align__(8) uint64_t s_full;
    __shared__ uint32_t s_ticket;
    const bool bal = a.bal_ctas > 0;
    uint32_t phase = 0;
    if (threadIdx.x == 0) {
        if (kTma) {
            tc::mbar_init(&s_full, 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        if (bal) s_ticket = atomicAdd(reinterpret_cast<uint32_t*>(static_cast<char*>(a.workspace) + 4), 1u);
    }
    __syncthreads();

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int p = lane_grp<G, K>(lane), j = lane_sgrp<G, K>(lane);
    const int64_t L = a.seqlen;
    const int64_t groups = (a.dim + CPC - 1) / CPC;
    const int64_t nch = (L + kT - 1) / kT;
    uint32_t* flags = nullptr;
    float* slots = nullptr;
    int64_t c = 0, uF, kF, uL, kLe;
    if (bal) {
        const int64_t P = a.bal_ctas, W = groups * a.batch * nch;
        const int64_t Wq = W / P, Wr = W % P;
        auto cut = [&](int64_t i) { return i * Wq + (i * Wr) / P; };
        c = s_ticket;
        const int64_t w0 = cut(c), w1 = cut(c + 1);
        uF = w0 / nch; kF = w0 % nch;
        uL = (w1 - 1) / nch; kLe = w1 - uL * nch;
        flags = reinterpret_cast<uint32_t*>(static_cast<char*>(a.workspace) + kSerialBalFlags);
        slots = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + serial_bal_slots_offset(P));
    } else {
        uF = uL = (int64_t)blockIdx.y * groups + blockIdx.x;
        kF = 0; kLe = nch;
    }
    // pieces in order: the head of unit uL, whole units uF+1 .. uL-1, the tail of uF
    // (one piece when the run lies in one unit)
    const int64_t n_pieces = uF == uL ? 1 : uL - uF + 1;
    for (int64_t pi = 0; pi < n_pieces; pi++) {
        int64_t u, kb, ke;
        if (n_pieces == 1) { u = uF; kb = kF; ke = kLe; }
        else if (pi == 0) { u = uL; kb = 0; ke = kLe; }
        else if (pi + 1 < n_pieces) { u = uF + pi; kb = 0; ke = nch; }
        else { u = uF; kb = kF; ke = nch; }
        const int64_t b = u / groups, grp = u % groups;
        const int64_t tb = kb * kT, te = min(L, ke * kT);
        const bool dep = bal && kb > 0, pub = bal && ke < nch;
        const int64_t d_warp0 = (grp * kWarps + warp) * CPW;
        // starting state: h0 at step 0, else the previous ticket's published slot
        bool got = true;
        if (dep) {
            uint32_t spins = 0;
            while (ld_acquire(&flags[c - 1]) == 0 && spins < a.spin_limit) {
                ++spins;
                __nanosleep(64);
            }
            got = ld_acquire(&flags[c - 1]) != 0;
            if (!got && threadIdx.x == 0) atomicExch(&g_prefill_status, __LINE__);
        }
        int64_t dR[K];
        bool okR[K];
        float h0[K][NPL];
#pragma unroll
        for (int k = 0; k < K; k++) {
            dR[k] = d_warp0 + p * K + k;
            okR[k] = dR[k] < a.dim;
            const int slot_ch = warp * CPW + p * K + k;
#pragma unroll
            for (int i = 0; i < NPL; i++) {
                float v = 0.f;
                if (dep) v = got ? __ldcg(slots + ((c - 1) * CPC + slot_ch) * N + j * NPL + i) : 0.f;
                else if (okR[k] && a.h0) v = a.h0[(b * a.dim + dR[k]) * N + j * NPL + i];
                h0[k][i] = v;
            }
        }
        A2Arr<N, G, K> A2;
        LaneStateT<N, G, K> S;
        lane_init<N, G, K>(a, dR, okR, j, A2, S, h0);
        const Tiles<N, G, Tin, K> tl{s_bc, s_db, s_p, s_stage, &s_full, &maps, grp * CPC};
        if (!serial_pass<N, G, K, Tin, Tout, kVec, true, kTma, kRev>(a, b, d_warp0, tb, te, A2, S, tl, &phase))
            return;
        if (te == L && a.h_last) {
#pragma unroll
            for (int k = 0; k < K; k++)
                if (okR[k]) {
#pragma unroll
                    for (int i = 0; i < NPL; i++)
                        a.h_last[(b * a.dim + dR[k]) * N + j * NPL + i] = lane_state<N, G, K, Tin>(S, k, i);
                }
        }
        if (pub) {
            const int slot_ch0 = warp * CPW + p * K;
#pragma unroll
            for (int k = 0; k < K; k++)
#pragma unroll
                for (int i = 0; i < NPL; i++)
                    slots[(c * CPC + slot_ch0 + k) * N + j * NPL + i] = lane_state<N, G, K, Tin>(S, k, i);
            __threadfence();
            __syncthreads();
            // (test hook: ticket drop_segment withholds its publication)
            if (threadIdx.x == 0 && c != a.drop_segment) st_release(&flags[c], 1u);
        }
    }
}

// ---------------------------------------------------------------------------
// Look-back kernel: time cut into segments of seg_len steps; one CTA per
// (channel group, segment), taken in the order of an atomic ticket, segment-major,
// so every segment a CTA waits on belongs to a CTA that has already started.
// A CTA (1) runs the aggregate pass over its segment from a zero state, giving
// each state's map over the segment: decay P = exp(A * sum dt) and offset H;
// (2) publishes (P, H) with flag AGG; (3) walks back over earlier segments until
// it meets a published inclusive prefix I (the state at that segment's end) and
// applies the maps of the segments in between to it, in order, which gives its
// carry (the same operations as a serial chain, so the result is deterministic); (4) publishes its own inclusive
// prefix with flag INCL; (5) runs the full pass from the carry. The last segment
// publishes nothing and skips (1). Every wait is bounded: on expiry the kernel
// records SSM_ERR_LOOKBACK_TIMEOUT in the workspace status word, continues with
// what it has (publishing so that later segments finish too) and the output is
// then unspecified.
// Workspace (zeroed by the host on the stream): [0] int32 status, [1] uint32
// ticket, [2..3] pad; then per (channel, segment) a descriptor: uint32 flag[N]
// (flag[j] covers the states of lane j of the channel's lane group), float P[N],
// H[N], I[N] (P in the Decay representation: the factor, or factor - 1 for fp32
// inputs). Published values are never rewritten.
// ---------------------------------------------------------------------------
constexpr uint32_t kFlagAgg = 1, kFlagIncl = 2;
constexpr int kErrLookbackTimeout = -7;

template <int N>
struct LbDesc {
    uint32_t flag[N];
    float P[N];
    float H[N];
    float I[N];
};

// kLookbackCtasPerSM CTAs per SM at least (the host plans the segments for exactly
// that many resident CTAs: none may wait for a slot)
template <int N, int G, typename Tin, typename Tout, bool kVec, bool kTma, bool kRev = false>
__global__ void __launch_bounds__(kThreads, kLookbackCtasPerSM)
    serial_lookback_kernel(ScanArgs a, const __grid_constant__ ScanMaps maps) {
    constexpr int K = max_k<N, G, Tin>();
    using Cfg = SerialCfg<N, G, Tin, K>;
    constexpr int NPL = Cfg::NPL, CPW = Cfg::CPW, kT = Cfg::kT;
    constexpr bool kAcc = sizeof(Tin) == 4;
    using Dec = Decay<kAcc>;
    __shared__ __align__(16) float s_bc[2][kT][2 * N];
    __shared__ __align__(16) float s_db[kWarps][CPW / K][Cfg::DBS];
    __shared__ __align__(16) float4 s_p[kWarps][K][kT / 4][Cfg::PS];
    __shared__ uint32_t s_ticket;
    __shared__ __align__(1024) unsigned char s_stage[kTma ? StageGeom<N, G, Tin, K>::BYTES : 16];
    __shared__ __align__(8) uint64_t s_full;
    uint32_t phase = 0;

    int32_t* status = static_cast<int32_t*>(a.workspace);
    uint32_t* ticket_ctr = reinterpret_cast<uint32_t*>(status + 1);
    LbDesc<N>* desc = reinterpret_cast<LbDesc<N>*>(static_cast<char*>(a.workspace) + 16);

    if (threadIdx.x == 0) {
        s_ticket = atomicAdd(ticket_ctr, 1u);
        if (kTma) {
            tc::mbar_init(&s_full, 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
    }
    __syncthreads();
    const int64_t ch_per_cta = (int64_t)kWarps * CPW;
    const int64_t groups = (a.dim + ch_per_cta - 1) / ch_per_cta;
    const int64_t per_seg = groups * a.batch;
    const int64_t tk = s_ticket;
    const int64_t seg = tk / per_seg;
    const int64_t rem = tk % per_seg;
    const int64_t b = rem / groups;
    const int64_t grp = rem % groups;
    const int64_t ts = seg * a.seg_len;
    const int64_t te = min(a.seqlen, ts + a.seg_len);
    const bool last = seg + 1 == a.n_seg;
    const bool publish = !last && seg != a.drop_segment;

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t d_warp0 = (grp * kWarps + warp) * CPW;
    const Tiles<N, G, Tin, K> tl{s_bc, s_db, s_p, s_stage, &s_full, &maps, grp * kWarps * CPW};
    const int p = lane_grp<G, K>(lane), j = lane_sgrp<G, K>(lane);
    int64_t dR[K], ch[K];
    bool okR[K];
#pragma unroll
    for (int k = 0; k < K; k++) {
        dR[k] = d_warp0 + p * K + k;
        okR[k] = dR[k] < a.dim;
        ch[k] = b * a.dim + dR[k];
    }
    A2Arr<N, G, K> A2;
    LaneStateT<N, G, K> S;

    // (1) the segment's map from a zero state
    lane_init<N, G, K>(a, dR, okR, j, A2, S, nullptr);
    float aggP[K][NPL], aggH[K][NPL];
#pragma unroll
    for (int k = 0; k < K; k++)
#pragma unroll
        for (int i = 0; i < NPL; i++) { aggP[k][i] = Dec::one(); aggH[k][i] = 0.f; }
    if (!last) {
        if (!serial_pass<N, G, K, Tin, Tout, kVec, false, kTma, kRev>(a, b, d_warp0, ts, te, A2, S, tl, &phase)) {
            // a failed copy wait: record it where the look-back reports, publish nothing
            // (later segments time out on their bounded waits and finish) and leave
            if (threadIdx.x == 0) atomicExch(status, kErrLookbackTimeout);
            return;
        }
#pragma unroll
        for (int k = 0; k < K; k++)
#pragma unroll
            for (int i = 0; i < NPL; i++) {
                aggP[k][i] = Dec::make(S.sdt[k] * lo_hi(A2[k][i / 2], i));
                aggH[k][i] = lane_state<N, G, K, Tin>(S, k, i);
            }
    }
    // (2)-(4) per lane, for each of its channels' states
    float carry[K][NPL];
#pragma unroll
    for (int k = 0; k < K; k++) {
#pragma unroll
        for (int i = 0; i < NPL; i++) carry[k][i] = 0.f;
        if (!okR[k]) continue;
        LbDesc<N>* mine = desc + ch[k] * a.n_seg + seg;
        if (seg == 0) {
#pragma unroll
            for (int i = 0; i < NPL; i++) carry[k][i] = a.h0 ? a.h0[ch[k] * N + j * NPL + i] : 0.f;
        } else {
            if (publish) {
#pragma unroll
                for (int i = 0; i < NPL; i++) {
                    mine->P[j * NPL + i] = aggP[k][i];
                    mine->H[j * NPL + i] = aggH[k][i];
                }
                st_release(&mine->flag[j], kFlagAgg);
            }
            // Walk back to the nearest segment whose inclusive prefix (the state at its
            // end) is published, then apply the maps of the segments after it in
            // order, h <- P h + H: the very operations a serial chain of inclusive
            // prefixes performs, so the carry is the same bits whichever prefix the
            // walk meets first (composing the maps backwards instead would round in
            // an order that depends on timing).
            int64_t found = -1;
            bool timed_out = false;
            for (int64_t s = seg - 1; s >= 0; s--) {
                const LbDesc<N>* pd = desc + ch[k] * a.n_seg + s;
                uint32_t f = ld_acquire(&pd->flag[j]);
                uint32_t spins = 0;
                while (f == 0 && spins < a.spin_limit) {
                    ++spins;
                    __nanosleep(64);
                    f = ld_acquire(&pd->flag[j]);
                }
                if (f == 0) {
                    timed_out = true;
                    break;
                }
                if (f == kFlagIncl) {
                    found = s;
                    break;
                }
            }
            if (!timed_out && found >= 0) {
                const LbDesc<N>* pf = desc + ch[k] * a.n_seg + found;
#pragma unroll
                for (int i = 0; i < NPL; i++) carry[k][i] = __ldcg(&pf->I[j * NPL + i]);
                for (int64_t s = found + 1; s < seg; s++) {
                    const LbDesc<N>* pd = desc + ch[k] * a.n_seg + s;
#pragma unroll
                    for (int i = 0; i < NPL; i++)
                        carry[k][i] = Dec::step(__ldcg(&pd->P[j * NPL + i]), carry[k][i], __ldcg(&pd->H[j * NPL + i]));
                }
            }
            if (timed_out) atomicExch(status, kErrLookbackTimeout);
        }
        // (4) the inclusive prefix: the state at this segment's end. On a timeout it
        // is still published (with the wrong carry) so that later segments finish.
        if (publish) {
#pragma unroll
            for (int i = 0; i < NPL; i++) mine->I[j * NPL + i] = Dec::step(aggP[k][i], carry[k][i], aggH[k][i]);
            st_release(&mine->flag[j], kFlagIncl);
        }
    }
    // (5) the full pass from the carry
    lane_init<N, G, K>(a, dR, okR, j, A2, S, carry);
    if (!serial_pass<N, G, K, Tin, Tout, kVec, true, kTma, kRev>(a, b, d_warp0, ts, te, A2, S, tl, &phase)) {
        if (threadIdx.x == 0) atomicExch(status, kErrLookbackTimeout);
        return;
    }
    if (last && a.h_last) {
#pragma unroll
        for (int k = 0; k < K; k++)
            if (okR[k]) {
#pragma unroll
                for (int i = 0; i < NPL; i++) a.h_last[ch[k] * N + j * NPL + i] = lane_state<N, G, K, Tin>(S, k, i);
            }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// bf16 (L, rows, batch) view with (kT, box_rows, 1) boxes (64-byte swizzled when
// sw64, see StageGeom): rows beyond
// `rows` (a CTA's last channels) and steps beyond L read as zeros
bool encode_bf16(CUtensorMap* map, const void* base, int64_t L, int64_t rows, int64_t batch, int kT, int box_rows,
                 bool sw64) {
    auto fn = encode_fn();
    if (!fn || !base) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)L, (cuuint64_t)rows, (cuuint64_t)batch};
    const cuuint64_t strides[2] = {(cuuint64_t)(L * 2), (cuuint64_t)(L * rows * 2)};
    const cuuint32_t box[3] = {(cuuint32_t)kT, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The bulk-copy input path is taken for bf16 inputs whose rows are 16-byte
// aligned (a.vec) when the tensor maps encode; `maps` is left zero otherwise.
template <int N, int G, int K, typename Tin>
bool make_maps(const ScanArgs& a, ScanMaps* maps) {
    memset(maps, 0, sizeof(*maps));
    if constexpr (sizeof(Tin) != 2) {
        return false;
    } else {
        using Cfg = SerialCfg<N, G, Tin, K>;
        constexpr int CPC = StageGeom<N, G, Tin, K>::CPC;
        if (!a.vec || a.seqlen <= 0 || a.seqlen >= ((int64_t)1 << 31) || a.dim >= ((int64_t)1 << 31)) return false;
        constexpr bool sw = StageGeom<N, G, Tin, K>::kSw64;
        return encode_bf16(&maps->u, a.u, a.seqlen, a.dim, a.batch, Cfg::kT, CPC, sw) &&
               encode_bf16(&maps->d, a.delta, a.seqlen, a.dim, a.batch, Cfg::kT, CPC, sw) &&
               (!a.z || encode_bf16(&maps->z, a.z, a.seqlen, a.dim, a.batch, Cfg::kT, CPC, sw)) &&
               encode_bf16(&maps->B, a.B, a.seqlen, N, a.batch, Cfg::kT, N, sw) &&
               encode_bf16(&maps->C, a.C, a.seqlen, N, a.batch, Cfg::kT, N, sw);
    }
}

template <int N, int G, typename Tin, typename Tout>
cudaError_t launch_serial(const ScanArgs& a_in, cudaStream_t s) {
    using Cfg = SerialCfg<N, G, Tin, 1>;
    if (a_in.batch == 0 || a_in.dim == 0) return cudaSuccess;
    ScanArgs a = a_in;
    a.bal_ctas = 0;
    const int64_t ch_per_cta = (int64_t)kWarps * Cfg::CPW;
    const int64_t groups = (a.dim + ch_per_cta - 1) / ch_per_cta;
    const int64_t units = groups * a.batch;
    ScanMaps maps;
    memset(&maps, 0, sizeof(maps));
    using KernelFn = void (*)(ScanArgs, ScanMaps);
    KernelFn k = nullptr;
    if constexpr (sizeof(Tin) == 2) {
        if (make_maps<N, G, 1, Tin>(a, &maps))
            k = a.reverse ? serial_scan_kernel<N, G, Tin, Tout, true, true, true>
                          : serial_scan_kernel<N, G, Tin, Tout, true, true>;
    }
    if (!k) {
        if (a.reverse) return cudaErrorInvalidValue;   // the reversed walk needs the bulk-copy path
        k = a.vec ? serial_scan_kernel<N, G, Tin, Tout, true, false> : serial_scan_kernel<N, G, Tin, Tout, false, false>;
    }
    // the work-balanced form when a workspace is given and the units do not already
    // divide evenly over the SMs: a multiple of the SM count, all CTAs resident
    int64_t P = 0;
    if (a.workspace && a.seqlen > 0) {
        int dev = 0, sms = 0, occ = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kThreads, 0) == cudaSuccess && sms > 0 &&
            units >= sms) {
            P = std::min<int64_t>((int64_t)occ * sms, (units / sms) * sms);
            if (P >= units || serial_bal_workspace_bytes(P, N, G) > a.workspace_bytes) P = 0;
        }
    }
    if (P > 0) {
        a.bal_ctas = P;
        const cudaError_t e = cudaMemsetAsync(a.workspace, 0, serial_bal_slots_offset(P), s);
        if (e != cudaSuccess) return e;
        k<<<(unsigned)P, kThreads, 0, s>>>(a, maps);
    } else {
        if (groups > 0x7fffffff || a.batch > 65535) return cudaErrorInvalidValue;
        k<<<dim3((unsigned)groups, (unsigned)a.batch), kThreads, 0, s>>>(a, maps);
    }
    return cudaGetLastError();
}

template <int N, int G, typename Tin, typename Tout>
cudaError_t launch_lookback(const ScanArgs& a, cudaStream_t s) {
    constexpr int K = max_k<N, G, Tin>();
    using Cfg = SerialCfg<N, G, Tin, K>;
    if (a.batch == 0 || a.dim == 0) return cudaSuccess;
    const int64_t ch_per_cta = (int64_t)kWarps * Cfg::CPW;
    const int64_t ctas = ((a.dim + ch_per_cta - 1) / ch_per_cta) * a.batch * a.n_seg;
    if (ctas > ((int64_t)1 << 31) - 1) return cudaErrorInvalidValue;
    ScanMaps maps;
    bool launched = false;
    if constexpr (sizeof(Tin) == 2) {
        if (make_maps<N, G, K, Tin>(a, &maps)) {
            if (a.reverse) serial_lookback_kernel<N, G, Tin, Tout, true, true, true><<<(unsigned)ctas, kThreads, 0, s>>>(a, maps);
            else serial_lookback_kernel<N, G, Tin, Tout, true, true><<<(unsigned)ctas, kThreads, 0, s>>>(a, maps);
            launched = true;
        }
    } else {
        memset(&maps, 0, sizeof(maps));
    }
    if (launched) {
    } else if (a.reverse) {
        return cudaErrorInvalidValue;   // the reversed walk needs the bulk-copy path
    } else if (a.vec) serial_lookback_kernel<N, G, Tin, Tout, true, false><<<(unsigned)ctas, kThreads, 0, s>>>(a, maps);
    else serial_lookback_kernel<N, G, Tin, Tout, false, false><<<(unsigned)ctas, kThreads, 0, s>>>(a, maps);
    return cudaGetLastError();
}

// lanes per channel: 4 for N >= 4 (2 also built for N = 16), else N
template <int N, typename Tin, typename Tout, bool kLB>
cudaError_t launch_g(const ScanArgs& a, int G, cudaStream_t s) {
    if constexpr (N >= 4) {
        if constexpr (N == 16) {
            if (G == 2) return kLB ? launch_lookback<N, 2, Tin, Tout>(a, s) : launch_serial<N, 2, Tin, Tout>(a, s);
        }
        return kLB ? launch_lookback<N, 4, Tin, Tout>(a, s) : launch_serial<N, 4, Tin, Tout>(a, s);
    } else {
        return kLB ? launch_lookback<N, N, Tin, Tout>(a, s) : launch_serial<N, N, Tin, Tout>(a, s);
    }
}

template <typename Tin, typename Tout, bool kLB>
cudaError_t launch_n(const ScanArgs& a, int G, cudaStream_t s) {
    switch (a.dstate) {
        case 1: return launch_g<1, Tin, Tout, kLB>(a, G, s);
        case 2: return launch_g<2, Tin, Tout, kLB>(a, G, s);
        case 4: return launch_g<4, Tin, Tout, kLB>(a, G, s);
        case 8: return launch_g<8, Tin, Tout, kLB>(a, G, s);
        case 16: return launch_g<16, Tin, Tout, kLB>(a, G, s);
    }
    return cudaErrorInvalidValue;
}

template <bool kLB>
cudaError_t dispatch(const ScanArgs& a, int G, cudaStream_t s) {
    if (a.in_dtype == kBF16)
        return a.out_dtype == kBF16 ? launch_n<__nv_bfloat16, __nv_bfloat16, kLB>(a, G, s)
                                    : launch_n<__nv_bfloat16, float, kLB>(a, G, s);
    return a.out_dtype == kBF16 ? launch_n<float, __nv_bfloat16, kLB>(a, G, s)
                                : launch_n<float, float, kLB>(a, G, s);
}

}  // namespace

int lookback_channels_per_cta(int dstate, int lanes_per_channel, int in_dtype) {
    const int npl = dstate / lanes_per_channel;
    const int k = (in_dtype == kBF16 && npl >= 2 && npl <= 4) ? 2 : 1;   // max_k()
    return kWarps * 32 * k / lanes_per_channel;
}

cudaError_t launch_scan_thread(const ScanArgs& a, int lanes_per_channel, cudaStream_t s) {
    return dispatch<false>(a, lanes_per_channel, s);
}

cudaError_t launch_scan_serial_lookback(const ScanArgs& a, int lanes_per_channel, cudaStream_t s) {
    return dispatch<true>(a, lanes_per_channel, s);
}

cudaError_t prefill_status(int* line, bool clear, cudaStream_t s) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(line, g_prefill_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && clear && *line != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_prefill_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

int serial_channels_per_cta(int dstate, int lanes_per_channel) { return kWarps * 32 / lanes_per_channel; }

size_t serial_bal_workspace_bytes(int64_t ctas, int dstate, int lanes_per_channel) {
    return serial_bal_slots_offset(ctas) +
           (size_t)ctas * (size_t)serial_channels_per_cta(dstate, lanes_per_channel) * (size_t)dstate * sizeof(float);
}

size_t lookback_workspace_bytes(int64_t batch, int64_t dim, int dstate, int64_t n_seg) {
    return 16 + (size_t)batch * (size_t)dim * (size_t)n_seg * sizeof(LbDesc<1>) * (size_t)dstate;
}

}  // namespace ssm
