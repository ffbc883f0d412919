// kernels_ssd.cu -- the Mamba-2 state-space-duality (SSD) scan on the tcgen05
// tensor cores.
//
// Model (Mamba SSM complete guide, section 6 "Mamba 2": multi-head SSM with a
// scalar A per head, computed by chunks -- matrix products inside a chunk, the
// recurrence carried from chunk to chunk). Per batch row b, head h (group g =
// h / (H / G)), step t, head channel p and state n:
//     dt_t   = softplus(dt_raw[b,t,h] + dt_bias[h])
//     H_t    = exp(dt_t A_h) H_{t-1} + dt_t x[b,t,h,:] (x) B[b,t,g,:]      (P x N)
//     y[t,p] = sum_n C[b,t,g,n] H_t[p,n] + D_h x[t,p],   y *= silu(z[t,p])
//
// Chunked form for a chunk of Q = 128 steps starting from state H0, with
// cs_t = sum_{k<=t} dt_k A_h (inclusive, within the chunk):
//     S      = C B^T                                          (Q x Q, over n)
//     M[t,s] = S[t,s] exp(cs_t - cs_s) dt_s  for s <= t, else 0
//     y      = M x + diag(exp(cs)) C H0^T + D x
//     H_end  = exp(cs_end) H0 + (w o x)^T B,   w_s = exp(cs_end - cs_s) dt_s
// Four tensor-core products per chunk, each M = 128 with an fp32 accumulator
// in tensor memory:
//     G1  S     = C  . B^T      A = C  (t x n, K-major)   B = B   (s x n, K-major)
//     G2  Yi    = M  . x        A = M  (t x s, K-major)   B = x   (s x p, MN-major)
//     G3  Ye    = C  . H0^T     A = C                      B = H0^T (n x p, MN-major)
//     G4  H^T  += B^T . (w o x) A = B^T (n x s, MN-major)  B = w o x (s x p, MN-major)
// then y = Yi + exp(cs_t) Ye + D x. The state H^T (n x p, fp32) stays in tensor
// memory for the whole sequence; it is rescaled by exp(cs_end) in place before
// G4 accumulates into it.
//
// Precision. x, B and C are bf16 inputs, exact as tensor-core operands. The three
// computed operands M, H0 and w o x are fp32 values; each is split into a bf16
// high part and a bf16 remainder (v = hi + lo to about 2^-17 relative) and
// multiplied as two products, so the tensor-core results carry fp32-like
// accuracy. With plain bf16 rounding the state's relative error of 2^-9 per
// chunk accumulates over its memory and leaves y far outside a 2e-3 bound.
//
// One CTA per (b, h), walking the chunks in order: sixteen compute warps (warp w
// reaches tensor-memory lanes 32 (w % 4) .. +31 and works on column quarter w / 4)
// and one control warp.
// Tensor memory (256 columns): S and then Ye in [0, 128), Yi in [128, 192),
// H^T in [192, 256). The tiles TMA moves (C, B, x, z in; y out) are 128-row tiles
// of 128-byte rows with 128-byte swizzling (one box per 64 columns); the tiles
// the threads compute (M, w o x, H) use the unswizzled core-matrix layout with
// stride_r = 128 B and stride_c = 2048 B, so 16-byte chunk (row r, column group
// j) sits at j * 2048 + r * 16 (tcgen05.cuh describes both).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <string.h>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace ssm {

__device__ int g_ssd_status;   // 0, or the source line of a wait that ran out of budget

namespace {

constexpr int kQ = 128;               // chunk length (steps)
constexpr int kP = 64;                // head channels
constexpr int kCompute = 512;       // sixteen compute warps
constexpr int kCtl = kCompute / 32; // the control warp: TMA copies and MMA issue
constexpr int kParts = kCompute / 128;   // column parts: warps per tensor-memory lane quarter
constexpr int kPc = kP / kParts;         // head channels (state / output columns) per warp: 16
constexpr int kSc = kQ / kParts;         // columns of S / M per warp: 32
constexpr int kThreads = kCompute + 32;
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr uint32_t kStrideC = 2048;   // bytes between column groups of a 128-row tile
// tensor-memory columns
constexpr uint32_t kColS = 0, kColYi = 128, kColYe = 192, kColH = 256, kTmemCols = 512;

// Shared-memory map (bytes) for state width N. The K-major tiles come first so
// that every descriptor reach stays inside the allocation. With N = 64 the
// inputs of the next chunk (C, B, x) load into a second stage while the current
// chunk computes; with N = 128 there is room for one stage only.
//   M hi/lo  : 128 x 128 bf16 each (t x s)
//   stage k  : C (128 x N), B (128 x N), x (128 x 64), swizzled, 64 columns per 16 KB atom
//   W hi/lo  : 128 x 64 each (s x p)
//   H hi/lo  : N x 64 each (n x p), column groups N * 16 bytes apart
//   z        : 128 x 64 (t x p), one stage; y is staged in the M area for its store
// G4 reads B^T as a 128-row operand (M = 128 along n); with N = 64 its rows
// 64..127 fall on whatever follows the B tile (inside the allocation) and only
// feed state rows 64..127, which nothing reads.
template <int kN>
struct Smem {
    static constexpr int kStages = kN == 64 ? 2 : 1;
    static constexpr uint32_t kTileM = 32768;
    static constexpr uint32_t kTileCB = (uint32_t)kN * 256;
    static constexpr uint32_t kTileX = 16384;
    static constexpr uint32_t kTileH = (uint32_t)kN * 128;
    static constexpr uint32_t kStrideH = (uint32_t)kN * 16;
    static constexpr uint32_t kMh = 0, kMl = kTileM;
    static constexpr uint32_t kStage0 = 2 * kTileM;
    static constexpr uint32_t kStageBytes = 2 * kTileCB + kTileX;
    static constexpr uint32_t kC = 0, kB = kTileCB, kX = 2 * kTileCB;   // within a stage
    static constexpr uint32_t kWh = kStage0 + kStages * kStageBytes, kWl = kWh + kTileX;
    static constexpr uint32_t kHh = kWl + kTileX, kHl = kHh + kTileH;
    static constexpr uint32_t kZ = kHl + kTileH;        // z of the current chunk (128 x 64)
    static constexpr uint32_t kBytes = kZ + kTileX;
    // y staged for its store: a bf16 y tile has the z tile's shape and swizzle and
    // is written over it in place (each thread reads its z chunks, then writes its
    // y chunks there), so the next M does not wait for the store; an fp32 y (twice
    // the size) goes to the M area, free once G2 is done
    static constexpr uint32_t kYbf16 = kZ, kYf32 = kMh;
    static_assert(kBytes <= 232448 - 3072, "shared memory (dynamic + up to 3 KB static)");
    static_assert(kStage0 + kB + 32768 <= kBytes, "G4 reach of stage 0");
    static_assert(kStage0 + (kStages - 1) * kStageBytes + kB + 32768 <= kBytes, "G4 reach of the last stage");
};

// Tensor maps of C, B, x, z and y: 3-D views (row elements, seqlen, batch) of the
// (batch, seqlen, row) arrays with 128-byte swizzling, box = 128 bytes x 128
// steps x 1 -- one 16 KB atom column of a tile; loads past seqlen arrive as zeros
// and stores past it are dropped.
struct SsdMaps {
    CUtensorMap c, b, x, z, y;
};

// offset of the 16-byte chunk (row r, column group j) in a tile
__device__ __forceinline__ uint32_t chunk_off(int r, int j) { return (uint32_t)j * kStrideC + (uint32_t)r * 16u; }

// fp32 -> (bf16 hi, bf16 lo) with hi + lo = v to ~2^-17 relative, packed in pairs
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    hi = *reinterpret_cast<uint32_t*>(&h);
    const float ha = __uint_as_float(hi << 16), hb = __uint_as_float(hi & 0xffff0000u);
    __nv_bfloat162 l = __floats2bfloat162_rn(a - ha, b - hb);
    lo = *reinterpret_cast<uint32_t*>(&l);
}
// split 8 consecutive values and store both 16-byte halves
__device__ __forceinline__ void split_store8(const float* v, unsigned char* hi_dst, unsigned char* lo_dst) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; i++) split2(v[2 * i], v[2 * i + 1], h[i], l[i]);
    *reinterpret_cast<uint4*>(hi_dst) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo_dst) = make_uint4(l[0], l[1], l[2], l[3]);
}
__device__ __forceinline__ void unpack8(uint4 v, float* out) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        out[2 * i] = __uint_as_float(w[i] << 16);
        out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// A CTA's run of (sequence, chunk) work (see ssd_chunk_scan_kernel): the tail of
// sequence uF from chunk kF, any whole sequences, the head of sequence uL up to
// chunk kLe; its ticket in the work-balanced launch.
struct SsdRun {
    int64_t uF, uL, kF, kLe, n_pieces;
    int64_t ticket;
};

// One sequence of a run: its index (batch row * nheads + head), batch row, head,
// group, A * log2(e), dt bias and D.
struct SsdSeq {
    int bh, b, h, g;
    float A2, bias, Dh;
};

// Barrier among the eight compute warps only (named barrier 1).
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }
// The same barrier, returning on every compute thread whether v held on any.
__device__ __forceinline__ bool compute_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, 512, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}
// Bounded wait that also gives up once another warp has raised the abort flag.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              uint32_t limit) {
    for (uint32_t i = 0; i < limit; i++) {
        if (tc::mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 63u && *abort_flag) return false;
    }
    return false;
}

// Roles. Warps 0-15 compute (warp w owns tensor-memory lanes 32 (w % 4) .. +31 and
// column quarter w / 4); warp 16 (the control warp) issues every TMA copy and
// every MMA. The two sides meet only through mbarriers, every wait bounded:
//   TMA -> all        s_load (inputs of a stage), s_zload (z)
//   MMA -> compute    s_bar[0] G1 done, s_bar[1] G3 + G4 done, s_bar[2] G2 done
//   compute -> ctl    s_ready[0] w o x and the rescaled state written,
//                     s_ready[1] M written, s_ready[2] chunk finished (y staged)
//   ctl -> compute    s_yfree: the previous y store has left the M area
template <int kN, bool kOutF32>
__global__ void __launch_bounds__(kThreads, 1)
    ssd_chunk_scan_kernel(const SsdArgs a, const __grid_constant__ SsdMaps m) {
    using S = Smem<kN>;
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ float s_cs2[2][kQ];   // cs_t * log2(e), by chunk parity
    __shared__ float s_dt[2][kQ];
    __shared__ float s_w[kQ];        // exp(cs_end - cs_t) dt_t
    __shared__ float s_wsum[4];
    __shared__ uint64_t s_bar[3];
    __shared__ uint64_t s_load[2];
    __shared__ uint64_t s_zload;
    __shared__ uint64_t s_ready[3];
    __shared__ uint64_t s_yfree;
    __shared__ uint64_t s_drain;     // products drained (failure path only)
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ SsdRun s_run;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int quad = warp & 3, part = warp >> 2;   // lane quarter, column part
    // the swizzled tiles need a 1024-byte aligned base
    if (tc::smem_u32(smem) & 1023u) {
        if (tid == 0) atomicExch(&g_ssd_status, __LINE__);
        return;
    }
    const int64_t H = a.nheads, L = a.seqlen, G = a.ngroups;
    const int64_t nchunks = (L + kQ - 1) / kQ;   // chunks per sequence
    // The CTA's run of (sequence, chunk) work, walked piece by piece (a piece: one
    // sequence's chunks [c0, c1)). Plain launch: sequence blockIdx.x, all its chunks.
    // Work-balanced launch (bal_ctas = P): the batch * nheads sequences laid end to
    // end and cut into P equal runs of at least nchunks chunks, taken by an atomic
    // ticket; a run is the head of its last sequence (from h0, the state at its end
    // then published in the ticket's workspace slot), any whole sequences, and the
    // tail of its first sequence (from the state the previous ticket published:
    // that CTA publishes after its head, which is shorter than this CTA's head plus
    // whole sequences, so at equal speed the wait is free, and a CTA only waits on
    // an earlier ticket, whose CTA is running). Each piece runs the chunk pipeline
    // below from its first chunk to its last (the pipeline drains between pieces);
    // the mbarrier phases follow a running chunk count v across pieces. The run is
    // kept in shared memory, read at piece boundaries only.
    const bool bal = a.bal_ctas > 0;
    if (tid == 0) {
        SsdRun r;
        r.ticket = 0;
        if (bal) {
            r.ticket = atomicAdd(reinterpret_cast<uint32_t*>(static_cast<char*>(a.workspace) + 4), 1u);
            const int64_t P = a.bal_ctas, W = a.batch * H * nchunks, Wq = W / P, Wr = W % P, t = r.ticket;
            const int64_t w0 = t * Wq + (t * Wr) / P, w1 = (t + 1) * Wq + ((t + 1) * Wr) / P;
            r.uF = w0 / nchunks; r.kF = w0 - r.uF * nchunks;
            r.uL = (w1 - 1) / nchunks; r.kLe = w1 - r.uL * nchunks;
        } else {
            r.uF = r.uL = blockIdx.x;
            r.kF = 0; r.kLe = nchunks;
        }
        r.n_pieces = r.uF == r.uL ? 1 : r.uL - r.uF + 1;
        s_run = r;
    }
    __syncthreads();
    const int n_pieces = (int)s_run.n_pieces;
    // piece pi: (sequence, first chunk, end chunk) -- the head of uL, whole
    // sequences uF+1 .. uL-1, the tail of uF
    auto piece = [&](int pi, int& u, int& c0, int& c1) {
        const SsdRun& r = s_run;
        if (r.n_pieces == 1) { u = (int)r.uF; c0 = (int)r.kF; c1 = (int)r.kLe; }
        else if (pi == 0) { u = (int)r.uL; c0 = 0; c1 = (int)r.kLe; }
        else if (pi + 1 < r.n_pieces) { u = (int)r.uF + pi; c0 = 0; c1 = (int)nchunks; }
        else { u = (int)r.uF; c0 = (int)r.kF; c1 = (int)nchunks; }
    };
    auto bal_flags = [&]() { return reinterpret_cast<uint32_t*>(static_cast<char*>(a.workspace) + 16); };
    auto bal_slots = [&]() {
        return reinterpret_cast<float*>(static_cast<char*>(a.workspace) + ssd_bal_slots_offset(a.bal_ctas));
    };
    // a piece's sequence (bh = batch row * nheads + head, below 2^31) and its
    // constants, made once per piece and passed to the helpers below
    auto make_seq = [&](int u) {
        SsdSeq q;
        q.bh = u; q.b = u / (int)H; q.h = u % (int)H; q.g = q.h / (int)(H / G);
        q.A2 = a.A[q.h] * kLog2e;
        q.bias = a.dt_bias ? a.dt_bias[q.h] : 0.f;
        q.Dh = a.D ? a.D[q.h] : 0.f;
        return q;
    };
    const __nv_bfloat16* zg = static_cast<const __nv_bfloat16*>(a.z);
    const unsigned short* dtb = static_cast<const unsigned short*>(a.dt);

    unsigned char* sMh = smem + S::kMh;
    unsigned char* sMl = smem + S::kMl;
    unsigned char* sWh = smem + S::kWh;
    unsigned char* sWl = smem + S::kWl;
    unsigned char* sHh = smem + S::kHh;
    unsigned char* sHl = smem + S::kHl;
    const uint32_t base = tc::smem_u32(smem);
    constexpr uint32_t kY = kOutF32 ? S::kYf32 : S::kYbf16;
    volatile int* abort_flag = &s_abort;
    const uint32_t wlim = a.wait_limit ? a.wait_limit : kWaitLimit;   // pipeline waits (not the drain)
    auto fail = [&](int line) {
        atomicExch(&g_ssd_status, line);
        *abort_flag = 1;
    };

    // ---- control-warp copies (whole warp, converged) ---------------------------------
    // Two stages (N = 64): C, B and x of chunk c on s_load[c & 1]. One stage
    // (N = 128): C and B on s_load[0], x on s_load[1]. Issue / consumption counts
    // per barrier let the failure path wait for exactly the phases in flight.
    uint32_t ld_issued0 = 0, ld_issued1 = 0, ld_seen0 = 0, ld_seen1 = 0, z_issued = 0, z_seen = 0;
    auto tma_cb = [&](const SsdSeq& q, int64_t c, int st, uint64_t* bar) {
        const int b = q.b, g = q.g;
        unsigned char* stg = smem + S::kStage0 + st * S::kStageBytes;
        constexpr int kJ = kN / 64;   // 64-column atoms of C and B
        if (lane < kJ)
            tc::tma_load_3d(stg + S::kC + lane * 16384, &m.c, (int)(g * kN) + 64 * lane, (int)(c * kQ), (int)b, bar);
        else if (lane < 2 * kJ)
            tc::tma_load_3d(stg + S::kB + (lane - kJ) * 16384, &m.b, (int)(g * kN) + 64 * (lane - kJ), (int)(c * kQ),
                            (int)b, bar);
    };
    auto tma_x = [&](const SsdSeq& q, int64_t c, int st, uint64_t* bar) {
        const int b = q.b, h = q.h;
        if (lane == 31)
            tc::tma_load_3d(smem + S::kStage0 + st * S::kStageBytes + S::kX, &m.x, (int)(h * kP), (int)(c * kQ),
                            (int)b, bar);
    };
    auto issue_stage = [&](const SsdSeq& q, int64_t c, int64_t v) {   // two stages: chunk c on stage v & 1
        const int st = (int)(v & 1);
        if (lane == 0) tc::mbar_expect_tx(&s_load[st], S::kStageBytes);
        __syncwarp();
        tma_cb(q, c, st, &s_load[st]);
        tma_x(q, c, st, &s_load[st]);
        if (st == 0) ld_issued0++; else ld_issued1++;
    };
    auto issue_cb1 = [&](const SsdSeq& q, int64_t c) {     // one stage
        if (lane == 0) tc::mbar_expect_tx(&s_load[0], 2 * S::kTileCB);
        __syncwarp();
        tma_cb(q, c, 0, &s_load[0]);
        ld_issued0++;
    };
    auto issue_x1 = [&](const SsdSeq& q, int64_t c) {
        if (lane == 0) tc::mbar_expect_tx(&s_load[1], S::kTileX);
        __syncwarp();
        tma_x(q, c, 0, &s_load[1]);
        ld_issued1++;
    };
    auto issue_z = [&](const SsdSeq& q, int64_t c) {
        const int b = q.b, h = q.h;
        if (lane == 0) {
            tc::mbar_expect_tx(&s_zload, S::kTileX);
            tc::tma_load_3d(smem + S::kZ, &m.z, (int)(h * kP), (int)(c * kQ), (int)b, &s_zload);
        }
        z_issued++;
    };
    // a piece's first copies (chunks c0 and c0 + 1 at running counts v0, v0 + 1)
    auto issue_first = [&](const SsdSeq& q, int c0, int c1, int v0) {
        if (S::kStages == 2) {
            issue_stage(q, c0, v0);
            if (c0 + 1 < c1) issue_stage(q, c0 + 1, v0 + 1);
        } else {
            issue_cb1(q, c0);
            issue_x1(q, c0);
        }
        if (zg) issue_z(q, c0);
    };

    if (warp == kCtl) {
        if (lane == 0) {
            for (int k = 0; k < 3; k++) tc::mbar_init(&s_bar[k], 1);
            tc::mbar_init(&s_load[0], 1);
            tc::mbar_init(&s_load[1], 1);
            tc::mbar_init(&s_zload, 1);
            for (int k = 0; k < 3; k++) tc::mbar_init(&s_ready[k], kCtl);   // one arrival per compute warp
            tc::mbar_init(&s_yfree, 1);
            tc::mbar_init(&s_drain, 1);
            *abort_flag = 0;
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncwarp();
        // the first piece's copies start while tensor memory is allocated
        int u, c0, c1;
        piece(0, u, c0, c1);
        if (c1 > c0) issue_first(make_seq(u), c0, c1, 0);
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
    const int row = 32 * quad + lane;   // this thread's tensor-memory lane: t (G1-G3) or n (G4)
    bool failed = false;
    // the control warp decides every wait as one (a lane that gave up while another
    // saw the phase complete would leave the warp split at its next __syncwarp)
    auto ctl_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, wait_or_abort(bar, parity, abort_flag, wlim));
    };

    if (warp == kCtl) {
        // =============================== control warp ===============================
        constexpr uint32_t idG1 = tc::idesc_bf16(128, 128, 0, 0);
        constexpr uint32_t idG2 = tc::idesc_bf16(128, kP, 0, 1);
        constexpr uint32_t idG4 = tc::idesc_bf16(128, kP, 1, 1);
        // G1 of chunk k: S = C B^T once C and B are in (S was last read by M(k-1)).
        // With two input stages it is issued right after G2 of the previous chunk, so
        // it runs under that chunk's epilogue; with one stage, when its C and B land.
        auto issue_g1 = [&](int64_t k) -> bool {
            const int stk = S::kStages == 2 ? (int)(k & 1) : 0;
            const uint32_t sCk = base + S::kStage0 + stk * S::kStageBytes + S::kC;
            const uint32_t sBk = sCk + S::kB - S::kC;
            uint64_t* bar = S::kStages == 2 ? &s_load[stk] : &s_load[0];
            const uint32_t p = S::kStages == 2 ? (uint32_t)((k >> 1) & 1) : (uint32_t)(k & 1);
            if (!ctl_wait(bar, p)) return false;
            if (S::kStages == 2 && stk == 1) ld_seen1++; else ld_seen0++;
            if (lane == 0) {
                tc::fence_after_sync();
                for (int j = 0; j < kN / 16; j++) {
                    const uint32_t off = (j >> 2) * 16384 + (j & 3) * 32;
                    tc::mma_bf16(tmem + kColS, tc::smem_desc_sw128(sCk + off, 16, 1024),
                                 tc::smem_desc_sw128(sBk + off, 16, 1024), idG1, j > 0);
                }
                tc::commit(&s_bar[0]);
            }
            __syncwarp();
            return true;
        };
        int v0 = 0;   // running chunk count at the piece's first chunk
        for (int pi = 0; pi < n_pieces && !failed; pi++) {
            int u, c0, c1;
            piece(pi, u, c0, c1);
            const SsdSeq q = make_seq(u);
            if (c1 <= c0) continue;   // an empty sequence: nothing to copy or multiply
            // the piece's first copies (the first piece's went out before the loop): the
            // previous piece's chunks are finished, its products done and its last y out
            // of the z tile, so every stage is free
            if (pi > 0) issue_first(q, c0, c1, v0);
            if (S::kStages == 2 && !issue_g1(v0)) {
                if (lane == 0) fail(__LINE__);
                failed = true;
                break;
            }
            for (int c = c0; c < c1 && !failed; c++) {
                const int v = v0 + (c - c0);
                const int st = S::kStages == 2 ? (int)(v & 1) : 0;
                const uint32_t par = (uint32_t)(v & 1);
                const uint32_t sC = base + S::kStage0 + st * S::kStageBytes + S::kC;
                const uint32_t sB = sC + S::kB - S::kC;
                const uint32_t sX = sC + S::kX - S::kC;
                if (S::kStages == 1 && !issue_g1(v)) {
                    if (lane == 0) fail(__LINE__);
                    failed = true;
                    break;
                }
                // G3, G4 once w o x and the rescaled state are written
                if (!ctl_wait(&s_ready[0], par)) {
                    if (lane == 0) fail(__LINE__);
                    failed = true;
                    break;
                }
                if (lane == 0) {
                    tc::fence_after_sync();
                    // G3: Ye = C Hh^T + C Hl^T (C: K-major, swizzled)
                    for (int hl = 0; hl < 2; hl++)
                        for (int k = 0; k < kN / 16; k++)
                            tc::mma_bf16(tmem + kColYe,
                                         tc::smem_desc_sw128(sC + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024),
                                         tc::smem_desc(base + (hl ? S::kHl : S::kHh) + k * 256, 128, S::kStrideH), idG2,
                                         hl > 0 || k > 0);
                    // G4: H^T += B^T (w o x)_hi + B^T (w o x)_lo (B^T: MN-major, swizzled,
                    // 64-row atoms 16 KB apart)
                    for (int hl = 0; hl < 2; hl++)
                        for (int k = 0; k < kQ / 16; k++)
                            tc::mma_bf16(tmem + kColH, tc::smem_desc_sw128(sB + k * 2048, 16384, 1024),
                                         tc::smem_desc(base + (hl ? S::kWl : S::kWh) + k * 256, 128, kStrideC), idG4,
                                         true);
                    tc::commit(&s_bar[1]);
                }
                __syncwarp();
                // G2 once M is written (and, with one stage, x is in)
                bool ok = ctl_wait(&s_ready[1], par);
                if (ok && S::kStages == 1) {
                    ok = ctl_wait(&s_load[1], par);
                    if (ok) ld_seen1++;
                }
                if (!ok) {
                    if (lane == 0) fail(__LINE__);
                    failed = true;
                    break;
                }
                if (lane == 0) {
                    tc::fence_after_sync();
                    // G2: Yi = Mh x + Ml x (x: MN-major, swizzled, one atom)
                    for (int hl = 0; hl < 2; hl++)
                        for (int k = 0; k < kQ / 16; k++)
                            tc::mma_bf16(tmem + kColYi,
                                         tc::smem_desc(base + (hl ? S::kMl : S::kMh) + k * 2 * kStrideC, kStrideC, 128),
                                         tc::smem_desc_sw128(sX + k * 2048, 16384, 1024), idG2, hl > 0 || k > 0);
                    tc::commit(&s_bar[2]);
                }
                __syncwarp();
                // two stages: the next chunk's G1 now (M(v) has read S)
                if (S::kStages == 2 && c + 1 < c1 && !issue_g1(v + 1)) {
                    if (lane == 0) fail(__LINE__);
                    failed = true;
                    break;
                }
                // one stage: the next chunk's C and B as soon as this chunk's products are done
                if (S::kStages == 1 && c + 1 < c1) {
                    if (!ctl_wait(&s_bar[2], par)) {
                        if (lane == 0) fail(__LINE__);
                        failed = true;
                        break;
                    }
                    issue_cb1(q, c + 1);
                }
                // chunk finished: y out; the next z and x (or the stage after next) in
                if (!ctl_wait(&s_ready[2], par)) {
                    if (lane == 0) fail(__LINE__);
                    failed = true;
                    break;
                }
                {
                    constexpr int kAtoms = kOutF32 ? 2 : 1;
                    if (lane < kAtoms)
                        tc::tma_store_3d(&m.y, q.h * kP + 32 * lane, (int)(c * kQ), q.b,
                                         smem + kY + lane * 16384);
                    tc::bulk_commit();
                }
                if (S::kStages == 2) {
                    if (c + 2 < c1) issue_stage(q, c + 2, v + 2);
                } else if (c + 1 < c1) {
                    issue_x1(q, c + 1);
                }
                tc::bulk_wait_read();   // y has left its staging tile (z's, or M's for fp32)
                if (zg) {
                    z_seen = (uint32_t)v + 1;   // the compute warps consumed z(v) before finishing
                    if (c + 1 < c1) issue_z(q, c + 1);
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&s_yfree);
            }
            v0 += c1 - c0;
        }
        if (failed) {
            // let the tensor core and the copy engine finish what they still owe
            // before the memory they write goes away
            if (lane == 0) {
                tc::commit(&s_drain);
                (void)tc::mbar_wait(&s_drain, 0, kWaitLimit);
            }
            for (; ld_seen0 < ld_issued0; ld_seen0++) (void)tc::mbar_wait(&s_load[0], ld_seen0 & 1u, kWaitLimit);
            for (; ld_seen1 < ld_issued1; ld_seen1++) (void)tc::mbar_wait(&s_load[1], ld_seen1 & 1u, kWaitLimit);
            for (; z_seen < z_issued; z_seen++) (void)tc::mbar_wait(&s_zload, z_seen & 1u, kWaitLimit);
        }
        tc::bulk_wait_read();
    } else {
        // =============================== compute warps ==============================
        // raw dt bits of step tid of chunk c (widened only where used, so loads stay
        // in flight across a chunk)
        auto load_dt = [&](const SsdSeq& q, int c, int c1) -> uint32_t {
            const int64_t t = (int64_t)c * kQ + tid;
            return (tid < kQ && c < c1 && t < L) ? (uint32_t)__ldg(dtb + ((int64_t)q.b * L + t) * H + q.h) : 0u;
        };
        // dt and the in-chunk cumulative sum of dt A (log2 domain) of chunk k (running
        // count vk) into s_cs2[vk & 1], s_dt[vk & 1] (and this thread's cs, dtv); all
        // compute threads
        auto scan_chunk = [&](const SsdSeq& q, int k, int vk, uint32_t bits, float& cs, float& dtv) {
            const int64_t rest = L - (int64_t)k * kQ;
            const int steps = (int)(rest < kQ ? rest : kQ);
            cs = 0.f;
            dtv = 0.f;
            if (tid < kQ) {
                if (tid < steps) {
                    const float v = __uint_as_float(bits << 16) + q.bias;
                    dtv = a.softplus ? softplus_acc<true>(v) : v;
                }
                cs = dtv * q.A2;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float u = __shfl_up_sync(0xffffffffu, cs, o);
                    if (lane >= o) cs += u;
                }
                if (lane == 31) s_wsum[warp] = cs;
            }
            compute_sync();
            if (tid < kQ) {
                for (int w = 0; w < warp; w++) cs += s_wsum[w];
                s_cs2[vk & 1][tid] = cs;
                s_dt[vk & 1][tid] = dtv;
            }
        };
        float cs = 0.f, dtv = 0.f;
        int v0 = 0;   // running chunk count at the piece's first chunk
        for (int pi = 0; pi < n_pieces && !failed; pi++) {
            int u, c0, c1;
            piece(pi, u, c0, c1);
            const SsdSeq q = make_seq(u);
            // the piece's starting state H^T[n][p]: h0[b,h,p,n] at chunk 0 (zero for
            // n >= N or without h0), else the state the previous ticket published (a
            // bounded wait; on expiry the failure is recorded and the run stops)
            const int64_t prev = s_run.ticket - 1;
            if (c0 > 0) {
                bool got = true;
                if (tid == 0) {
                    uint32_t spins = 0;
                    while (ld_acquire_u32(bal_flags() + prev) == 0 && spins < a.spin_limit && !*abort_flag) {
                        ++spins;
                        __nanosleep(64);
                    }
                    got = ld_acquire_u32(bal_flags() + prev) != 0;
                }
                if (compute_any(!got)) {
                    if (tid == 0) fail(__LINE__);
                    failed = true;
                    break;
                }
                (void)ld_acquire_u32(bal_flags() + prev);   // this thread's own acquire
            }
            float hv[kPc];
#pragma unroll
            for (int j = 0; j < kPc; j++) {
                const int p = kPc * part + j;
                float x = 0.f;
                if (row < kN) {
                    if (c0 > 0) x = __ldcg(bal_slots() + (prev * kP + p) * kN + row);
                    else if (a.h0) x = a.h0[((int64_t)q.bh * kP + p) * kN + row];
                }
                hv[j] = x;
            }
            if (c1 <= c0) {   // an empty sequence: its final state is the initial one
                if (c1 == nchunks && a.h_last && row < kN) {
#pragma unroll
                    for (int j = 0; j < kPc; j++) a.h_last[((int64_t)q.bh * kP + kPc * part + j) * kN + row] = hv[j];
                }
                continue;
            }
            uint32_t dt_next = load_dt(q, c0 + 1, c1);
            scan_chunk(q, c0, v0, load_dt(q, c0, c1), cs, dtv);
            compute_sync();   // the first chunk's cumulative decays are visible
            // split for G3, and resident rescaled by the first chunk's total decay for G4
            if (row < kN) {
#pragma unroll
                for (int k = 0; k < kPc / 8; k++)
                    split_store8(hv + 8 * k, sHh + ((kPc / 8) * part + k) * S::kStrideH + row * 16,
                                 sHl + ((kPc / 8) * part + k) * S::kStrideH + row * 16);
            }
            {
                const float e0 = ex2(s_cs2[v0 & 1][kQ - 1]);
#pragma unroll
                for (int j = 0; j < kPc; j++) hv[j] *= e0;
            }
            tc::tmem_st16(tmem + lane_base + kColH + kPc * part, hv);
            tc::tmem_wait_st();
            for (int c = c0; c < c1; c++) {
                const int v = v0 + (c - c0);
                const int st = S::kStages == 2 ? (int)(v & 1) : 0;
                const uint32_t par = (uint32_t)(v & 1);
                unsigned char* stg = smem + S::kStage0 + st * S::kStageBytes;
                const float* cs2 = s_cs2[v & 1];
                const float* dts = s_dt[v & 1];
                // ---- this chunk's x in --------------------------------------------------
                {
                    uint64_t* bar = S::kStages == 2 ? &s_load[st] : &s_load[1];
                    const uint32_t p = S::kStages == 2 ? (uint32_t)((v >> 1) & 1) : par;
                    const bool ok = wait_or_abort(bar, p, abort_flag, wlim);
                    if (compute_any(!ok)) {
                        if (tid == 0) fail(__LINE__);
                        failed = true;
                        break;
                    }
                }
                const float cs2_end = cs2[kQ - 1];
                if (tid < kQ) s_w[tid] = ex2(cs2_end - cs) * dtv;
                compute_sync();
                // ---- w o x, split; rescale the resident state by exp(cs_end) -------------
                for (int i = tid; i < kQ * (kP / 8); i += kCompute) {
                    float v[8];
                    unpack8(*reinterpret_cast<const uint4*>(stg + S::kX + tc::sw128(i & (kQ - 1), i >> 7)), v);
                    const float w = s_w[i & (kQ - 1)];
    #pragma unroll
                    for (int k = 0; k < 8; k++) v[k] *= w;
                    split_store8(v, sWh + 16 * i, sWl + 16 * i);
                }
                tc::fence_proxy_async();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0 && !(a.withhold_arrive && warp == 0 && v == 0)) tc::mbar_arrive(&s_ready[0]);
                // ---- M from S: decay mask, split into the two A operands of G2 -----------
                {
                    bool ok = wait_or_abort(&s_bar[0], par, abort_flag, wlim);
                    if (ok && kOutF32 && v > 0) ok = wait_or_abort(&s_yfree, (uint32_t)((v - 1) & 1), abort_flag, wlim);
                    if (compute_any(!ok)) {
                        if (tid == 0) fail(__LINE__);
                        failed = true;
                        break;
                    }
                }
                tc::fence_after_sync();
                {
                    const float cs_t = cs2[row];
                    // a 32-column block is, for this warp's 32 rows, all above the
                    // diagonal (zeros), all on or below it (no mask), or crossing it
    #pragma unroll
                    for (int blk = 0; blk < kSc / 32; blk++) {
                        const int s0 = kSc * part + 32 * blk;
                        if (s0 > 32 * quad + 31) {
                            const uint4 zero = make_uint4(0, 0, 0, 0);
    #pragma unroll
                            for (int k = 0; k < 4; k++) {
                                *reinterpret_cast<uint4*>(sMh + chunk_off(row, s0 / 8 + k)) = zero;
                                *reinterpret_cast<uint4*>(sMl + chunk_off(row, s0 / 8 + k)) = zero;
                            }
                            continue;
                        }
                        float v[32];
                        tc::tmem_ld32(tmem + lane_base + kColS + s0, v);
                        tc::tmem_wait_ld();
                        if (s0 + 31 <= 32 * quad) {
    #pragma unroll
                            for (int j = 0; j < 32; j++) v[j] = v[j] * ex2(cs_t - cs2[s0 + j]) * dts[s0 + j];
                        } else {
    #pragma unroll
                            for (int j = 0; j < 32; j++) {
                                const int s = s0 + j;
                                v[j] = s <= row ? v[j] * ex2(cs_t - cs2[s]) * dts[s] : 0.f;
                            }
                        }
    #pragma unroll
                        for (int k = 0; k < 4; k++)
                            split_store8(v + 8 * k, sMh + chunk_off(row, s0 / 8 + k), sMl + chunk_off(row, s0 / 8 + k));
                    }
                }
                tc::fence_proxy_async();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&s_ready[1]);
                // the next chunk's dt scan while the last product runs
                float cs_next = 0.f, dtv_next = 0.f;
                if (c + 1 < c1) {
                    scan_chunk(q, c + 1, v + 1, dt_next, cs_next, dtv_next);
                    dt_next = load_dt(q, c + 2, c1);
                }
                // ---- products in; epilogue: y = Yi + exp(cs_t) Ye + D x, gated, staged ----
                {
                    bool ok = wait_or_abort(&s_bar[2], par, abort_flag, wlim) &&
                              wait_or_abort(&s_bar[1], par, abort_flag, wlim);
                    if (ok && zg) ok = wait_or_abort(&s_zload, par, abort_flag, wlim);
                    if (compute_any(!ok)) {
                        if (tid == 0) fail(__LINE__);
                        failed = true;
                        break;
                    }
                }
                tc::fence_after_sync();
                {
                    float yi[kPc], ye[kPc];
                    tc::tmem_ld16(tmem + lane_base + kColYi + kPc * part, yi);
                    tc::tmem_ld16(tmem + lane_base + kColYe + kPc * part, ye);
                    tc::tmem_wait_ld();
                    const float e = ex2(cs2[row]);   // exp(cs_t)
                    float out[kPc];
    #pragma unroll
                    for (int k = 0; k < kPc / 8; k++) {
                        float xv[8];
                        unpack8(*reinterpret_cast<const uint4*>(stg + S::kX + tc::sw128(row, (kPc / 8) * part + k)), xv);
                        float zv[8];
                        if (zg)
                            unpack8(*reinterpret_cast<const uint4*>(smem + S::kZ + tc::sw128(row, (kPc / 8) * part + k)),
                                    zv);
    #pragma unroll
                        for (int i = 0; i < 8; i++) {
                            float yv = fmaf(e, ye[8 * k + i], yi[8 * k + i]);
                            yv = fmaf(q.Dh, xv[i], yv);
                            if (zg) yv *= silu_acc<false>(zv[i]);
                            out[8 * k + i] = yv;
                        }
                    }
                    // rows past seqlen are staged too; the store drops them
                    unsigned char* sy = smem + kY;
                    if constexpr (kOutF32) {   // two atoms: columns 0-31 and 32-63, 4 per chunk
                        constexpr int kPerAtom = 32 / kPc;
    #pragma unroll
                        for (int k = 0; k < kPc / 4; k++)
                            *reinterpret_cast<float4*>(sy + (part / kPerAtom) * 16384 +
                                                       tc::sw128(row, (kPc / 4) * (part % kPerAtom) + k)) =
                                make_float4(out[4 * k], out[4 * k + 1], out[4 * k + 2], out[4 * k + 3]);
                    } else {
    #pragma unroll
                        for (int k = 0; k < kPc / 8; k++)
                            Vec16<__nv_bfloat16>::store(
                                reinterpret_cast<__nv_bfloat16*>(sy + tc::sw128(row, (kPc / 8) * part + k)), out + 8 * k);
                    }
                }
                // ---- the new state: G3's split operand for the next chunk, and the resident
                // copy rescaled by the next chunk's total decay for G4 to accumulate into
                if (c + 1 < c1) {
                    float hn[kPc];
                    tc::tmem_ld16(tmem + lane_base + kColH + kPc * part, hn);
                    tc::tmem_wait_ld();
                    if (row < kN) {
    #pragma unroll
                        for (int k = 0; k < kPc / 8; k++)
                            split_store8(hn + 8 * k, sHh + ((kPc / 8) * part + k) * S::kStrideH + row * 16,
                                         sHl + ((kPc / 8) * part + k) * S::kStrideH + row * 16);
                    }
                    const float e_next = ex2(s_cs2[(v + 1) & 1][kQ - 1]);
    #pragma unroll
                    for (int j = 0; j < kPc; j++) hn[j] *= e_next;
                    tc::tmem_st16(tmem + lane_base + kColH + kPc * part, hn);
                    tc::tmem_wait_st();
                }
                tc::fence_proxy_async();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&s_ready[2]);
                cs = cs_next;
                dtv = dtv_next;
            }
            if (failed) break;
            // the piece's final state: h_last at its sequence's end, else this ticket's
            // slot, then published for the next ticket's tail
            {
                float hf[kPc];
                tc::tmem_ld16(tmem + lane_base + kColH + kPc * part, hf);
                tc::tmem_wait_ld();
                if (c1 == nchunks) {
                    if (a.h_last && row < kN) {
#pragma unroll
                        for (int j = 0; j < kPc; j++) a.h_last[((int64_t)q.bh * kP + kPc * part + j) * kN + row] = hf[j];
                    }
                } else {
                    if (row < kN) {
#pragma unroll
                        for (int j = 0; j < kPc; j++)
                            bal_slots()[(s_run.ticket * kP + kPc * part + j) * kN + row] = hf[j];
                    }
                    __threadfence();
                    compute_sync();
                    // (test hook: ticket drop_ticket withholds its publication)
                    if (tid == 0 && s_run.ticket != a.drop_ticket) st_release_u32(bal_flags() + s_run.ticket, 1u);
                }
            }
            v0 += c1 - c0;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
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

// (row elements, seqlen, batch) view of bf16 (esize 2) or fp32 (esize 4) rows,
// 128-byte x 128-step boxes, 128-byte swizzled in shared memory
bool encode_rows(CUtensorMap* map, const void* base, int64_t row, int64_t L, int64_t batch, int esize = 2) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)row, (cuuint64_t)L, (cuuint64_t)batch};
    const cuuint64_t strides[2] = {(cuuint64_t)(row * esize), (cuuint64_t)(row * L * esize)};
    const cuuint32_t box[3] = {(cuuint32_t)(128 / esize), (cuuint32_t)kQ, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
              const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kN, bool kOutF32>
cudaError_t launch_n(const SsdArgs& a, cudaStream_t s) {
    SsdMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (a.seqlen > 0) {
        const int64_t bc_row = a.ngroups * kN, x_row = a.nheads * kP;
        if (!encode_rows(&maps.c, a.C, bc_row, a.seqlen, a.batch) ||
            !encode_rows(&maps.b, a.B, bc_row, a.seqlen, a.batch) ||
            !encode_rows(&maps.x, a.x, x_row, a.seqlen, a.batch) ||
            (a.z && !encode_rows(&maps.z, a.z, x_row, a.seqlen, a.batch)) ||
            !encode_rows(&maps.y, a.y, x_row, a.seqlen, a.batch, kOutF32 ? 4 : 2))
            return cudaErrorInvalidValue;
    }
    auto k = ssd_chunk_scan_kernel<kN, kOutF32>;
    constexpr uint32_t bytes = Smem<kN>::kBytes;
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, k);
    if (e != cudaSuccess) return e;
    if (fa.sharedSizeBytes + bytes > 232448) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    // The work-balanced launch when a workspace is given and the sequences do not
    // already fill whole rounds of the resident CTAs: P = (resident CTAs), or fewer,
    // a multiple of the SM count and at most the sequence count (runs of at least
    // one whole sequence). At (4, 4096, 80 heads) 320 one-sequence CTAs took three
    // rounds (352 us) where 296 took two (236 us) and 148 one (120 us).
    SsdArgs b = a;
    b.bal_ctas = 0;
    const int64_t units = a.batch * a.nheads;
    const int64_t nch = (a.seqlen + kQ - 1) / kQ;
    if (a.workspace && a.seqlen > 0 && units * nch < ((int64_t)1 << 31)) {   // 32-bit chunk counts in the kernel
        int dev = 0, sms = 0, occ = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kThreads, bytes) == cudaSuccess && sms > 0 &&
            occ > 0) {
            int64_t P = (int64_t)occ * sms;
            if (P > (units / sms) * sms) P = (units / sms) * sms;
            if (P > 0 && P < units && units % P != 0 && ssd_bal_workspace_bytes(P, kN) <= a.workspace_bytes)
                b.bal_ctas = P;
        }
    }
    if (b.bal_ctas > 0) {
        e = cudaMemsetAsync(b.workspace, 0, ssd_bal_slots_offset(b.bal_ctas), s);
        if (e != cudaSuccess) return e;
        k<<<(unsigned)b.bal_ctas, kThreads, bytes, s>>>(b, maps);
    } else {
        k<<<(unsigned)units, kThreads, bytes, s>>>(b, maps);
    }
    return cudaGetLastError();
}

}  // namespace

int64_t ssd_chunk_len() { return kQ; }

size_t ssd_bal_workspace_bytes(int64_t ctas, int dstate) {
    return ssd_bal_slots_offset(ctas) + (size_t)ctas * kP * (size_t)dstate * sizeof(float);
}

cudaError_t launch_ssd_scan(const SsdArgs& a, cudaStream_t s) {
    if (a.batch * a.nheads == 0) return cudaSuccess;
    const bool f32 = a.out_dtype == kF32;
    if (a.dstate == 128) return f32 ? launch_n<128, true>(a, s) : launch_n<128, false>(a, s);
    return f32 ? launch_n<64, true>(a, s) : launch_n<64, false>(a, s);
}

cudaError_t ssd_status(int* line, bool clear, cudaStream_t s) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(line, g_ssd_status, sizeof(int), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && clear && *line != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_ssd_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    return e;
}

}  // namespace ssm
