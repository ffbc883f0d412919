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
// One CTA of 256 threads per (b, h), walking the chunks in order. Warp w reaches
// tensor-memory lanes 32 (w % 4) .. +31 and works on column half w / 4.
// Tensor memory (256 columns): S and then Ye in [0, 128), Yi in [128, 192),
// H^T in [192, 256). Shared memory holds every operand tile in the unswizzled
// core-matrix layout (tcgen05.cuh) with 128 rows, stride_r = 128 B and
// stride_c = 2048 B, so 16-byte chunk (row r, column group j) sits at
// j * 2048 + r * 16.
#include <cuda_bf16.h>
#include <stdint.h>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace ssm {

__device__ int g_ssd_status;   // 0, or the source line of a wait that ran out of budget

namespace {

constexpr int kQ = 128;               // chunk length (steps)
constexpr int kP = 64;                // head channels
constexpr int kThreads = 256;
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr uint32_t kTileBig = 32768;  // 128 x 128 bf16
constexpr uint32_t kTileX = 16384;    // 128 x 64 bf16
// shared-memory map (bytes); the K-major tiles first so that every descriptor
// reach stays inside the allocation
constexpr uint32_t kOffMh = 0;
constexpr uint32_t kOffMl = kOffMh + kTileBig;
constexpr uint32_t kOffC = kOffMl + kTileBig;
constexpr uint32_t kOffB = kOffC + kTileBig;
constexpr uint32_t kOffX = kOffB + kTileBig;
constexpr uint32_t kOffWh = kOffX + kTileX;
constexpr uint32_t kOffWl = kOffWh + kTileX;
constexpr uint32_t kOffHh = kOffWl + kTileX;
constexpr uint32_t kOffHl = kOffHh + kTileX;
constexpr uint32_t kSmemBytes = kOffHl + kTileX;   // 212992
constexpr uint32_t kStrideC = 2048;                 // bytes between column groups
// tensor-memory columns
constexpr uint32_t kColS = 0, kColYe = 0, kColYi = 128, kColH = 192, kTmemCols = 256;

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

// Issue K/16 MMAs: D (+)= A . B over K. Operand descriptors advance by
// `astep` / `bstep` bytes per K step of 16.
__device__ __forceinline__ void mma_chain(uint32_t d, uint32_t a_addr, uint32_t a_lbo, uint32_t a_sbo,
                                          uint32_t astep, uint32_t b_addr, uint32_t b_lbo, uint32_t b_sbo,
                                          uint32_t bstep, uint32_t idesc, int ksteps, bool acc) {
    for (int k = 0; k < ksteps; k++)
        tc::mma_bf16(d, tc::smem_desc(a_addr + k * astep, a_lbo, a_sbo),
                     tc::smem_desc(b_addr + k * bstep, b_lbo, b_sbo), idesc, acc || k > 0);
}

template <int kN, bool kOutF32>
__global__ void __launch_bounds__(kThreads, 1) ssd_chunk_scan_kernel(SsdArgs a) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ float s_cs2[kQ];      // cs_t * log2(e)
    __shared__ float s_dt[kQ];
    __shared__ float s_e[kQ];        // exp(cs_t)
    __shared__ float s_w[kQ];        // exp(cs_end - cs_t) dt_t
    __shared__ float s_wsum[4];
    __shared__ uint64_t s_bar;
    __shared__ uint32_t s_tmem;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int quad = warp & 3, half = warp >> 2;
    const int64_t bh = blockIdx.x;
    const int64_t H = a.nheads, L = a.seqlen, G = a.ngroups;
    const int64_t b = bh / H, h = bh % H, g = h / (H / G);
    const float A2 = a.A[h] * kLog2e;
    const float bias = a.dt_bias ? a.dt_bias[h] : 0.f;
    const float Dh = a.D ? a.D[h] : 0.f;
    const __nv_bfloat16* xg = static_cast<const __nv_bfloat16*>(a.x);
    const __nv_bfloat16* dtg = static_cast<const __nv_bfloat16*>(a.dt);
    const __nv_bfloat16* Bg = static_cast<const __nv_bfloat16*>(a.B);
    const __nv_bfloat16* Cg = static_cast<const __nv_bfloat16*>(a.C);
    const __nv_bfloat16* zg = static_cast<const __nv_bfloat16*>(a.z);

    unsigned char* sMh = smem + kOffMh;
    unsigned char* sMl = smem + kOffMl;
    unsigned char* sC = smem + kOffC;
    unsigned char* sB = smem + kOffB;
    unsigned char* sX = smem + kOffX;
    unsigned char* sWh = smem + kOffWh;
    unsigned char* sWl = smem + kOffWl;
    unsigned char* sHh = smem + kOffHh;
    unsigned char* sHl = smem + kOffHl;
    const uint32_t base = tc::smem_u32(smem);

    // B^T serves G4 as a 128-row operand; with N = 64 its rows 64..127 stay zero
    if (kN < 128)
        for (int i = tid; i < (int)(kTileBig / 16); i += kThreads)
            reinterpret_cast<uint4*>(sB)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        tc::mbar_init(&s_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = s_tmem;
    const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
    const int row = 32 * quad + lane;   // this thread's tensor-memory lane: t (G1-G3) or n (G4)

    // initial state: H^T[n][p] = h0[b,h,p,n] (zero for n >= N or without h0)
    {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; j++) {
            const int p = 32 * half + j;
            v[j] = (a.h0 && row < kN) ? a.h0[(bh * kP + p) * kN + row] : 0.f;
        }
        tc::tmem_st32(tmem + lane_base + kColH + 32 * half, v);
#pragma unroll
        for (int k = 0; k < 4; k++)
            split_store8(v + 8 * k, sHh + chunk_off(row, 4 * half + k), sHl + chunk_off(row, 4 * half + k));
        tc::tmem_wait_st();
    }
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();

    constexpr uint32_t idG1 = tc::idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t idG2 = tc::idesc_bf16(128, kP, 0, 1);
    constexpr uint32_t idG4 = tc::idesc_bf16(128, kP, 1, 1);
    uint32_t phase = 0;
    bool failed = false;
    const int64_t nchunks = (L + kQ - 1) / kQ;

    for (int64_t c = 0; c < nchunks; c++) {
        const int64_t t0 = c * kQ;
        const int q = (int)((L - t0) < kQ ? (L - t0) : kQ);
        // ---- stage C, B (q x N) and x (q x 64) with zero-filled tails ----------
        {
            constexpr int kCJ = kN / 8;
            for (int i = tid; i < kQ * kCJ; i += kThreads) {
                const int r = i / kCJ, j = i % kCJ;
                const int rr = r < q ? r : 0;
                const int64_t gi = ((b * L + t0 + rr) * G + g) * kN + 8 * j;
                tc::cp_async16(sC + chunk_off(r, j), Cg + gi, r < q ? 16u : 0u);
                tc::cp_async16(sB + chunk_off(r, j), Bg + gi, r < q ? 16u : 0u);
            }
            for (int i = tid; i < kQ * (kP / 8); i += kThreads) {
                const int r = i & (kQ - 1), j = i >> 7;
                const int rr = r < q ? r : 0;
                tc::cp_async16(sX + chunk_off(r, j), xg + ((b * L + t0 + rr) * H + h) * kP + 8 * j,
                               r < q ? 16u : 0u);
            }
            tc::cp_async_commit();
        }
        // ---- dt and the in-chunk cumulative sum of dt A (log2 domain) ----------
        float cs = 0.f, dtv = 0.f;
        if (tid < kQ) {
            if (tid < q) {
                const float v = __bfloat162float(dtg[(b * L + t0 + tid) * H + h]) + bias;
                dtv = a.softplus ? softplus_acc<true>(v) : v;
            }
            cs = dtv * A2;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float u = __shfl_up_sync(0xffffffffu, cs, o);
                if (lane >= o) cs += u;
            }
            if (lane == 31) s_wsum[warp] = cs;
        }
        __syncthreads();
        if (tid < kQ) {
            for (int w = 0; w < warp; w++) cs += s_wsum[w];
            s_cs2[tid] = cs;
            s_dt[tid] = dtv;
        }
        tc::cp_async_wait_all();
        tc::fence_proxy_async();
        __syncthreads();
        // ---- G1: S = C B^T ------------------------------------------------------
        if (tid == 0) {
            tc::fence_after_sync();
            mma_chain(tmem + kColS, base + kOffC, kStrideC, 128, 2 * kStrideC, base + kOffB, kStrideC, 128,
                      2 * kStrideC, idG1, kN / 16, false);
            tc::commit(&s_bar);
        }
        const float cs2_end = s_cs2[kQ - 1];
        if (tid < kQ) {
            s_e[tid] = ex2(cs);
            s_w[tid] = ex2(cs2_end - cs) * dtv;
        }
        __syncthreads();
        // ---- w o x, split; rescale the resident state by exp(cs_end) -------------
        for (int i = tid; i < kQ * (kP / 8); i += kThreads) {
            float v[8];
            unpack8(*reinterpret_cast<const uint4*>(sX + 16 * i), v);
            const float w = s_w[i & (kQ - 1)];
#pragma unroll
            for (int k = 0; k < 8; k++) v[k] *= w;
            split_store8(v, sWh + 16 * i, sWl + 16 * i);
        }
        {
            const float e_end = ex2(cs2_end);
            float v[32];
            tc::tmem_ld32(tmem + lane_base + kColH + 32 * half, v);
            tc::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; j++) v[j] *= e_end;
            tc::tmem_st32(tmem + lane_base + kColH + 32 * half, v);
            tc::tmem_wait_st();
        }
        tc::fence_proxy_async();
        // ---- M from S: decay mask, split into the two A operands of G2 -----------
        {
            const bool ok = tc::mbar_wait(&s_bar, phase, kWaitLimit);
            if (__syncthreads_or(!ok)) {
                if (tid == 0) atomicExch(&g_ssd_status, __LINE__);
                failed = true;
                break;
            }
            phase ^= 1;
            tc::fence_after_sync();
            const float cs_t = s_cs2[row];
#pragma unroll
            for (int blk = 0; blk < 2; blk++) {
                const int s0 = 64 * half + 32 * blk;
                float v[32];
                tc::tmem_ld32(tmem + lane_base + kColS + s0, v);
                tc::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 32; j++) {
                    const int s = s0 + j;
                    v[j] = s <= row ? v[j] * ex2(cs_t - s_cs2[s]) * s_dt[s] : 0.f;
                }
#pragma unroll
                for (int k = 0; k < 4; k++)
                    split_store8(v + 8 * k, sMh + chunk_off(row, s0 / 8 + k), sMl + chunk_off(row, s0 / 8 + k));
            }
        }
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();
        // ---- G2, G3, G4 -------------------------------------------------------------
        if (tid == 0) {
            tc::fence_after_sync();
            // G2: Yi = Mh x + Ml x
            mma_chain(tmem + kColYi, base + kOffMh, kStrideC, 128, 2 * kStrideC, base + kOffX, 128, kStrideC,
                      256, idG2, kQ / 16, false);
            mma_chain(tmem + kColYi, base + kOffMl, kStrideC, 128, 2 * kStrideC, base + kOffX, 128, kStrideC,
                      256, idG2, kQ / 16, true);
            // G3: Ye = C Hh^T + C Hl^T
            mma_chain(tmem + kColYe, base + kOffC, kStrideC, 128, 2 * kStrideC, base + kOffHh, 128, kStrideC,
                      256, idG2, kN / 16, false);
            mma_chain(tmem + kColYe, base + kOffC, kStrideC, 128, 2 * kStrideC, base + kOffHl, 128, kStrideC,
                      256, idG2, kN / 16, true);
            // G4: H^T += B^T (w o x)_hi + B^T (w o x)_lo
            mma_chain(tmem + kColH, base + kOffB, 128, kStrideC, 256, base + kOffWh, 128, kStrideC, 256, idG4,
                      kQ / 16, true);
            mma_chain(tmem + kColH, base + kOffB, 128, kStrideC, 256, base + kOffWl, 128, kStrideC, 256, idG4,
                      kQ / 16, true);
            tc::commit(&s_bar);
        }
        {
            const bool ok = tc::mbar_wait(&s_bar, phase, kWaitLimit);
            if (__syncthreads_or(!ok)) {
                if (tid == 0) atomicExch(&g_ssd_status, __LINE__);
                failed = true;
                break;
            }
            phase ^= 1;
        }
        tc::fence_after_sync();
        // ---- epilogue: y = Yi + exp(cs_t) Ye + D x, gated ---------------------------
        {
            float yi[32], ye[32];
            tc::tmem_ld32(tmem + lane_base + kColYi + 32 * half, yi);
            tc::tmem_ld32(tmem + lane_base + kColYe + 32 * half, ye);
            tc::tmem_wait_ld();
            if (row < q) {
                const float e = s_e[row];
                const int64_t gi = ((b * L + t0 + row) * H + h) * kP + 32 * half;
                float out[32];
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    float xv[8];
                    unpack8(*reinterpret_cast<const uint4*>(sX + chunk_off(row, 4 * half + k)), xv);
                    float zv[8];
                    if (zg) unpack8(__ldg(reinterpret_cast<const uint4*>(zg + gi + 8 * k)), zv);
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        float yv = fmaf(e, ye[8 * k + i], yi[8 * k + i]);
                        yv = fmaf(Dh, xv[i], yv);
                        if (zg) yv *= silu_acc<false>(zv[i]);
                        out[8 * k + i] = yv;
                    }
                }
                if constexpr (kOutF32) {
                    float* yo = static_cast<float*>(a.y) + gi;
#pragma unroll
                    for (int k = 0; k < 8; k++)
                        reinterpret_cast<float4*>(yo)[k] =
                            make_float4(out[4 * k], out[4 * k + 1], out[4 * k + 2], out[4 * k + 3]);
                } else {
                    __nv_bfloat16* yo = static_cast<__nv_bfloat16*>(a.y) + gi;
#pragma unroll
                    for (int k = 0; k < 4; k++) Vec16<__nv_bfloat16>::store(yo + 8 * k, out + 8 * k);
                }
            }
        }
        // ---- the new state as G3's split operand for the next chunk -----------------
        if (c + 1 < nchunks) {
            float v[32];
            tc::tmem_ld32(tmem + lane_base + kColH + 32 * half, v);
            tc::tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 4; k++)
                split_store8(v + 8 * k, sHh + chunk_off(row, 4 * half + k), sHl + chunk_off(row, 4 * half + k));
        }
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncthreads();
    }

    if (!failed && a.h_last && row < kN) {
        tc::fence_after_sync();
        float v[32];
        tc::tmem_ld32(tmem + lane_base + kColH + 32 * half, v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; j++) a.h_last[(bh * kP + 32 * half + j) * kN + row] = v[j];
    }
    if (failed) {
        // let whatever the tensor core still owes (the phase that timed out)
        // complete before its memory goes
        (void)tc::mbar_wait(&s_bar, phase, kWaitLimit);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

template <int kN, bool kOutF32>
cudaError_t launch_n(const SsdArgs& a, cudaStream_t s) {
    auto k = ssd_chunk_scan_kernel<kN, kOutF32>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    k<<<(unsigned)(a.batch * a.nheads), kThreads, kSmemBytes, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

int64_t ssd_chunk_len() { return kQ; }

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
