// kernels_conv.cu -- the causal depthwise conv1d + silu that feeds the scan, and its
// single-token decode update.
//
// What is computed (Mamba SSM complete guide (youngju.dev), section 5, "complete
// Mamba implementation": MambaBlock.__init__ builds a depthwise nn.Conv1d with
// kernel d_conv and padding d_conv - 1, forward keeps the first seqlen outputs and
// applies silu before the SSM). PyTorch's Conv1d is a cross-correlation over the
// input padded on the left, so for width W = d_conv:
//     out[b,d,t] = silu( bias[d] + sum_{k<W} w[d,k] * xp[b,d,t+k] ),
//     xp[t'] = x[t' - (W-1)] for t' >= W-1, else the conv state (the W-1 inputs
//     before this call, oldest first; zeros when none).
// The decode update applies the same sum to (state, x_t) and shifts x_t into the
// state.
//
// Why not fused into the scan's prologue: in the block, x_proj maps the conv
// output u to the scan's delta, B and C, so u has to be in memory before the scan
// starts; the scan reads it like any input. The conv is therefore its own pass,
// HBM-bound: per token*channel it reads the input once and writes u once.
//
// Prefill layout: a warp walks a segment of one (b, d) row in blocks of 32
// 16-byte vectors (256 bf16 or 128 fp32 steps); lane i owns vector i of the
// block, so each load and store instruction moves 512 contiguous bytes. The W-1
// inputs before a lane's vector come from lane i-1 by shuffle; lane 0 takes the
// previous block's last inputs (carried in registers) or, at the segment start,
// reads them from x (or the conv state). Each lane keeps its next four vectors
// in flight. Rows are cut into segments only when there are too few rows to
// fill the GPU.
#include <string.h>

#include "common.cuh"
#include "launch.h"

namespace ssm {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;

// V outputs at row[t ..], those before te only.
template <typename Tout, int V, bool kVec>
__device__ __forceinline__ void store_v(Tout* row, int64_t t, int64_t te, const float* v) {
    if (kVec && t + V <= te) {
        if constexpr (sizeof(Tout) == 2 && V == 8) {
            Vec16<Tout>::store(row + t, v);
            return;
        } else if constexpr (sizeof(Tout) == 4) {
#pragma unroll
            for (int k = 0; k < V; k += 4) Vec16<Tout>::store(row + t + k, v + k);
            return;
        } else {   // bf16 out, fp32 in: 4 values, 8 bytes
            __nv_bfloat162 h0 = __floats2bfloat162_rn(v[0], v[1]), h1 = __floats2bfloat162_rn(v[2], v[3]);
            *reinterpret_cast<uint2*>(row + t) =
                make_uint2(*reinterpret_cast<uint32_t*>(&h0), *reinterpret_cast<uint32_t*>(&h1));
            return;
        }
    }
#pragma unroll
    for (int k = 0; k < V; k++)
        if (t + k < te) row[t + k] = from_f32<Tout>(v[k]);
}

// the padded input at time tau < 0 or tau >= 0 of one row: x itself, else the state
template <typename Tin>
__device__ __forceinline__ float padded(const Tin* xr, const float* st, int hw, int64_t tau) {
    if (tau >= 0) return to_f32(xr[tau]);
    return st ? st[hw + tau] : 0.f;
}

// raw 16-byte vector at row[t ..] (zero past L; element loads when not whole)
template <typename T, bool kVec>
__device__ __forceinline__ uint4 load_raw(const T* row, int64_t t, int64_t L) {
    constexpr int V = Vec16<T>::kN;
    if (kVec && t + V <= L) return __ldg(reinterpret_cast<const uint4*>(row + t));
    float f[V];
#pragma unroll
    for (int k = 0; k < V; k++) f[k] = (t + k < L) ? to_f32(row[t + k]) : 0.f;
    T tmp[V];
#pragma unroll
    for (int k = 0; k < V; k++) tmp[k] = from_f32<T>(f[k]);
    uint4 r;
    memcpy(&r, tmp, 16);
    return r;
}

template <typename T>
__device__ __forceinline__ void widen(const uint4& r, float* out) {
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

// blocks of 32 vectors each lane keeps in flight: 4 x 512 bytes per warp, so the
// ~32 resident warps of an SM hold ~64 KB of loads in flight (HBM latency x the
// SM's share of the bandwidth)
#ifndef SSM_CONV_DEPTH
#define SSM_CONV_DEPTH 4
#endif
constexpr int kDepth = SSM_CONV_DEPTH;

template <typename Tin, typename Tout, int W, bool kVec>
__global__ void __launch_bounds__(kThreads) causal_conv1d_kernel(ConvArgs a) {
    constexpr bool kAcc = sizeof(Tin) == 4;
    constexpr int V = Vec16<Tin>::kN;
    constexpr int HW = W - 1;            // halo width
    constexpr int HA = HW > 0 ? HW : 1;  // array size
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t rows = a.batch * a.dim;
    if (gw >= rows * a.n_seg) return;    // whole warp
    const int64_t row = gw / a.n_seg, seg = gw % a.n_seg;
    const int64_t d = row % a.dim, L = a.seqlen;
    const int64_t tb = seg * a.seg_len, te = min(L, tb + a.seg_len);
    const Tin* xr = static_cast<const Tin*>(a.x) + row * L;
    Tout* orow = static_cast<Tout*>(a.out) + row * L;
    const float* st_in = a.state_in ? a.state_in + row * HW : nullptr;
    float w[W];
#pragma unroll
    for (int k = 0; k < W; k++) w[k] = a.w[d * W + k];
    const float bias = a.bias ? a.bias[d] : 0.f;

    // the first blocks' loads go out before anything else
    const int64_t nblk = te > tb ? (te - tb + 32 * V - 1) / (32 * V) : 0;
    uint4 ring[kDepth];
#pragma unroll
    for (int u = 0; u < kDepth; u++)
        if (u < nblk) ring[u] = load_raw<Tin, kVec>(xr, tb + (int64_t)(u * 32 + lane) * V, L);

    // inputs before the segment (every lane holds them; lane 0 uses them)
    float h[HA];
#pragma unroll
    for (int j = 0; j < HW; j++) h[j] = padded(xr, st_in, HW, tb - HW + j);
    // the state a following call continues from: the last W-1 padded inputs,
    // written by the segment-0 warp after it has read the incoming state (so the
    // two may be the same array)
    __syncwarp();
    if (seg == 0 && a.state_out && lane == 0) {
        float so[HA];
#pragma unroll
        for (int j = 0; j < HW; j++) so[j] = padded(xr, st_in, HW, L - HW + j);
#pragma unroll
        for (int j = 0; j < HW; j++) a.state_out[row * HW + j] = so[j];
    }

    for (int64_t b0 = 0; b0 < nblk; b0 += kDepth) {
#pragma unroll
        for (int u = 0; u < kDepth; u++) {
            const int64_t bk = b0 + u;
            if (bk >= nblk) break;                   // warp-uniform
            const int64_t t = tb + (bk * 32 + lane) * V;
            float v[V];
            widen<Tin>(ring[u], v);
            if (bk + kDepth < nblk) ring[u] = load_raw<Tin, kVec>(xr, t + (int64_t)kDepth * 32 * V, L);
            // the W-1 inputs before this lane's vector
            float prev[HA];
#pragma unroll
            for (int j = 0; j < HW; j++) {
                const float up = __shfl_up_sync(0xffffffffu, v[V - HW + j], 1);
                prev[j] = lane == 0 ? h[j] : up;
            }
#pragma unroll
            for (int j = 0; j < HW; j++) h[j] = __shfl_sync(0xffffffffu, v[V - HW + j], 31);
            float o[V];
#pragma unroll
            for (int k = 0; k < V; k++) {
                float acc = bias;
#pragma unroll
                for (int i = 0; i < W; i++) {
                    const int e = k + i;   // index into prev ++ v
                    acc = fmaf(w[i], e < HW ? prev[e] : v[e - HW], acc);
                }
                o[k] = a.silu ? silu_acc<kAcc>(acc) : acc;
            }
            if (t < te) store_v<Tout, V, kVec>(orow, t, te, o);
        }
    }
}

// One decode token of the conv. A thread takes kUpdCh = 4 channels spaced by the
// grid's thread count, so each load instruction of a warp reads consecutive
// channels (coalesced), and issues all their loads before any arithmetic: 4W
// loads in flight per thread. (One channel per thread leaves the kernel waiting
// on HBM latency; 4 or 8 consecutive channels per thread with 16-byte state
// vectors measured slower: a warp's vector loads then stride over 4-8 times the
// bytes per instruction.) Each channel's output uses (state, x); its state drops
// the oldest entry and takes x.
constexpr int kUpdCh = 4;

template <int W>
__device__ __forceinline__ float conv_token(const ConvArgs& a, int64_t d, const float* s, float xt) {
    float acc = a.bias ? a.bias[d] : 0.f;
#pragma unroll
    for (int j = 0; j < W - 1; j++) acc = fmaf(a.w[d * W + j], s[j], acc);
    return fmaf(a.w[d * W + W - 1], xt, acc);
}

template <typename Tin, typename Tout, int W>
__global__ void __launch_bounds__(256) conv_update_kernel(ConvArgs a) {
    constexpr bool kAcc = sizeof(Tin) == 4;
    constexpr int HW = W - 1;
    constexpr int HA = HW > 0 ? HW : 1;
    const int64_t n = a.batch * a.dim;
    const int64_t stride = (int64_t)gridDim.x * 256;
    const int64_t i0 = (int64_t)blockIdx.x * 256 + threadIdx.x;
    const Tin* xp = static_cast<const Tin*>(a.x);
    Tout* op = static_cast<Tout*>(a.out);
    float s[kUpdCh][HA], xt[kUpdCh];
#pragma unroll
    for (int c = 0; c < kUpdCh; c++) {
        const int64_t i = i0 + c * stride;
        if (i < n) {
#pragma unroll
            for (int j = 0; j < HW; j++) s[c][j] = a.state_out[i * HW + j];
            xt[c] = to_f32(xp[i]);
        }
    }
#pragma unroll
    for (int c = 0; c < kUpdCh; c++) {
        const int64_t i = i0 + c * stride;
        if (i < n) {
            const float acc = conv_token<W>(a, i % a.dim, s[c], xt[c]);
            op[i] = from_f32<Tout>(a.silu ? silu_acc<kAcc>(acc) : acc);
            float* st = a.state_out + i * HW;
#pragma unroll
            for (int j = 0; j + 1 < HW; j++) st[j] = s[c][j + 1];
            if constexpr (HW > 0) st[HW - 1] = xt[c];
        }
    }
}

template <typename Tin, typename Tout, int W>
cudaError_t launch_fwd(const ConvArgs& a, cudaStream_t s) {
    const int64_t warps = a.batch * a.dim * a.n_seg;
    if (warps == 0) return cudaSuccess;
    const int64_t ctas = (warps + kWarps - 1) / kWarps;
    if (ctas > ((int64_t)1 << 31) - 1) return cudaErrorInvalidValue;
    if (a.vec) causal_conv1d_kernel<Tin, Tout, W, true><<<(unsigned)ctas, kThreads, 0, s>>>(a);
    else causal_conv1d_kernel<Tin, Tout, W, false><<<(unsigned)ctas, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin, typename Tout, int W>
cudaError_t launch_upd(const ConvArgs& a, cudaStream_t s) {
    const int64_t n = a.batch * a.dim;
    if (n == 0) return cudaSuccess;
    const int64_t ctas = ((n + kUpdCh - 1) / kUpdCh + 255) / 256;
    if (ctas > ((int64_t)1 << 31) - 1) return cudaErrorInvalidValue;
    conv_update_kernel<Tin, Tout, W><<<(unsigned)ctas, 256, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
cudaError_t by_width(const ConvArgs& a, bool update, cudaStream_t s) {
    switch (a.width) {
        case 1: return update ? launch_upd<Tin, Tout, 1>(a, s) : launch_fwd<Tin, Tout, 1>(a, s);
        case 2: return update ? launch_upd<Tin, Tout, 2>(a, s) : launch_fwd<Tin, Tout, 2>(a, s);
        case 3: return update ? launch_upd<Tin, Tout, 3>(a, s) : launch_fwd<Tin, Tout, 3>(a, s);
        default: return update ? launch_upd<Tin, Tout, 4>(a, s) : launch_fwd<Tin, Tout, 4>(a, s);
    }
}

cudaError_t dispatch(const ConvArgs& a, bool update, cudaStream_t s) {
    if (a.in_dtype == kBF16)
        return a.out_dtype == kBF16 ? by_width<__nv_bfloat16, __nv_bfloat16>(a, update, s)
                                    : by_width<__nv_bfloat16, float>(a, update, s);
    return a.out_dtype == kBF16 ? by_width<float, __nv_bfloat16>(a, update, s) : by_width<float, float>(a, update, s);
}

}  // namespace

int conv_block_steps(int in_dtype) { return 32 * (in_dtype == kBF16 ? 8 : 4); }

cudaError_t launch_causal_conv1d(const ConvArgs& a, cudaStream_t s) { return dispatch(a, false, s); }
cudaError_t launch_conv_update(const ConvArgs& a, cudaStream_t s) { return dispatch(a, true, s); }

}  // namespace ssm
